"""Seeded synthetic inputs for the sparse-attention workloads.

Holds random numbers, index lists and workload shapes only -- none of the
attention arithmetic.  The CPU oracle and the CUDA path both consume the
buffers made here (the float32 normals are rounded to fp16/bf16 once, and the
same rounded tensors go to both sides).

Index lists and tensors are always generated in the canonical BSND order
([B, S1, N2, topK] for indices, [B, S, N, D] for q/k/v) and permuted for BNSD,
so one seed describes one problem in either layout.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so (plain C, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, i32, f64 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32, ctypes.c_double
            vp = ctypes.c_void_p
            lib.syn_normal_f32.argtypes = [u64, u64, i64, vp]
            lib.syn_normal_f32.restype = None
            lib.syn_index_uniform.argtypes = [u64, i64, i32, i32, ctypes.c_int, vp]
            lib.syn_index_uniform.restype = ctypes.c_int
            lib.syn_index_causal_mix.argtypes = [u64, i32, i32, i32, i32, i32, f64, i32, vp]
            lib.syn_index_causal_mix.restype = ctypes.c_int
            lib.syn_bsr_pattern.argtypes = [u64, i32, i32, f64, vp, vp]
            lib.syn_bsr_pattern.restype = i64
            _lib = lib
    return _lib


_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def normal(seed: int, stream: int, shape, dtype: str) -> torch.Tensor:
    """N(0,1) samples of `shape`, rounded (nearest-even) to fp16 or bf16."""
    n = int(np.prod(shape))
    buf = np.empty(n, dtype=np.float32)
    if n:
        _load().syn_normal_f32(seed, stream, n, buf.ctypes.data)
    return torch.from_numpy(buf).reshape(shape).to(_TORCH_DTYPE[dtype])


def normal_f32(seed: int, stream: int, shape) -> torch.Tensor:
    """N(0,1) float32 samples of `shape` (not rounded)."""
    n = int(np.prod(shape))
    buf = np.empty(n, dtype=np.float32)
    if n:
        _load().syn_normal_f32(seed, stream, n, buf.ctypes.data)
    return torch.from_numpy(buf).reshape(shape)


FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def quantize_per_head(x: torch.Tensor, fmt: str, head_axis: int):
    """FP8 codes of float32 `x` with one scale per index of `head_axis`:
    scale = max |x| over the head / the format's largest finite value, codes
    = x / scale converted (nearest) by torch.  Returns (float8 tensor, float32
    scales)."""
    dims = [a for a in range(x.dim()) if a != head_axis]
    amax = x.abs().amax(dim=dims).clamp_min(1e-12)
    scale = (amax / FP8_MAX[fmt]).to(torch.float32)
    shape = [1] * x.dim()
    shape[head_axis] = -1
    codes = (x / scale.view(shape)).to(FP8_TORCH[fmt])
    return codes, scale


def index_uniform(seed: int, rows: int, rng: int, topk: int, sorted_: bool) -> np.ndarray:
    """rows x topk distinct draws from [0, rng), random order or ascending."""
    out = np.empty((rows, topk), dtype=np.int32)
    rc = _load().syn_index_uniform(seed, rows, rng, topk, int(sorted_), out.ctypes.data)
    if rc:
        raise ValueError(f"syn_index_uniform failed ({rc})")
    return out


def index_causal_mix(seed, B, S1, N2, S2, topk, masked_frac, full_masked_rows) -> np.ndarray:
    """[B, S1, N2, topk] lists: ~masked_frac of each row above the bottom-right
    diagonal, the rest visible; rows (b=0, s1 < full_masked_rows) entirely above
    it (drawn with replacement)."""
    out = np.empty((B, S1, N2, topk), dtype=np.int32)
    rc = _load().syn_index_causal_mix(seed, B, S1, N2, S2, topk, masked_frac, full_masked_rows,
                                      out.ctypes.data)
    if rc:
        raise ValueError(f"syn_index_causal_mix failed ({rc})")
    return out


def bsr_pattern(seed: int, MB: int, NB: int, p: float):
    """(indptr, indices) of an MB x NB block pattern: diagonal always set,
    other blocks independently with probability p, columns ascending."""
    lib = _load()
    indptr = np.empty(MB + 1, dtype=np.int32)
    nnz = lib.syn_bsr_pattern(seed, MB, NB, p, indptr.ctypes.data, None)
    indices = np.empty(max(int(nnz), 1), dtype=np.int32)
    lib.syn_bsr_pattern(seed, MB, NB, p, indptr.ctypes.data, indices.ctypes.data)
    return indptr, indices[: int(nnz)]


# ---------------------------------------------------------------------------
# Workload descriptions


@dataclasses.dataclass(frozen=True)
class SfaCase:
    """One top-K sparse attention problem and its input recipe."""

    name: str
    B: int
    S1: int
    S2: int
    N1: int
    N2: int
    Dk: int
    Dv: int
    topK: int
    dtype: str              # "f16" | "bf16"
    layout: str             # "BSND" | "BNSD"
    causal: bool
    scale: float
    value_is_key_prefix: bool = False
    index_kind: str = "uniform"     # "uniform" | "sorted" | "causal_mix"
    masked_frac: float = 0.0        # causal_mix only
    full_masked_rows: int = 0       # causal_mix only
    seed: int = 1234

    @property
    def G(self) -> int:
        return self.N1 // self.N2

    def replace(self, **kw) -> "SfaCase":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class BsrCase:
    """One block-sparse attention problem and its input recipe."""

    name: str
    M: int
    N: int
    R: int
    C: int
    Hq: int
    Hkv: int
    d: int
    dtype: str
    p: float
    sm_scale: float
    seed: int = 1238
    causal: bool = False            # bottom-right causal (only without a mask)
    mask_keep: float = 0.0          # > 0: per-element block mask, each element kept with this p
    fp8: str = ""                   # "e4m3" / "e5m2": q, k, v in that format (dtype = out's)

    @property
    def MB(self) -> int:
        return (self.M + self.R - 1) // self.R

    @property
    def NB(self) -> int:
        return self.N // self.C

    def replace(self, **kw) -> "BsrCase":
        return dataclasses.replace(self, **kw)


# The five workloads (data seed = 1234 + workload number - 1).
TINY = SfaCase("tiny", B=1, S1=4, S2=64, N1=4, N2=1, Dk=64, Dv=64, topK=16, dtype="f16",
               layout="BSND", causal=False, scale=1.0 / math.sqrt(64), seed=1234)
GQA_DECODE = SfaCase("gqa_decode", B=16, S1=1, S2=8192, N1=32, N2=8, Dk=128, Dv=128, topK=1024,
                     dtype="bf16", layout="BNSD", causal=True, scale=0.08839,
                     index_kind="sorted", seed=1235)
MLA_DECODE = SfaCase("mla_decode", B=32, S1=1, S2=8192, N1=128, N2=1, Dk=576, Dv=512, topK=2048,
                     dtype="bf16", layout="BSND", causal=True, scale=0.04167,
                     value_is_key_prefix=True, seed=1236)
MLA_MTP = MLA_DECODE.replace(name="mla_mtp", S1=4)
PREFILL = SfaCase("sparse_prefill", B=2, S1=2048, S2=16384, N1=64, N2=8, Dk=192, Dv=128, topK=2048,
                  dtype="f16", layout="BSND", causal=True, scale=0.07217, value_is_key_prefix=True,
                  index_kind="causal_mix", masked_frac=0.10, full_masked_rows=8, seed=1237)
BSR = BsrCase("bsr", M=16384, N=16384, R=64, C=64, Hq=32, Hkv=8, d=128, dtype="f16", p=0.10,
              sm_scale=1.0 / math.sqrt(128), seed=1238)

# The operator page's call example (§6 额外信息): B=2, S1=1024, S2=8192, 32/8 heads,
# Dk=Dv=128, topK=512, fp16, BSND, non-causal, indices a random permutation prefix per row.
CALL_EXAMPLE = SfaCase("call_example", B=2, S1=1024, S2=8192, N1=32, N2=8, Dk=128, Dv=128,
                       topK=512, dtype="f16", layout="BSND", causal=False,
                       scale=1.0 / math.sqrt(128), seed=1239)
SFA_WORKLOADS = {c.name: c for c in (TINY, GQA_DECODE, MLA_DECODE, MLA_MTP, PREFILL, CALL_EXAMPLE)}
BSR_CAUSAL = BSR.replace(name="bsr_causal", causal=True)
BSR_MASK = BSR.replace(name="bsr_mask", mask_keep=0.5)
# The block-sparse workload with q, k, v in E4M3 and per-head scales
# (BlockSparseAttentionWrapper plan() kv_data_type, run() scale_q / k / v),
# fp16 out.
BSR_FP8 = BSR.replace(name="bsr_fp8", fp8="e4m3")
BSR_WORKLOADS = {c.name: c for c in (BSR, BSR_CAUSAL, BSR_MASK, BSR_FP8)}


@dataclasses.dataclass(frozen=True)
class VarBsrCase:
    """One variable block-sparse problem (per-kv-head block masks and block
    sizes, HND tensors) and its input recipe."""

    name: str
    M: int              # qo_len
    N: int              # kv_len
    MB: int             # row blocks per kv head
    NB: int             # column blocks per kv head
    Hq: int
    Hkv: int
    d: int
    dtype: str
    p: float            # each (kv head, row block, column block) set with this probability
    sm_scale: float
    seed: int = 1240
    causal: bool = False

    def replace(self, **kw) -> "VarBsrCase":
        return dataclasses.replace(self, **kw)


# 16384 x 16384 per head, 256 x 256 blocks of random sizes (mean 64), 10% set
VARBSR = VarBsrCase("varbsr", M=16384, N=16384, MB=256, NB=256, Hq=32, Hkv=8, d=128,
                    dtype="f16", p=0.10, sm_scale=1.0 / math.sqrt(128))
VARBSR_WORKLOADS = {VARBSR.name: VARBSR}


def _to_layout(t: torch.Tensor, layout: str) -> torch.Tensor:
    """Canonical [B, S, N, D] -> the requested layout (contiguous)."""
    return t if layout == "BSND" else t.permute(0, 2, 1, 3).contiguous()


def make_sfa_inputs(case: SfaCase) -> dict:
    """CPU tensors q, k, v, idx for `case` in its layout.

    Streams: q = 0, k = 1, v = 2 of the data seed; indices use seed + 1.  With
    value_is_key_prefix, v is the strided view k[..., :Dv] (no copy)."""
    c = case
    q = normal(c.seed, 0, (c.B, c.S1, c.N1, c.Dk), c.dtype)
    k = normal(c.seed, 1, (c.B, c.S2, c.N2, c.Dk), c.dtype)
    if c.index_kind == "causal_mix":
        idx = index_causal_mix(c.seed + 1, c.B, c.S1, c.N2, c.S2, c.topK, c.masked_frac,
                               c.full_masked_rows)
    else:
        idx = index_uniform(c.seed + 1, c.B * c.S1 * c.N2, c.S2, c.topK, c.index_kind == "sorted")
        idx = idx.reshape(c.B, c.S1, c.N2, c.topK)
    q = _to_layout(q, c.layout)
    k = _to_layout(k, c.layout)
    idx = _to_layout(torch.from_numpy(idx), c.layout)
    if c.value_is_key_prefix:
        v = k[..., : c.Dv]
    else:
        v = _to_layout(normal(c.seed, 2, (c.B, c.S2, c.N2, c.Dv), c.dtype), c.layout)
    return {"q": q, "k": k, "v": v, "idx": idx}


def bsr_mask(seed: int, nnz: int, R: int, C: int, keep: float) -> np.ndarray:
    """(nnz, R, C) bool per-element block mask, each element set with
    probability `keep` (numpy PCG64 stream of `seed`)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.random((nnz, R, C)) < keep


def make_bsr_inputs(case: BsrCase) -> dict:
    """CPU tensors q (M,Hq,d), k/v (N,Hkv,d) in NHD order, int32 indptr/indices,
    and (mask_keep > 0) the (nnz, R, C) bool mask.  With case.fp8, q / k / v
    are float8 codes of the same normals quantised per head, and scale_q
    (Hq) / scale_k / scale_v (Hkv) float32 hold their scales."""
    c = case
    indptr, indices = bsr_pattern(c.seed + 1, c.MB, c.NB, c.p)
    if c.fp8:
        q, sq = quantize_per_head(normal_f32(c.seed, 0, (c.M, c.Hq, c.d)), c.fp8, 1)
        k, sk = quantize_per_head(normal_f32(c.seed, 1, (c.N, c.Hkv, c.d)), c.fp8, 1)
        v, sv = quantize_per_head(normal_f32(c.seed, 2, (c.N, c.Hkv, c.d)), c.fp8, 1)
        scales = {"scale_q": sq, "scale_k": sk, "scale_v": sv}
    else:
        q = normal(c.seed, 0, (c.M, c.Hq, c.d), c.dtype)
        k = normal(c.seed, 1, (c.N, c.Hkv, c.d), c.dtype)
        v = normal(c.seed, 2, (c.N, c.Hkv, c.d), c.dtype)
        scales = {"scale_q": None, "scale_k": None, "scale_v": None}
    out = {"q": q, "k": k, "v": v, "indptr": torch.from_numpy(indptr),
           "indices": torch.from_numpy(indices.copy()), "mask": None, **scales}
    if c.mask_keep > 0:
        out["mask"] = bsr_mask(c.seed + 2, int(indptr[-1]), c.R, c.C, c.mask_keep)
    return out


def block_sizes(rng, heads: int, nblocks: int, total: int) -> np.ndarray:
    """(heads, nblocks) int32 sizes summing to `total` per head: nblocks - 1
    cut points drawn uniformly from [0, total] (so a block may be empty)."""
    cuts = np.sort(rng.integers(0, total + 1, size=(heads, nblocks - 1)), axis=1)
    edges = np.concatenate([np.zeros((heads, 1), np.int64), cuts,
                            np.full((heads, 1), total, np.int64)], axis=1)
    return np.diff(edges, axis=1).astype(np.int32)


def make_varbsr_inputs(case: VarBsrCase) -> dict:
    """CPU tensors q (Hq,M,d), k/v (Hkv,N,d) in HND order, and (numpy PCG64
    streams of seed + 1) the (Hkv,MB,NB) bool block mask map and int32 row
    (Hkv,MB) and column (Hkv,NB) block sizes."""
    c = case
    q = normal(c.seed, 0, (c.Hq, c.M, c.d), c.dtype)
    k = normal(c.seed, 1, (c.Hkv, c.N, c.d), c.dtype)
    v = normal(c.seed, 2, (c.Hkv, c.N, c.d), c.dtype)
    rng = np.random.Generator(np.random.PCG64(c.seed + 1))
    row_sz = block_sizes(rng, c.Hkv, c.MB, c.M)
    col_sz = block_sizes(rng, c.Hkv, c.NB, c.N)
    mask_map = rng.random((c.Hkv, c.MB, c.NB)) < c.p
    return {"q": q, "k": k, "v": v, "block_mask_map": mask_map, "block_row_sz": row_sz,
            "block_col_sz": col_sz}


def varbsr_counts(case: VarBsrCase, mask_map, row_sz, col_sz) -> dict:
    """Useful FLOPs (2*2*d per allowed (row, column, qo head)).  Without causal
    the allowed elements of kv head g are the sum over set blocks of
    row size x column size; with causal, those on or below the bottom-right
    diagonal."""
    c = case
    G = c.Hq // c.Hkv
    allowed = 0
    for g in range(c.Hkv):
        rs = np.asarray(row_sz[g], np.int64)
        cs = np.asarray(col_sz[g], np.int64)
        mm = np.asarray(mask_map[g], bool)
        if not c.causal:
            allowed += int((rs[:, None] * cs[None, :] * mm).sum())
            continue
        r0 = np.concatenate([[0], np.cumsum(rs)[:-1]])
        c0 = np.concatenate([[0], np.cumsum(cs)[:-1]])
        off = c.N - c.M
        for rb in range(c.MB):
            rows = np.arange(r0[rb], r0[rb] + rs[rb])
            for cb in np.nonzero(mm[rb])[0]:
                allowed += int(np.clip(rows + off - c0[cb] + 1, 0, cs[cb]).sum())
    return {"flops": 4 * c.d * allowed * G, "allowed": allowed * G}   # (row, column, qo head)


def sfa_counts(case: SfaCase, idx: torch.Tensor | None = None) -> dict:
    """Algorithmic work of one call: useful FLOPs (2*(Dk+Dv) per unmasked
    (query head, slot) pair), gathered K/V bytes (per selected slot per KV
    group; V counted separately unless it is the key prefix), and the bytes of
    q, indices and output."""
    c = case
    E = 2
    slots = c.B * c.N2 * c.S1 * c.topK
    if idx is not None and c.causal:
        t = idx if c.layout == "BSND" else idx.permute(0, 2, 1, 3)
        s1 = torch.arange(c.S1, dtype=torch.int64).view(1, c.S1, 1, 1)
        unmasked = int((t.to(torch.int64) <= s1 + (c.S2 - c.S1)).sum())
    else:
        unmasked = slots
    flops = 2 * (c.Dk + c.Dv) * unmasked * c.G
    row_bytes = c.Dk * E + (0 if c.value_is_key_prefix else c.Dv * E)
    gathered = slots * row_bytes
    other = (c.B * c.S1 * c.N1 * c.Dk * E + slots * 4 + c.B * c.S1 * c.N1 * c.Dv * E)
    return {"flops": flops, "gathered_bytes": gathered, "other_bytes": other,
            "slots": slots, "unmasked_slots": unmasked}


def bsr_counts(case: BsrCase, indptr: torch.Tensor, indices: torch.Tensor | None = None,
               mask: np.ndarray | None = None) -> dict:
    """Useful FLOPs (2*2*d per allowed (row, column, qo head)) and the K/V bytes
    each (row block, kv head) work item reads (64x64 blocks of K and V).  With
    a mask the allowed elements are its set bits; with causal (and no mask)
    those on or below the bottom-right diagonal, and blocks wholly above it
    are not read."""
    c = case
    ip = indptr.to(torch.int64)
    rows_in_block = torch.full((c.MB,), c.R, dtype=torch.int64)
    rows_in_block[-1] = c.M - (c.MB - 1) * c.R
    blocks_per_row = ip[1:] - ip[:-1]
    nnz = int(ip[-1])
    read_blocks = nnz
    if mask is not None:
        # rows past M in the last block row are not query rows
        valid = np.ones((nnz, c.R, 1), dtype=bool)
        last0 = int(ip[c.MB - 1])
        valid[last0:, int(rows_in_block[-1]):, :] = False
        allowed = int((mask & valid).sum())
    elif c.causal and indices is not None:
        ix = indices.to(torch.int64).numpy()
        allowed, read_blocks = 0, 0
        off = c.N - c.M
        for br in range(c.MB):
            r0, r1 = br * c.R, br * c.R + int(rows_in_block[br])
            for k in range(int(ip[br]), int(ip[br + 1])):
                c0 = int(ix[k]) * c.C
                if c0 > r1 - 1 + off:
                    continue
                read_blocks += 1
                rows = np.arange(r0, r1)
                allowed += int(np.clip(rows + off - c0 + 1, 0, c.C).sum())
    else:
        allowed = int((blocks_per_row * rows_in_block).sum()) * c.C
    flops = 4 * c.d * allowed * c.Hq
    gathered = read_blocks * c.C * c.Hkv * c.d * 2 * 2
    return {"flops": flops, "gathered_bytes": gathered, "nnz": nnz, "allowed": allowed}
