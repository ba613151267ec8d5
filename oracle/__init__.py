"""CPU oracle for sparse flash attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never calls it, and shares no code with it.

The arithmetic lives in ``sfa_oracle.c`` (plain C, IEEE double, OpenMP over
query rows).  This module compiles it with gcc, loads it with ctypes and
marshals CPU tensors into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

LAYOUTS = {"BSND": 0, "BNSD": 1}
DTYPES = {"f16": 0, "bf16": 1}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle into liboracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """ctypes handle of an oracle shared object with its signatures set."""
    lib = ctypes.CDLL(path)
    vp, i64, ci, cd = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    sfa_common = [vp, vp, vp, i64, vp] + [ci] * 8 + [cd, ci, ci, ci]
    lib.oracle_sfa.argtypes = sfa_common + [vp, vp]
    lib.oracle_sfa.restype = ci
    lib.oracle_sfa_rows.argtypes = sfa_common + [vp, i64, vp, vp]
    lib.oracle_sfa_rows.restype = ci
    bsr_common = [vp, vp, vp, vp, vp] + [ci] * 7 + [cd, ci]
    lib.oracle_bsr.argtypes = bsr_common + [vp, vp]
    lib.oracle_bsr.restype = ci
    lib.oracle_bsr_rows.argtypes = bsr_common + [vp, i64, vp, vp]
    lib.oracle_bsr_rows.restype = ci
    bsr_ex = [vp, vp, vp, vp, vp, vp, ci] + bsr_common[5:]
    lib.oracle_bsr_ex.argtypes = bsr_ex + [vp, vp]
    lib.oracle_bsr_ex.restype = ci
    bsr_cap = bsr_ex[:-1] + [cd] + bsr_ex[-1:]          # ..., scale, softcap, dtype
    lib.oracle_bsr_cap.argtypes = bsr_cap + [vp, vp]
    lib.oracle_bsr_cap.restype = ci
    lib.oracle_bsr_rows_cap.argtypes = bsr_cap + [vp, i64, vp, vp]
    lib.oracle_bsr_rows_cap.restype = ci
    lib.oracle_varbsr_cap.argtypes = [vp] * 6 + [ci] * 8 + [cd, cd, ci, vp, vp]
    lib.oracle_varbsr_cap.restype = ci
    lib.oracle_varbsr_rows_cap.argtypes = [vp] * 6 + [ci] * 8 + [cd, cd, ci, vp, i64, vp, vp]
    lib.oracle_varbsr_rows_cap.restype = ci
    lib.oracle_bsr_rows_ex.argtypes = bsr_ex + [vp, i64, vp, vp]
    lib.oracle_bsr_rows_ex.restype = ci
    lib.oracle_varbsr.argtypes = [vp] * 6 + [ci] * 8 + [cd, ci, vp, vp]
    lib.oracle_varbsr.restype = ci
    lib.oracle_varbsr_rows.argtypes = [vp] * 6 + [ci] * 8 + [cd, ci, vp, ctypes.c_int64, vp, vp]
    lib.oracle_varbsr_rows.restype = ci
    lib.oracle_decode.argtypes = [vp, i64, ci, vp]
    lib.oracle_decode.restype = None
    lib.oracle_bsr_scaled.argtypes = ([vp] * 6 + [ci] * 8 + [cd, cd, ci, ci] + [vp] * 3 +
                                      [vp, i64, vp, vp])
    lib.oracle_bsr_scaled.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


# element type codes of the C oracle
DTYPE_CODES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}


def _dtype_of(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"oracle takes fp16/bf16 tensors, got {t.dtype}")


def _any_dtype_of(t: torch.Tensor) -> int:
    """Element type code of a 16-bit or 8-bit floating-point tensor."""
    fp8 = {getattr(torch, "float8_e4m3fn", None): 2, getattr(torch, "float8_e5m2", None): 3}
    if t.dtype in fp8 and t.dtype is not None:
        return fp8[t.dtype]
    return _dtype_of(t)


def decode(codes, dtype: str) -> np.ndarray:
    """float64 values the oracle reads for uint8 (E4M3 / E5M2) or uint16
    (f16 / bf16) codes."""
    code = DTYPE_CODES[dtype]
    arr = np.ascontiguousarray(codes, dtype=np.uint8 if code >= 2 else np.uint16)
    out = np.empty(arr.size)
    _load().oracle_decode(arr.ctypes.data, arr.size, code, out.ctypes.data)
    return out.reshape(arr.shape)


def _ptr(t: torch.Tensor) -> int:
    if t.device.type != "cpu":
        raise TypeError("oracle takes CPU tensors")
    return t.data_ptr()


def _value_ld(v: torch.Tensor) -> int:
    """Element distance between consecutive value rows; v must be rows of
    `ld` elements (contiguous, or the prefix view key[..., :Dv]).  Strides of
    size-1 dimensions are ignored."""
    if v.is_contiguous():
        return v.shape[-1]
    d, st = list(v.shape), list(v.stride())
    ld = v.shape[-1]
    for ax in (2, 1, 0):
        if d[ax] > 1:
            inner = int(np.prod(d[ax + 1:3]))
            ld = st[ax] // inner
            break
    ok = st[3] == 1 and ld >= d[3]
    for ax in (0, 1, 2):
        if d[ax] > 1 and st[ax] != ld * int(np.prod(d[ax + 1:3])):
            ok = False
    if not ok:
        raise ValueError("value must be contiguous rows (or a prefix view of key)")
    return ld


def _check(rc: int, what: str):
    if rc == -2:
        raise OracleError(f"{what}: index out of range")
    if rc != 0:
        raise OracleError(f"{what}: invalid arguments ({rc})")


def sfa_dims(q, k, v, idx, layout):
    if layout == "BSND":
        B, S1, N1, Dk = q.shape
        _, S2, N2, _ = k.shape
    else:
        B, N1, S1, Dk = q.shape
        _, N2, S2, _ = k.shape
    return B, S1, S2, N1, N2, Dk, v.shape[-1], idx.shape[-1]


def sfa(q, k, v, idx, scale, layout="BSND", causal=False):
    """Top-K sparse attention on CPU tensors.  Returns (y, lse) as float64
    numpy arrays; y in the input layout, lse [B,S1,N1] (BSND) / [B,N1,S1]."""
    B, S1, S2, N1, N2, Dk, Dv, topK = sfa_dims(q, k, v, idx, layout)
    for t in (q, k, idx):
        assert t.is_contiguous()
    assert idx.dtype == torch.int32
    if layout == "BSND":
        y = np.empty((B, S1, N1, Dv))
        lse = np.empty((B, S1, N1))
    else:
        y = np.empty((B, N1, S1, Dv))
        lse = np.empty((B, N1, S1))
    rc = _load().oracle_sfa(_ptr(q), _ptr(k), _ptr(v), _value_ld(v), _ptr(idx), B, S1, S2, N1,
                            N2, Dk, Dv, topK, float(scale), LAYOUTS[layout], int(bool(causal)),
                            _dtype_of(q), y.ctypes.data, lse.ctypes.data)
    _check(rc, "oracle_sfa")
    return y, lse


def sfa_rows(q, k, v, idx, scale, rows, layout="BSND", causal=False):
    """Selected output rows: rows is an (n, 3) int array of (b, n1, s1).
    Returns (y_rows (n, Dv), lse_rows (n,))."""
    B, S1, S2, N1, N2, Dk, Dv, topK = sfa_dims(q, k, v, idx, layout)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    y = np.empty((n, Dv))
    lse = np.empty(n)
    rc = _load().oracle_sfa_rows(_ptr(q), _ptr(k), _ptr(v), _value_ld(v), _ptr(idx), B, S1, S2,
                                 N1, N2, Dk, Dv, topK, float(scale), LAYOUTS[layout],
                                 int(bool(causal)), _dtype_of(q), rows.ctypes.data, n,
                                 y.ctypes.data, lse.ctypes.data)
    _check(rc, "oracle_sfa_rows")
    return y, lse


def pack_mask(mask):
    """plan()'s `mask` (nnz, R, C) bool as the packed bytes the oracle reads:
    flattened, most significant bit first within each byte."""
    m = np.ascontiguousarray(np.asarray(mask, dtype=bool).reshape(-1))
    return np.packbits(m, bitorder="big")


def _mask_args(mask, packed_mask):
    if packed_mask is not None:
        pm = np.ascontiguousarray(packed_mask, dtype=np.uint8)
    elif mask is not None:
        pm = pack_mask(mask)
    else:
        return None, 0
    return pm, pm.ctypes.data


def bsr(q, k, v, indptr, indices, M, N, R, C, scale, mask=None, packed_mask=None, causal=False,
        softcap=0.0):
    """Block-sparse attention, NHD tensors.  Returns (y (M,Hq,d), lse (M,Hq)).
    mask: (nnz, R, C) bool per stored block (or packed_mask bytes); causal
    applies only without a mask; softcap > 0 soft-caps the scaled logits."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    indptr = indptr.to(torch.int32).contiguous()
    indices = indices.to(torch.int32).contiguous()
    y = np.empty((M, Hq, d))
    lse = np.empty((M, Hq))
    ind_ptr = _ptr(indices) if indices.numel() else 0
    keep, pm_ptr = _mask_args(mask, packed_mask)
    rc = _load().oracle_bsr_cap(_ptr(q), _ptr(k), _ptr(v), _ptr(indptr), ind_ptr, pm_ptr,
                                int(bool(causal)), M, N, R, C, Hq, Hkv, d, float(scale),
                                float(softcap), _dtype_of(q), y.ctypes.data, lse.ctypes.data)
    _check(rc, "oracle_bsr")
    del keep
    return y, lse


def bsr_scaled(q, k, v, indptr, indices, M, N, R, C, scale, scale_q=None, scale_k=None,
               scale_v=None, rows=None, mask=None, packed_mask=None, causal=False, softcap=0.0):
    """Block-sparse attention (NHD) on q and k / v of any of fp16, bf16,
    float8_e4m3fn, float8_e5m2 (q may differ from k / v), with run()'s
    per-head dequantisation scales (scale_q [Hq], scale_k / scale_v [Hkv];
    None = 1.0).  rows None: (y (M, Hq, d), lse (M, Hq)); rows (n, 2) of
    (query row, qo head): (y (n, d), lse (n))."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if _any_dtype_of(k) != _any_dtype_of(v):
        raise TypeError("k and v must share an element type")
    indptr = indptr.to(torch.int32).contiguous()
    indices = indices.to(torch.int32).contiguous()
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()

    def scales(x, n):
        if x is None:
            return None
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))
        if a.size != n:
            raise ValueError("a scale per head expected")
        return a
    sq, sk, sv = scales(scale_q, Hq), scales(scale_k, Hkv), scales(scale_v, Hkv)
    if rows is None:
        r_ptr, n = None, M * Hq
        y, lse = np.empty((M, Hq, d)), np.empty((M, Hq))
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        r_ptr, n = rows.ctypes.data, rows.shape[0]
        y, lse = np.empty((n, d)), np.empty(n)
    ind_ptr = _ptr(indices) if indices.numel() else 0
    keep, pm_ptr = _mask_args(mask, packed_mask)
    rc = _load().oracle_bsr_scaled(
        _ptr(q), _ptr(k), _ptr(v), _ptr(indptr), ind_ptr, pm_ptr, int(bool(causal)), M, N, R, C,
        Hq, Hkv, d, float(scale), float(softcap), _any_dtype_of(q), _any_dtype_of(k),
        None if sq is None else sq.ctypes.data, None if sk is None else sk.ctypes.data,
        None if sv is None else sv.ctypes.data, r_ptr, n, y.ctypes.data, lse.ctypes.data)
    _check(rc, "oracle_bsr_scaled")
    del keep
    return y, lse


def bsr_rows(q, k, v, indptr, indices, M, N, R, C, scale, rows, mask=None, packed_mask=None,
             causal=False, softcap=0.0):
    """Selected rows: rows is (n, 2) of (query row i, qo head h)."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    indptr = indptr.to(torch.int32).contiguous()
    indices = indices.to(torch.int32).contiguous()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    y = np.empty((n, d))
    lse = np.empty(n)
    ind_ptr = _ptr(indices) if indices.numel() else 0
    keep, pm_ptr = _mask_args(mask, packed_mask)
    rc = _load().oracle_bsr_rows_cap(_ptr(q), _ptr(k), _ptr(v), _ptr(indptr), ind_ptr, pm_ptr,
                                     int(bool(causal)), M, N, R, C, Hq, Hkv, d, float(scale),
                                     float(softcap), _dtype_of(q), rows.ctypes.data, n,
                                     y.ctypes.data, lse.ctypes.data)
    _check(rc, "oracle_bsr_rows")
    del keep
    return y, lse


def varbsr(q, k, v, block_mask_map, block_row_sz, block_col_sz, scale, causal=False, softcap=0.0):
    """Variable block-sparse attention, HND tensors: q (Hq, M, d), k/v (Hkv, N, d),
    block_mask_map (Hkv, MB, NB) bool, block_row_sz (Hkv, MB), block_col_sz
    (Hkv, NB).  Returns (y (Hq, M, d), lse (Hq, M))."""
    Hq, M, d = q.shape
    Hkv, N = k.shape[0], k.shape[1]
    mm = np.ascontiguousarray(np.asarray(block_mask_map, dtype=bool).astype(np.uint8))
    rs = np.ascontiguousarray(np.asarray(block_row_sz, dtype=np.int32))
    cs = np.ascontiguousarray(np.asarray(block_col_sz, dtype=np.int32))
    MB, NB = mm.shape[1], mm.shape[2]
    y = np.empty((Hq, M, d))
    lse = np.empty((Hq, M))
    rc = _load().oracle_varbsr_cap(_ptr(q.contiguous()), _ptr(k.contiguous()),
                                   _ptr(v.contiguous()), mm.ctypes.data, rs.ctypes.data,
                                   cs.ctypes.data, MB, NB, M, N, Hq, Hkv, d, int(bool(causal)),
                                   float(scale), float(softcap), _dtype_of(q), y.ctypes.data,
                                   lse.ctypes.data)
    _check(rc, "oracle_varbsr")
    return y, lse


def varbsr_rows(q, k, v, block_mask_map, block_row_sz, block_col_sz, scale, rows, causal=False,
                softcap=0.0):
    """Rows `rows` (flat h * M + i) of varbsr(): (y (n, d), lse (n))."""
    Hq, M, d = q.shape
    Hkv, N = k.shape[0], k.shape[1]
    mm = np.ascontiguousarray(np.asarray(block_mask_map, dtype=bool).astype(np.uint8))
    rs = np.ascontiguousarray(np.asarray(block_row_sz, dtype=np.int32))
    cs = np.ascontiguousarray(np.asarray(block_col_sz, dtype=np.int32))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    y = np.empty((n, d))
    lse = np.empty(n)
    rc = _load().oracle_varbsr_rows_cap(_ptr(q.contiguous()), _ptr(k.contiguous()),
                                        _ptr(v.contiguous()), mm.ctypes.data, rs.ctypes.data,
                                        cs.ctypes.data, mm.shape[1], mm.shape[2], M, N, Hq, Hkv,
                                        d, int(bool(causal)), float(scale), float(softcap),
                                        _dtype_of(q), rows.ctypes.data, n, y.ctypes.data,
                                        lse.ctypes.data)
    _check(rc, "oracle_varbsr_rows")
    return y, lse


# ---------------------------------------------------------------------------
# Precision standard ("SparseFlashAttention 算子 API 描述", §4 精度要求):
# relative error re = |actual - golden| / (|golden| + 1e-7) over the compared
# points; MERE = mean(re), MARE = max(re); pass iff MERE < Thr and
# MARE < 10 * Thr, with Thr = 2^-10 (fp16) or 2^-7 (bf16).  Near-zero golden
# values: an element also passes the MARE test when |actual - golden| <= cap
# (1e-2 fp16, 4e-2 bf16).

THRESHOLD = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7, "e4m3": 2.0 ** -3, "e5m2": 2.0 ** -2}
ABS_CAP = {"f16": 1e-2, "bf16": 4e-2, "e4m3": 4e-2, "e5m2": 4e-2}


def round_to(x, dtype: str) -> np.ndarray:
    """Round float64 values to fp16 / bf16 (nearest-even) and back."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to({"f16": torch.float16, "bf16": torch.bfloat16}[dtype]).to(torch.float64).numpy()


def precision_report(actual, golden, dtype: str, round_golden: bool = True,
                     out_dtype: str | None = None) -> dict:
    """MERE / MARE of `actual` against `golden`.  The golden of the operator
    spec returns its output in the input dtype, so by default the float64
    oracle values are rounded to `dtype` before comparing.  For the 8-bit
    formats (thresholds 2^-3 E4M3, 2^-2 E5M2) the output is 16-bit:
    `out_dtype` names it, the golden is rounded to it, and the near-zero cap
    is bf16's (the 8-bit paths' P carries about bf16's precision)."""
    a = np.asarray(actual, dtype=np.float64).ravel()
    g = np.asarray(golden, dtype=np.float64).ravel()
    if round_golden:
        g = round_to(g, out_dtype or dtype)
    if a.shape != g.shape:
        raise ValueError("shape mismatch")
    thr = THRESHOLD[dtype]
    if a.size == 0:
        return {"n": 0, "mere": 0.0, "mare": 0.0, "mare_capped": 0.0, "max_abs": 0.0,
                "threshold": thr, "passed": True, "finite": True}
    diff = np.abs(a - g)
    re = diff / (np.abs(g) + 1e-7)
    capped = np.where(diff <= ABS_CAP[dtype], 0.0, re)
    big = np.abs(g) >= 1e-3
    mere = float(re.mean())
    mare_c = float(capped.max())
    finite = bool(np.isfinite(a).all())
    return {"n": int(a.size), "mere": mere, "mere_big": float(re[big].mean()) if big.any() else 0.0,
            "mare": float(re.max()), "mare_capped": mare_c, "max_abs": float(diff.max()),
            "threshold": thr, "finite": finite,
            "passed": finite and mere < thr and mare_c < 10 * thr}
