"""Python binding of libsfa_gb300.so (sparse flash attention for GB300).

Argument marshalling only: every function here forwards to the C entry point
of the same name declared in include/sfa.h; all computation runs in the
library's CUDA kernels.  Tensors are passed as device pointers (torch is used
for device memory and streams only).  If the shared library has not been
built, loading raises -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LIB_PATH = _build.LIB_PATH

SFA_OK = 0
SFA_ERR_INVALID_ARG = 1
SFA_ERR_UNSUPPORTED = 2
SFA_ERR_WORKSPACE = 3
SFA_ERR_INDEX_RANGE = 4
SFA_ERR_CUDA = 5
SFA_ERR_DEVICE_TIMEOUT = 6

LAYOUTS = {"BSND": 0, "BNSD": 1}
KV_LAYOUTS = {"NHD": 0, "HND": 1}
DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}

# Every entry point of include/sfa.h.
EXPORTS = ("sfa_run", "sfa_run_ex", "sfa_workspace_size", "sfa_get_last_error",
           "sfa_status_string", "sfa_kernel_launches", "sfa_run_noalloc", "bsr_plan", "bsr_plan_int_workspace_size", "bsr_run",
           "bsr_plan_destroy", "bsr_plan_masked", "bsr_plan_masked_int_workspace_size",
           "varbsr_plan", "varbsr_plan_int_workspace_size", "varbsr_plan_dims", "varbsr_run",
           "varbsr_plan_destroy", "bsr_plan_set_logits_soft_cap",
           "varbsr_plan_set_logits_soft_cap", "bsr_plan_set_kv_layout",
           "bsr_plan_set_data_types", "bsr_run_scaled", "sfa_gather_probe",
           "sfa_gather_probe_tma")


class SfaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class SfaOptions(ctypes.Structure):
    _fields_ = [("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("value_is_key_prefix", ctypes.c_int), ("validate_indices", ctypes.c_int),
                ("num_splits", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("num_ctas", ctypes.c_int), ("inputs_ready", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library (nvcc, sm_103a)."""
    return _build.build(force=force)


def load():
    """ctypes handle of the built library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; call build() first")
            lib = ctypes.CDLL(LIB_PATH)
            vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            sfa_args = [vp, vp, vp, vp] + [ci] * 8 + [cf, ci, ci, ci, vp, vp, vp]
            lib.sfa_run.argtypes = sfa_args
            lib.sfa_run.restype = ci
            lib.sfa_run_noalloc.argtypes = sfa_args
            lib.sfa_run_noalloc.restype = ci
            lib.sfa_run_ex.argtypes = sfa_args + [ctypes.POINTER(SfaOptions)]
            lib.sfa_run_ex.restype = ci
            lib.sfa_workspace_size.argtypes = [ci] * 8 + [ctypes.POINTER(sz)]
            lib.sfa_workspace_size.restype = ci
            lib.sfa_get_last_error.argtypes = [vp]
            lib.sfa_get_last_error.restype = ci
            lib.sfa_status_string.argtypes = [ci]
            lib.sfa_status_string.restype = ctypes.c_char_p
            lib.sfa_kernel_launches.argtypes = []
            lib.sfa_kernel_launches.restype = ctypes.c_uint64
            lib.bsr_plan.argtypes = [vp, vp] + [ci] * 8 + [cf, ci, vp, sz, vp, sz, vp,
                                                          ctypes.POINTER(vp)]
            lib.bsr_plan.restype = ci
            lib.bsr_plan_int_workspace_size.argtypes = [vp] + [ci] * 7 + [ctypes.POINTER(sz)]
            lib.bsr_plan_int_workspace_size.restype = ci
            lib.bsr_plan_masked.argtypes = [vp, vp, vp] + [ci] * 8 + [cf, ci, vp, sz, vp, sz, vp,
                                                                   ctypes.POINTER(vp)]
            lib.bsr_plan_masked.restype = ci
            lib.bsr_plan_masked_int_workspace_size.argtypes = [vp] + [ci] * 8 + [ctypes.POINTER(sz)]
            lib.bsr_plan_masked_int_workspace_size.restype = ci
            lib.bsr_run.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            lib.bsr_run.restype = ci
            lib.bsr_plan_destroy.argtypes = [vp]
            lib.bsr_plan_destroy.restype = None
            lib.varbsr_plan.argtypes = [vp, vp, vp] + [ci] * 6 + [cf, ci, vp, sz, vp,
                                                               ctypes.POINTER(vp)]
            lib.varbsr_plan.restype = ci
            lib.varbsr_plan_int_workspace_size.argtypes = [vp, vp, vp] + [ci] * 6 + [ctypes.POINTER(sz)]
            lib.varbsr_plan_int_workspace_size.restype = ci
            lib.varbsr_plan_dims.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci)]
            lib.varbsr_plan_dims.restype = ci
            lib.varbsr_run.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            lib.varbsr_run.restype = ci
            lib.varbsr_plan_destroy.argtypes = [vp]
            lib.varbsr_plan_destroy.restype = None
            lib.bsr_plan_set_logits_soft_cap.argtypes = [vp, cf]
            lib.bsr_plan_set_logits_soft_cap.restype = ci
            lib.varbsr_plan_set_logits_soft_cap.argtypes = [vp, cf]
            lib.varbsr_plan_set_logits_soft_cap.restype = ci
            lib.bsr_plan_set_kv_layout.argtypes = [vp, ci]
            lib.bsr_plan_set_kv_layout.restype = ci
            lib.bsr_plan_set_data_types.argtypes = [vp, ci, ci, ci]
            lib.bsr_plan_set_data_types.restype = ci
            lib.bsr_run_scaled.argtypes = [vp] * 10
            lib.bsr_run_scaled.restype = ci
            lib.sfa_gather_probe.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, sz, vp]
            lib.sfa_gather_probe.restype = ci
            lib.sfa_gather_probe_tma.argtypes = [vp, vp, vp] + [ci] * 8 + [vp]
            lib.sfa_gather_probe_tma.restype = ci
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().sfa_status_string(int(status)).decode()


def _ptr(x) -> int | None:
    """Device/host address of a tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != SFA_OK:
        raise SfaError(status, what)


def _enum(v, table):
    return table[v] if isinstance(v, str) else int(v)


def sfa_run(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale, layout, causal, dtype,
            out, lse=None, stream=None, check=True) -> int:
    """Forwards to sfa_run(); returns the status (raises unless check=False)."""
    st = load().sfa_run(_ptr(q), _ptr(k), _ptr(v), _ptr(sparse_idx), B, S1, S2, N1, N2, Dk, Dv,
                        topK, float(scale), _enum(layout, LAYOUTS), int(bool(causal)),
                        _enum(dtype, DTYPES), _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check(st, "sfa_run")
    return st


def sfa_run_ex(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale, layout, causal, dtype,
               out, lse=None, stream=None, workspace=None, workspace_bytes=0,
               value_is_key_prefix=False, validate_indices=False, num_splits=0,
               ctas_per_sm=0, num_ctas=0, inputs_ready=False, check=True) -> int:
    """Forwards to sfa_run_ex() with an sfa_options built from the keywords."""
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    opt = SfaOptions(_ptr(workspace), int(workspace_bytes), int(bool(value_is_key_prefix)),
                     int(bool(validate_indices)), int(num_splits), int(ctas_per_sm),
                     int(num_ctas), int(bool(inputs_ready)))
    st = load().sfa_run_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(sparse_idx), B, S1, S2, N1, N2, Dk, Dv,
                           topK, float(scale), _enum(layout, LAYOUTS), int(bool(causal)),
                           _enum(dtype, DTYPES), _ptr(out), _ptr(lse), _stream(stream),
                           ctypes.byref(opt))
    if check:
        _check(st, "sfa_run_ex")
    return st


def sfa_run_noalloc(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale, layout, causal,
                    dtype, out, lse=None, stream=None, check=True) -> int:
    """Forwards to sfa_run_noalloc(): same arguments as sfa_run, for callers
    that cannot allocate device memory (the library keeps the split partials
    in a fixed device array of SFA_NOALLOC_SCRATCH_BYTES)."""
    st = load().sfa_run_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(sparse_idx), B, S1, S2, N1, N2,
                                Dk, Dv, topK, float(scale), _enum(layout, LAYOUTS),
                                int(bool(causal)), _enum(dtype, DTYPES), _ptr(out), _ptr(lse),
                                _stream(stream))
    if check:
        _check(st, "sfa_run_noalloc")
    return st


SFA_NOALLOC_SCRATCH_BYTES = 8 << 20


def sfa_gather_probe(k, v, sparse_idx, B, S1, S2, N2, Dk, Dv, topK, layout, sink, stream=None):
    """Forwards to sfa_gather_probe() (measurement only): the call's K/V row
    gather alone.  sink: a device tensor of >= 2 * SM count * 4 bytes."""
    _check(load().sfa_gather_probe(_ptr(k), _ptr(v), _ptr(sparse_idx), B, S1, S2, N2, Dk, Dv,
                                   topK, _enum(layout, LAYOUTS), _ptr(sink),
                                   sink.numel() * sink.element_size(), _stream(stream)),
           "sfa_gather_probe")


def sfa_gather_probe_tma(k, v, sparse_idx, B, S1, S2, N2, Dk, Dv, topK, layout, stream=None):
    """Forwards to sfa_gather_probe_tma() (measurement only): the same rows
    moved by TMA row gathers (k, v contiguous, or v is k)."""
    _check(load().sfa_gather_probe_tma(_ptr(k), _ptr(v), _ptr(sparse_idx), B, S1, S2, N2, Dk, Dv,
                                       topK, _enum(layout, LAYOUTS), _stream(stream)),
           "sfa_gather_probe_tma")


def sfa_workspace_size(B, S1, N1, N2, Dk, Dv, topK, num_splits=0) -> int:
    out = ctypes.c_size_t(0)
    _check(load().sfa_workspace_size(B, S1, N1, N2, Dk, Dv, topK, num_splits, ctypes.byref(out)),
           "sfa_workspace_size")
    return out.value


def sfa_kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return int(load().sfa_kernel_launches())


def sfa_get_last_error(stream=None) -> int:
    """Status of the device error word (synchronises the stream)."""
    return load().sfa_get_last_error(_stream(stream))


class BsrPlan:
    """Owner of a bsr_plan_t handle (destroyed with the object)."""

    def __init__(self, handle: int, int_ws, M, N, Hq, d):
        self.handle = handle
        self.int_ws = int_ws          # keeps the device work list alive
        self.M, self.N, self.Hq, self.d = M, N, Hq, d

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.bsr_plan_destroy(self.handle)
            self.handle = None


def bsr_plan_int_workspace_size(indptr_host, M, N, R, C, num_qo_heads, num_kv_heads,
                                head_dim) -> int:
    out = ctypes.c_size_t(0)
    _check(load().bsr_plan_int_workspace_size(_ptr(indptr_host), M, N, R, C, num_qo_heads,
                                              num_kv_heads, head_dim, ctypes.byref(out)),
           "bsr_plan_int_workspace_size")
    return out.value


def bsr_plan_masked_int_workspace_size(indptr_host, M, N, R, C, num_qo_heads, num_kv_heads,
                                       head_dim, with_mask) -> int:
    out = ctypes.c_size_t(0)
    _check(load().bsr_plan_masked_int_workspace_size(_ptr(indptr_host), M, N, R, C, num_qo_heads,
                                                     num_kv_heads, head_dim, int(bool(with_mask)),
                                                     ctypes.byref(out)),
           "bsr_plan_masked_int_workspace_size")
    return out.value


def pack_block_mask(mask):
    """plan()'s `mask` (nnz, R, C) bool -> the packed bytes bsr_plan_masked
    reads: flattened in stored-block order, most significant bit first."""
    import numpy as np
    m = mask.detach().cpu().numpy() if hasattr(mask, "detach") else np.asarray(mask)
    return np.packbits(np.ascontiguousarray(m.astype(bool).reshape(-1)), bitorder="big")


def bsr_plan(indptr_host, indices_host, M, N, R, C, num_qo_heads, num_kv_heads, head_dim,
             causal=False, sm_scale=0.0, dtype="f16", int_ws=None, float_ws=None,
             stream=None, mask=None, packed_mask=None, logits_soft_cap=0.0,
             kv_layout="NHD") -> BsrPlan:
    """Forwards to bsr_plan(), or to bsr_plan_masked() when a per-element
    mask ((nnz, R, C) bool) or its packed bytes are given, then to
    bsr_plan_set_logits_soft_cap() when logits_soft_cap > 0 and to
    bsr_plan_set_kv_layout() when kv_layout is not NHD.  indptr/indices are
    host int32 tensors; int_ws a device uint8 tensor (allocated here with
    torch if None)."""
    import numpy as np
    import torch
    if mask is not None and packed_mask is None:
        packed_mask = pack_block_mask(mask)
    if packed_mask is not None:
        packed_mask = np.ascontiguousarray(packed_mask, dtype=np.uint8)
    if int_ws is None:
        need = bsr_plan_masked_int_workspace_size(indptr_host, M, N, R, C, num_qo_heads,
                                                  num_kv_heads, head_dim, packed_mask is not None)
        int_ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    fws_bytes = 0 if float_ws is None else float_ws.numel() * float_ws.element_size()
    handle = ctypes.c_void_p(0)
    args = (M, N, R, C, num_qo_heads, num_kv_heads, head_dim, int(bool(causal)), float(sm_scale),
            _enum(dtype, DTYPES), _ptr(int_ws), int_ws.numel() * int_ws.element_size(),
            _ptr(float_ws), fws_bytes, _stream(stream), ctypes.byref(handle))
    ind = _ptr(indices_host) if indices_host.numel() else None
    if packed_mask is None:
        st = load().bsr_plan(_ptr(indptr_host), ind, *args)
    else:
        st = load().bsr_plan_masked(_ptr(indptr_host), ind, packed_mask.ctypes.data, *args)
    _check(st, "bsr_plan")
    plan = BsrPlan(handle.value, int_ws, M, N, num_qo_heads, head_dim)
    if logits_soft_cap > 0:
        bsr_plan_set_logits_soft_cap(plan, logits_soft_cap)
    if _enum(kv_layout, KV_LAYOUTS) != 0:
        bsr_plan_set_kv_layout(plan, kv_layout)
    return plan


def bsr_plan_set_kv_layout(plan: BsrPlan, kv_layout):
    """k / v layout of later bsr_run calls: "NHD" (N, Hkv, d) or "HND" (Hkv, N, d)."""
    _check(load().bsr_plan_set_kv_layout(plan.handle, _enum(kv_layout, KV_LAYOUTS)),
           "bsr_plan_set_kv_layout")


def bsr_plan_set_logits_soft_cap(plan: BsrPlan, logits_soft_cap: float):
    _check(load().bsr_plan_set_logits_soft_cap(plan.handle, float(logits_soft_cap)),
           "bsr_plan_set_logits_soft_cap")


def bsr_run(plan: BsrPlan, q, k, v, out, lse=None, stream=None):
    _check(load().bsr_run(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                          _stream(stream)), "bsr_run")


def bsr_plan_set_data_types(plan: BsrPlan, q_dtype, kv_dtype, o_dtype):
    """plan()'s q / kv / o data types: "f16", "bf16", "e4m3", "e5m2"."""
    _check(load().bsr_plan_set_data_types(plan.handle, _enum(q_dtype, DTYPES),
                                          _enum(kv_dtype, DTYPES), _enum(o_dtype, DTYPES)),
           "bsr_plan_set_data_types")


def bsr_run_scaled(plan: BsrPlan, q, k, v, scale_q=None, scale_k=None, scale_v=None, out=None,
                   lse=None, stream=None):
    """run() with per-head float32 device scales (None = 1.0).  FP8 tensors
    may be torch float8 or uint8 tensors holding the codes."""
    _check(load().bsr_run_scaled(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(scale_q),
                                 _ptr(scale_k), _ptr(scale_v), _ptr(out), _ptr(lse),
                                 _stream(stream)), "bsr_run_scaled")


def bsr_plan_destroy(plan: BsrPlan):
    if plan.handle:
        load().bsr_plan_destroy(plan.handle)
        plan.handle = None


class VarBsrPlan:
    """Owner of a varbsr_plan_t handle (destroyed with the object)."""

    def __init__(self, handle: int, int_ws, Hq, d):
        self.handle = handle
        self.int_ws = int_ws          # keeps the device tile and work lists alive
        self.Hq, self.d = Hq, d
        qo, kv = ctypes.c_int(0), ctypes.c_int(0)
        _check(load().varbsr_plan_dims(handle, ctypes.byref(qo), ctypes.byref(kv)),
               "varbsr_plan_dims")
        self.qo_len, self.kv_len = qo.value, kv.value

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.varbsr_plan_destroy(self.handle)
            self.handle = None


def _varbsr_host_args(block_mask_map, block_row_sz, block_col_sz):
    import numpy as np

    def host(x, dt):
        x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
        return np.ascontiguousarray(x.astype(dt))
    mm = host(block_mask_map, bool).view(np.uint8)
    rs = host(block_row_sz, np.int32)
    cs = host(block_col_sz, np.int32)
    if mm.ndim != 3 or rs.shape != mm.shape[:2] or cs.shape != (mm.shape[0], mm.shape[2]):
        raise ValueError("block_mask_map (Hkv, MB, NB), block_row_sz (Hkv, MB), "
                         "block_col_sz (Hkv, NB) expected")
    return mm, rs, cs


def varbsr_plan_int_workspace_size(block_mask_map, block_row_sz, block_col_sz, num_qo_heads,
                                   num_kv_heads, head_dim, causal=False) -> int:
    mm, rs, cs = _varbsr_host_args(block_mask_map, block_row_sz, block_col_sz)
    out = ctypes.c_size_t(0)
    _check(load().varbsr_plan_int_workspace_size(mm.ctypes.data, rs.ctypes.data, cs.ctypes.data,
                                                 mm.shape[1], mm.shape[2], num_qo_heads,
                                                 num_kv_heads, head_dim, int(bool(causal)),
                                                 ctypes.byref(out)),
           "varbsr_plan_int_workspace_size")
    return out.value


def varbsr_plan(block_mask_map, block_row_sz, block_col_sz, num_qo_heads, num_kv_heads,
                head_dim, causal=False, sm_scale=0.0, dtype="f16", int_ws=None,
                stream=None, logits_soft_cap=0.0) -> VarBsrPlan:
    """Forwards to varbsr_plan().  The block mask map and sizes may be numpy
    arrays or tensors on any device (they are read on the host); int_ws is a
    device uint8 tensor (allocated here with torch if None)."""
    import torch
    mm, rs, cs = _varbsr_host_args(block_mask_map, block_row_sz, block_col_sz)
    if int_ws is None:
        need = varbsr_plan_int_workspace_size(mm, rs, cs, num_qo_heads, num_kv_heads, head_dim,
                                              causal)
        int_ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    handle = ctypes.c_void_p(0)
    _check(load().varbsr_plan(mm.ctypes.data, rs.ctypes.data, cs.ctypes.data, mm.shape[1],
                              mm.shape[2], num_qo_heads, num_kv_heads, head_dim,
                              int(bool(causal)), float(sm_scale), _enum(dtype, DTYPES),
                              _ptr(int_ws), int_ws.numel() * int_ws.element_size(),
                              _stream(stream), ctypes.byref(handle)), "varbsr_plan")
    plan = VarBsrPlan(handle.value, int_ws, num_qo_heads, head_dim)
    if logits_soft_cap > 0:
        varbsr_plan_set_logits_soft_cap(plan, logits_soft_cap)
    return plan


def varbsr_plan_set_logits_soft_cap(plan: VarBsrPlan, logits_soft_cap: float):
    _check(load().varbsr_plan_set_logits_soft_cap(plan.handle, float(logits_soft_cap)),
           "varbsr_plan_set_logits_soft_cap")


def varbsr_run(plan: VarBsrPlan, q, k, v, out, lse=None, stream=None):
    _check(load().varbsr_run(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                             _stream(stream)), "varbsr_run")


def varbsr_plan_destroy(plan: VarBsrPlan):
    if plan.handle:
        load().varbsr_plan_destroy(plan.handle)
        plan.handle = None


# ---------------------------------------------------------------------------
# Convenience: allocate outputs with torch and call the entry points above.

def sparse_flash_attention(query, key, value, sparse_indices, scale, layout="BSND",
                           causal=False, return_lse=False, stream=None, **opts):
    """Shapes as in the operator spec; value may be key[..., :Dv] (prefix view)."""
    import torch
    if layout == "BSND":
        B, S1, N1, Dk = query.shape
        _, S2, N2, _ = key.shape
        out_shape, lse_shape = (B, S1, N1, value.shape[-1]), (B, S1, N1)
    else:
        B, N1, S1, Dk = query.shape
        _, N2, S2, _ = key.shape
        out_shape, lse_shape = (B, N1, S1, value.shape[-1]), (B, N1, S1)
    Dv = value.shape[-1]
    topK = sparse_indices.shape[-1]
    dtype = {torch.float16: "f16", torch.bfloat16: "bf16"}[query.dtype]
    prefix = value.data_ptr() == key.data_ptr()
    if not prefix:
        value = value.contiguous()
    out = torch.empty(out_shape, dtype=query.dtype, device=query.device)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=query.device) if return_lse else None
    v_arg = key if prefix else value
    sfa_run_ex(query, key, v_arg, sparse_indices, B, S1, S2, N1, N2, Dk, Dv, topK, scale, layout,
               causal, dtype, out, lse, stream, value_is_key_prefix=prefix, **opts)
    return (out, lse) if return_lse else out
