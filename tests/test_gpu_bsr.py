"""GPU parity of the block-sparse path against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_serving_sfa_gb300 as sfa
import synth
from tests.golden import fixtures
from tests.sfa_testlib import LSE_ATOL, LSE_RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    sfa.build()
    sfa.load()


def run_bsr(q, k, v, indptr, indices, M, N, R, C, scale, dtype):
    Hq, d, Hkv = q.shape[1], q.shape[2], k.shape[1]
    plan = sfa.bsr_plan(indptr, indices, M, N, R, C, Hq, Hkv, d, sm_scale=scale, dtype=dtype)
    out = torch.empty_like(q.cuda())
    lse = torch.empty((M, Hq), dtype=torch.float32, device="cuda")
    sfa.bsr_run(plan, q.cuda(), k.cuda(), v.cuda(), out, lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def compare(out, lse, y, l, dtype):
    rep = oracle.precision_report(out.float().numpy(), y, dtype)
    assert rep["passed"], rep
    lg = lse.numpy().astype(np.float64)
    empty = np.isneginf(l)
    assert np.array_equal(np.isneginf(lg), empty)
    np.testing.assert_allclose(lg[~empty], l[~empty], atol=LSE_ATOL, rtol=LSE_RTOL)
    if empty.any():
        assert np.all(out.float().numpy()[empty] == 0.0)


def test_worked_example():
    fx = fixtures.bsr_3x3_example()
    M, N, Hq, Hkv, d = fx["M"], fx["N"], fx["num_qo_heads"], fx["num_kv_heads"], fx["head_dim"]
    q = synth.normal(11, 0, (M, Hq, d), "f16")
    k = synth.normal(11, 1, (N, Hkv, d), "f16")
    v = synth.normal(11, 2, (N, Hkv, d), "f16")
    ip = torch.tensor(fx["indptr"], dtype=torch.int32)
    ix = torch.tensor(fx["indices"], dtype=torch.int32)
    scale = 1 / math.sqrt(d)
    out, lse = run_bsr(q, k, v, ip, ix, M, N, 1, 1, scale, "f16")
    y, l = oracle.bsr(q, k, v, ip, ix, M, N, 1, 1, scale)
    compare(out, lse, y, l, "f16")


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype,p", [
    (200, 192, 64, 64, 8, 2, 128, "f16", 0.3),
    (130, 256, 64, 32, 4, 4, 64, "bf16", 0.4),
    (97, 120, 16, 24, 6, 3, 192, "f16", 0.5),
    (64, 64, 100, 8, 2, 1, 256, "bf16", 0.5),
    (300, 320, 128, 64, 4, 1, 128, "bf16", 0.2),
    (33, 40, 1, 1, 2, 2, 64, "f16", 0.3),
])
def test_shapes(M, N, R, C, Hq, Hkv, d, dtype, p):
    case = synth.BsrCase("t", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=p,
                         sm_scale=1 / math.sqrt(d), seed=77)
    x = synth.make_bsr_inputs(case)
    out, lse = run_bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                       case.sm_scale, dtype)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C, case.sm_scale)
    compare(out, lse, y, l, dtype)


def test_empty_rows_and_plan_reuse():
    M, N, R, C = 128, 128, 32, 32
    indptr = torch.tensor([0, 2, 2, 3, 3], dtype=torch.int32)    # block rows 1 and 3 empty
    indices = torch.tensor([0, 3, 1], dtype=torch.int32)
    q = synth.normal(5, 0, (M, 4, 64), "f16")
    k = synth.normal(5, 1, (N, 2, 64), "f16")
    v = synth.normal(5, 2, (N, 2, 64), "f16")
    plan = sfa.bsr_plan(indptr, indices, M, N, R, C, 4, 2, 64, sm_scale=0.125, dtype="f16")
    y, l = oracle.bsr(q, k, v, indptr, indices, M, N, R, C, 0.125)
    for _ in range(2):             # the plan is reusable
        out = torch.empty((M, 4, 64), dtype=torch.float16, device="cuda")
        lse = torch.empty((M, 4), dtype=torch.float32, device="cuda")
        sfa.bsr_run(plan, q.cuda(), k.cuda(), v.cuda(), out, lse)
        torch.cuda.synchronize()
        compare(out.cpu(), lse.cpu(), y, l, "f16")
        assert torch.all(out[32:64] == 0) and torch.all(torch.isneginf(lse[32:64]))


def test_full_workload_sampled():
    case = synth.BSR
    x = synth.make_bsr_inputs(case)
    out, lse = run_bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N, case.R,
                       case.C, case.sm_scale, case.dtype)
    rng = np.random.default_rng(1)
    rows = np.stack([rng.integers(0, case.M, 48), rng.integers(0, case.Hq, 48)], axis=1)
    # the edges of every work item (one row block x one kv head, two M-tiles
    # of 128 / G rows): rows 0, TR - 1, TR and R - 1 of each row block, the
    # qo head rotating over the heads from block to block
    tr = 128 // (case.Hq // case.Hkv)
    edge = [[rb * case.R + off, (7 * rb + j) % case.Hq]
            for rb in range(case.MB) for j, off in enumerate((0, tr - 1, tr, case.R - 1))
            if rb * case.R + off < case.M]
    rows = np.concatenate([rows, edge, [[0, 0], [case.M - 1, case.Hq - 1]]])
    assert len(rows) > 1000
    y, l = oracle.bsr_rows(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                           case.R, case.C, case.sm_scale, rows)
    got = torch.stack([out[i, h] for i, h in rows])
    gl = torch.stack([lse[i, h] for i, h in rows])
    compare(got, gl, y, l, case.dtype)
    assert torch.isfinite(out.float()).all()


# ---------------------------------------------------------------------------
# tensor-core path (head_dim 64/128, C % 64 == 0, Hq/Hkv divides 128)

@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype,p", [
    (256, 256, 64, 64, 8, 2, 128, "f16", 0.5),      # G = 4, 32 rows per tile
    (190, 320, 64, 64, 8, 8, 128, "bf16", 0.4),     # G = 1, 128 rows per tile, ragged M
    (300, 256, 100, 128, 4, 2, 64, "f16", 0.5),     # G = 2, C = 2 x 64, R not a tile multiple
    (128, 384, 32, 64, 16, 2, 128, "bf16", 0.3),    # G = 8, 16 rows per tile
    (96, 192, 48, 64, 16, 1, 64, "f16", 0.6),       # G = 16, 8 rows per tile
])
def test_tensor_core_shapes(M, N, R, C, Hq, Hkv, d, dtype, p):
    case = synth.BsrCase("tc", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=p,
                         sm_scale=1 / math.sqrt(d), seed=55)
    x = synth.make_bsr_inputs(case)
    out, lse = run_bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                       case.sm_scale, dtype)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C, case.sm_scale)
    compare(out, lse, y, l, dtype)


def test_tensor_core_empty_block_rows():
    M, N, R, C = 256, 256, 64, 64
    indptr = torch.tensor([0, 3, 3, 4, 4], dtype=torch.int32)   # block rows 1 and 3 empty
    indices = torch.tensor([0, 2, 3, 1], dtype=torch.int32)
    q = synth.normal(8, 0, (M, 8, 128), "bf16")
    k = synth.normal(8, 1, (N, 2, 128), "bf16")
    v = synth.normal(8, 2, (N, 2, 128), "bf16")
    out, lse = run_bsr(q, k, v, indptr, indices, M, N, R, C, 0.09, "bf16")
    y, l = oracle.bsr(q, k, v, indptr, indices, M, N, R, C, 0.09)
    compare(out, lse, y, l, "bf16")
    assert torch.all(out[64:128] == 0) and torch.all(torch.isneginf(lse[192:256]))
    assert sfa.sfa_get_last_error() == sfa.SFA_OK


def test_tensor_core_large_scores_rescale():
    """Scores spanning a wide range exercise the conditional O rescale."""
    M, N, R, C = 128, 512, 64, 64
    indptr = torch.tensor([0, 8, 16], dtype=torch.int32)
    indices = torch.arange(8, dtype=torch.int32).repeat(2)
    q = (synth.normal(9, 0, (M, 4, 128), "f16").float() * 3).half()
    k = (synth.normal(9, 1, (N, 1, 128), "f16").float()
         * torch.linspace(0.2, 4.0, N).view(N, 1, 1)).half()
    v = synth.normal(9, 2, (N, 1, 128), "f16")
    out, lse = run_bsr(q, k, v, indptr, indices, M, N, R, C, 0.0884, "f16")
    y, l = oracle.bsr(q, k, v, indptr, indices, M, N, R, C, 0.0884)
    compare(out, lse, y, l, "f16")


# ---------------------------------------------------------------------------
# plan()'s per-element mask and causal, on both kernels (tensor cores: head_dim
# 64/128 with C % 64 == 0; register-tiled kernel otherwise)

def run_bsr_masked(q, k, v, indptr, indices, M, N, R, C, scale, dtype, mask=None, causal=False):
    Hq, d, Hkv = q.shape[1], q.shape[2], k.shape[1]
    plan = sfa.bsr_plan(indptr, indices, M, N, R, C, Hq, Hkv, d, sm_scale=scale, dtype=dtype,
                        mask=mask, causal=causal)
    out = torch.empty_like(q.cuda())
    lse = torch.empty((M, Hq), dtype=torch.float32, device="cuda")
    sfa.bsr_run(plan, q.cuda(), k.cuda(), v.cuda(), out, lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


MASK_SHAPES = [
    # M, N, R, C, Hq, Hkv, d, dtype
    (256, 256, 64, 64, 8, 2, 128, "f16"),     # tensor cores, G = 4
    (200, 256, 64, 128, 4, 4, 64, "bf16"),    # tensor cores, C = 2 x 64, ragged last row block
    (130, 192, 32, 64, 16, 1, 128, "bf16"),   # tensor cores, G = 16
    (97, 120, 16, 24, 6, 3, 192, "f16"),      # register-tiled kernel
    (64, 96, 8, 32, 2, 1, 64, "f16"),         # register-tiled kernel (C % 64 != 0)
]


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype", MASK_SHAPES)
@pytest.mark.parametrize("keep", [0.5, 0.05])
def test_element_mask(M, N, R, C, Hq, Hkv, d, dtype, keep):
    case = synth.BsrCase("m", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=0.4,
                         sm_scale=1 / math.sqrt(d), seed=81, mask_keep=keep)
    x = synth.make_bsr_inputs(case)
    out, lse = run_bsr_masked(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                              case.sm_scale, dtype, mask=x["mask"])
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                      case.sm_scale, mask=x["mask"])
    compare(out, lse, y, l, dtype)


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype", MASK_SHAPES)
def test_causal(M, N, R, C, Hq, Hkv, d, dtype):
    case = synth.BsrCase("c", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=0.5,
                         sm_scale=1 / math.sqrt(d), seed=82)
    x = synth.make_bsr_inputs(case)
    out, lse = run_bsr_masked(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                              case.sm_scale, dtype, causal=True)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                      case.sm_scale, causal=True)
    compare(out, lse, y, l, dtype)


def test_mask_wins_over_causal_and_masked_rows_are_zero():
    M, N, R, C, Hq, Hkv, d = 256, 256, 64, 64, 8, 2, 128
    case = synth.BsrCase("z", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype="f16", p=0.5,
                         sm_scale=1 / math.sqrt(d), seed=83, mask_keep=0.5)
    x = synth.make_bsr_inputs(case)
    mask = x["mask"].copy()
    mask[:, 5, :] = False          # row 5 of every block row: nothing visible
    out, lse = run_bsr_masked(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                              case.sm_scale, "f16", mask=mask, causal=True)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                      case.sm_scale, mask=mask)
    compare(out, lse, y, l, "f16")
    rows = np.arange(5, M, R)
    assert torch.all(out[rows] == 0) and torch.all(torch.isneginf(lse[rows]))


def test_causal_first_step_wholly_masked_for_top_rows():
    """Bottom-right causal with kv_len - qo_len = 200 and each block row's
    columns listed last to first: block row 0 keeps block 2 (keys 256..383,
    seen by its rows 56..63) and processes it first, so its rows 0..55 see
    nothing in their first step and their first allowed keys only in the
    next (P must be 0, not NaN, while a row's running max is still -inf)."""
    M, N, R, C, Hq, Hkv, d = 184, 384, 64, 128, 8, 2, 128
    case = synth.BsrCase("r", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype="f16", p=0.7,
                         sm_scale=1 / math.sqrt(d), seed=84)
    x = synth.make_bsr_inputs(case)
    ip = x["indptr"].numpy()
    ix = x["indices"].numpy().copy()
    for rb in range(len(ip) - 1):
        ix[ip[rb]:ip[rb + 1]] = ix[ip[rb]:ip[rb + 1]][::-1].copy()
    assert 2 in ix[ip[0]:ip[1]] and ix[ip[0]] == max(ix[ip[0]:ip[1]])
    ix_t = torch.from_numpy(ix)
    out, lse = run_bsr_masked(x["q"], x["k"], x["v"], x["indptr"], ix_t, M, N, R, C,
                              case.sm_scale, "f16", causal=True)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], ix_t, M, N, R, C, case.sm_scale,
                      causal=True)
    compare(out, lse, y, l, "f16")


def test_element_mask_first_blocks_hidden_from_top_rows():
    """The per-element mask hides each block row's first two stored blocks
    from its top half of rows, which then see their first allowed key only in
    a later step (P = 0 while a row's max is -inf); rows left with nothing
    are +0 with lse -inf."""
    M, N, R, C, Hq, Hkv, d = 256, 512, 64, 64, 8, 2, 128
    case = synth.BsrCase("f", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", p=0.5,
                         sm_scale=1 / math.sqrt(d), seed=85, mask_keep=0.5)
    x = synth.make_bsr_inputs(case)
    mask = x["mask"].copy()
    ip = x["indptr"].numpy()
    for rb in range(len(ip) - 1):
        for k in range(ip[rb], min(ip[rb] + 2, ip[rb + 1])):
            mask[k, : R // 2, :] = False
    out, lse = run_bsr_masked(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                              case.sm_scale, "bf16", mask=mask)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                      case.sm_scale, mask=mask)
    compare(out, lse, y, l, "bf16")


def test_masked_plan_reuse():
    """A masked plan stays valid for several runs on different inputs."""
    M, N, R, C, Hq, Hkv, d = 128, 192, 64, 64, 4, 1, 64
    case = synth.BsrCase("r", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype="bf16", p=0.6,
                         sm_scale=0.125, seed=84, mask_keep=0.7)
    x = synth.make_bsr_inputs(case)
    plan = sfa.bsr_plan(x["indptr"], x["indices"], M, N, R, C, Hq, Hkv, d, sm_scale=0.125,
                        dtype="bf16", mask=x["mask"])
    for seed in (1, 2):
        q = synth.normal(seed, 0, (M, Hq, d), "bf16")
        out = torch.empty_like(q.cuda())
        lse = torch.empty((M, Hq), dtype=torch.float32, device="cuda")
        sfa.bsr_run(plan, q.cuda(), x["k"].cuda(), x["v"].cuda(), out, lse)
        torch.cuda.synchronize()
        y, l = oracle.bsr(q, x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C, 0.125,
                          mask=x["mask"])
        compare(out.cpu(), lse.cpu(), y, l, "bf16")


# ---------------------------------------------------------------------------
# k / v in HND layout ("flashinfer.prefill.single_prefill_with_kv_cache",
# kv_layout): the same problem as with NHD tensors, k and v permuted to
# (num_kv_heads, N, head_dim); the oracle gets the NHD tensors.

HND_SHAPES = [
    # M, N, R, C, Hq, Hkv, d, dtype, mode
    (256, 384, 64, 64, 8, 2, 128, "f16", "plain"),     # 128-key tensor-core kernel
    (200, 256, 64, 128, 4, 4, 64, "bf16", "plain"),    # C = 2 x 64, ragged last row block
    (256, 320, 64, 64, 16, 2, 128, "bf16", "causal"),  # causal mode, N > M
    (130, 192, 32, 64, 16, 1, 128, "f16", "mask"),     # 64-key kernel, per-element mask
    (97, 120, 16, 24, 6, 3, 192, "f16", "plain"),      # register-tiled kernel
    (64, 96, 8, 32, 2, 1, 64, "bf16", "mask"),         # register-tiled kernel with a mask
]


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype,mode", HND_SHAPES)
def test_hnd_kv_layout(M, N, R, C, Hq, Hkv, d, dtype, mode):
    case = synth.BsrCase("h", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=0.45,
                         sm_scale=1 / math.sqrt(d), seed=91, mask_keep=0.5 if mode == "mask" else 0.0)
    x = synth.make_bsr_inputs(case)
    causal = mode == "causal"
    plan = sfa.bsr_plan(x["indptr"], x["indices"], M, N, R, C, Hq, Hkv, d, sm_scale=case.sm_scale,
                        dtype=dtype, causal=causal, mask=x["mask"], kv_layout="HND")
    k_hnd = x["k"].permute(1, 0, 2).contiguous().cuda()
    v_hnd = x["v"].permute(1, 0, 2).contiguous().cuda()
    q = x["q"].cuda()
    out = torch.empty_like(q)
    lse = torch.empty((M, Hq), dtype=torch.float32, device="cuda")
    sfa.bsr_run(plan, q, k_hnd, v_hnd, out, lse)
    torch.cuda.synchronize()
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C,
                      case.sm_scale, mask=x["mask"], causal=causal)
    compare(out.cpu(), lse.cpu(), y, l, dtype)
    # the same plan switched back to NHD reads the original tensors
    sfa.bsr_plan_set_kv_layout(plan, "NHD")
    out2 = torch.empty_like(q)
    sfa.bsr_run(plan, q, x["k"].cuda(), x["v"].cuda(), out2, lse)
    torch.cuda.synchronize()
    compare(out2.cpu(), lse.cpu(), y, l, dtype)
    assert sfa.load().bsr_plan_set_kv_layout(plan.handle, 2) == sfa.SFA_ERR_INVALID_ARG
