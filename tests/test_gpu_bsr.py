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
    rows = np.concatenate([rows, [[0, 0], [case.M - 1, case.Hq - 1]]])
    y, l = oracle.bsr_rows(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                           case.R, case.C, case.sm_scale, rows)
    got = torch.stack([out[i, h] for i, h in rows])
    gl = torch.stack([lse[i, h] for i, h in rows])
    compare(got, gl, y, l, case.dtype)
    assert torch.isfinite(out.float()).all()
