"""GPU parity of plan()'s logits_soft_cap (both block-sparse wrappers) against
the CPU oracle, on every block-sparse kernel: the 128-key tensor-core kernel
(plain, causal, variable), the 64-key kernel (per-element mask) and the
register-tiled kernel (other head dims)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_serving_sfa_gb300 as sfa
import synth
from tests.test_gpu_bsr import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    sfa.build()
    sfa.load()


def run(case, x, cap, plan=None):
    if plan is None:
        plan = sfa.bsr_plan(x["indptr"], x["indices"], case.M, case.N, case.R, case.C, case.Hq,
                            case.Hkv, case.d, sm_scale=case.sm_scale, dtype=case.dtype,
                            causal=case.causal, mask=x["mask"], logits_soft_cap=cap)
    out = torch.empty_like(x["q"].cuda())
    lse = torch.empty((case.M, case.Hq), dtype=torch.float32, device="cuda")
    sfa.bsr_run(plan, x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), out, lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


SHAPES = [
    # M, N, R, C, Hq, Hkv, d, dtype, causal, mask_keep    (kernel)
    (256, 320, 64, 64, 8, 2, 128, "f16", False, 0.0),     # 128-key, plain, odd block count rows
    (200, 256, 64, 64, 8, 2, 128, "bf16", True, 0.0),     # 128-key, causal
    (256, 256, 64, 128, 4, 4, 64, "f16", False, 0.5),     # 64-key, per-element mask
    (97, 120, 16, 24, 6, 3, 192, "bf16", False, 0.0),     # register-tiled
]


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,d,dtype,causal,keep", SHAPES)
@pytest.mark.parametrize("cap", [0.6, 20.0])
def test_bsr_soft_cap(M, N, R, C, Hq, Hkv, d, dtype, causal, keep, cap):
    c = synth.BsrCase("c", M=M, N=N, R=R, C=C, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=0.5,
                      sm_scale=1.5 / math.sqrt(d), seed=61, causal=causal, mask_keep=keep)
    x = synth.make_bsr_inputs(c)
    out, lse = run(c, x, cap)
    y, l = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, R, C, c.sm_scale,
                      mask=x["mask"], causal=causal, softcap=cap)
    compare(out, lse, y, l, dtype)


def test_soft_cap_set_and_cleared_on_a_plan():
    c = synth.BsrCase("r", M=128, N=192, R=64, C=64, Hq=8, Hkv=2, d=128, dtype="f16", p=0.6,
                      sm_scale=0.2, seed=62)
    x = synth.make_bsr_inputs(c)
    plan = sfa.bsr_plan(x["indptr"], x["indices"], c.M, c.N, c.R, c.C, c.Hq, c.Hkv, c.d,
                        sm_scale=c.sm_scale, dtype="f16")
    args = (x["q"], x["k"], x["v"], x["indptr"], x["indices"], c.M, c.N, c.R, c.C, c.sm_scale)
    sfa.bsr_plan_set_logits_soft_cap(plan, 1.0)
    out, lse = run(c, x, 0.0, plan=plan)
    y, l = oracle.bsr(*args, softcap=1.0)
    compare(out, lse, y, l, "f16")
    for bad in (float("nan"), float("inf")):
        with pytest.raises(sfa.SfaError):
            sfa.bsr_plan_set_logits_soft_cap(plan, bad)
    sfa.bsr_plan_set_logits_soft_cap(plan, 0.0)
    out, lse = run(c, x, 0.0, plan=plan)
    y, l = oracle.bsr(*args)
    compare(out, lse, y, l, "f16")


@pytest.mark.parametrize("causal", [False, True])
def test_varbsr_soft_cap(causal):
    c = synth.VarBsrCase("v", M=300, N=500, MB=7, NB=9, Hq=8, Hkv=2, d=128, dtype="bf16", p=0.4,
                         sm_scale=0.15, seed=63, causal=causal)
    x = synth.make_varbsr_inputs(c)
    plan = sfa.varbsr_plan(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"], c.Hq,
                           c.Hkv, c.d, causal=causal, sm_scale=c.sm_scale, dtype=c.dtype,
                           logits_soft_cap=2.5)
    q = x["q"].cuda()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    sfa.varbsr_run(plan, q, x["k"].cuda(), x["v"].cuda(), out, lse)
    torch.cuda.synchronize()
    y, l = oracle.varbsr(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                         x["block_col_sz"], c.sm_scale, causal=causal, softcap=2.5)
    compare(out.cpu(), lse.cpu(), y, l, c.dtype)
