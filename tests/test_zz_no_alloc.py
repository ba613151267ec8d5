"""sfa_run_noalloc: the entry point for callers that cannot allocate device
memory (for example a serving engine that reserved nearly all HBM for its KV
cache up front, or a plugin host that forbids libraries from allocating).  It
keeps its split partials in a fixed device array inside the library instead
of an allocated workspace.  These tests call it through the C ABI and check
its output against sfa_run's on the same inputs, on consecutive calls (the
array keeps the previous call's contents), and that a shape needing more
scratch than the array holds is rejected.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_serving_sfa_gb300 as sfa
import synth
from tests import sfa_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    sfa.build()
    sfa.load()


def call(fn, case, dev, out, lse):
    return fn(dev["q"], dev["k"], dev["v"], dev["idx"], case.B, case.S1, case.S2, case.N1,
              case.N2, case.Dk, case.Dv, case.topK, case.scale, case.layout, case.causal,
              case.dtype, out, lse, None, check=False)


def outputs(case, dev):
    shape = ((case.B, case.S1, case.N1, case.Dv) if case.layout == "BSND"
             else (case.B, case.N1, case.S1, case.Dv))
    lshape = shape[:3]
    return (torch.empty(shape, dtype=dev["q"].dtype, device="cuda"),
            torch.empty(lshape, dtype=torch.float32, device="cuda"))


def same_within_tolerance(case, out_a, lse_a, out_b, lse_b):
    rep = oracle.precision_report(out_a.float().cpu().numpy(), out_b.float().cpu().numpy(),
                                  case.dtype, round_golden=False)
    assert rep["passed"], rep
    la, lb = lse_a.cpu().numpy(), lse_b.cpu().numpy()
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(la[fin], lb[fin], atol=T.LSE_ATOL, rtol=T.LSE_RTOL)


CASES = [
    synth.GQA_DECODE,       # splits > 1: partials go through the scratch array
    synth.SfaCase("noalloc_causal", B=2, S1=16, S2=64, N1=8, N2=2, Dk=192, Dv=128, topK=40,
                  dtype="f16", layout="BSND", causal=True, scale=0.07,
                  value_is_key_prefix=True, index_kind="causal_mix", masked_frac=0.1,
                  full_masked_rows=4, seed=99),
]


def test_noalloc_matches_sfa_run_on_consecutive_calls():
    prepared = []
    for case in CASES:
        dev = T.to_dev(synth.make_sfa_inputs(case))
        ref_out, ref_lse = outputs(case, dev)
        assert call(sfa.sfa_run, case, dev, ref_out, ref_lse) == sfa.SFA_OK
        prepared.append((case, dev, ref_out, ref_lse))
    torch.cuda.synchronize()
    # two calls in a row per case, alternating cases so the array always holds
    # the other shape's partials when a call starts
    for _ in range(2):
        for case, dev, ref_out, ref_lse in prepared:
            out, lse = outputs(case, dev)
            out.fill_(7.0)
            lse.fill_(7.0)
            assert call(sfa.sfa_run_noalloc, case, dev, out, lse) == sfa.SFA_OK
            torch.cuda.synchronize()
            same_within_tolerance(case, out, lse, ref_out, ref_lse)


def test_noalloc_rejects_shapes_beyond_the_array():
    case = synth.MLA_DECODE.replace(B=4)
    need = sfa.sfa_workspace_size(case.B, case.S1, case.N1, case.N2, case.Dk, case.Dv, case.topK)
    assert need > sfa.SFA_NOALLOC_SCRATCH_BYTES
    dev = T.to_dev(synth.make_sfa_inputs(case))
    out, lse = outputs(case, dev)
    out.fill_(7.0)
    assert call(sfa.sfa_run_noalloc, case, dev, out, lse) == sfa.SFA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)          # nothing was launched
