"""sfa_run_noalloc: the entry point for callers that cannot allocate device
memory (for example a serving engine that reserved nearly all HBM for its KV
cache up front, or a plugin host that forbids libraries from allocating).  It
keeps its split partials in a fixed device array inside the library instead
of an allocated workspace.  These tests call it through the C ABI and check
its output against sfa_run's and against the CPU oracle on the same inputs,
on consecutive calls of shapes whose partials differ (the array keeps the
previous call's contents), and that a shape needing more scratch than the
array holds is rejected.

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


def generic_splits(case, num_sms):
    """Split count of the generic kernel's plan as the header documents it:
    about two CTAs per SM (one CTA per 4 query heads, or per 8 when the group
    is larger than 4), at most min(ceil(topK / 64), 32) splits of whole
    32-slot chunks."""
    hb = 8 if case.G > 4 else 4
    ctas = case.B * case.N2 * case.S1 * (-(-case.G // hb))
    want = min(-(-2 * num_sms // ctas), min(-(-case.topK // 64), 32))
    per = -(-case.topK // max(want, 1))
    per = -(-per // 32) * 32
    return -(-case.topK // per)


# Three shapes, each with splits > 1, called in turn: every call finds the
# previous shape's partials (other rows, Dv or values) in the array, so a
# partial the kernel failed to write would show up as a mismatch.
CASES = [
    synth.GQA_DECODE,
    synth.SfaCase("noalloc_small_dv", B=1, S1=2, S2=900, N1=4, N2=2, Dk=128, Dv=64, topK=512,
                  dtype="f16", layout="BSND", causal=True, scale=0.09,
                  index_kind="causal_mix", masked_frac=0.1, full_masked_rows=1, seed=99),
    synth.GQA_DECODE.replace(name="gqa_decode_other_values", seed=777),
]


def test_cases_use_the_scratch_array():
    num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    for case in CASES:
        assert generic_splits(case, num_sms) > 1, case.name
    rows = {(c.B * c.S1 * c.N1, c.Dv) for c in CASES[:2]}
    assert len(rows) == 2


def test_noalloc_matches_sfa_run_and_the_oracle_on_consecutive_calls():
    prepared = []
    for case in CASES:
        host = synth.make_sfa_inputs(case)
        dev = T.to_dev(host)
        ref_out, ref_lse = outputs(case, dev)
        assert call(sfa.sfa_run, case, dev, ref_out, ref_lse) == sfa.SFA_OK
        prepared.append((case, host, dev, ref_out, ref_lse))
    torch.cuda.synchronize()
    # two rounds over the three shapes: two calls in a row of each entry
    for rnd in range(2):
        for case, host, dev, ref_out, ref_lse in prepared:
            out, lse = outputs(case, dev)
            out.fill_(7.0)
            lse.fill_(7.0)
            assert call(sfa.sfa_run_noalloc, case, dev, out, lse) == sfa.SFA_OK
            torch.cuda.synchronize()
            same_within_tolerance(case, out, lse, ref_out, ref_lse)
            if rnd == 0:
                T.check_full(case, host, out, lse)


def test_noalloc_rejects_shapes_beyond_the_array():
    case = synth.MLA_DECODE.replace(B=4)
    rows = case.B * case.S1 * case.N1
    need = rows * min(-(-case.topK // 64), 32) * (case.Dv + 2) * 4
    assert need > sfa.SFA_NOALLOC_SCRATCH_BYTES
    dev = T.to_dev(synth.make_sfa_inputs(case))
    out, lse = outputs(case, dev)
    out.fill_(7.0)
    assert call(sfa.sfa_run_noalloc, case, dev, out, lse) == sfa.SFA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)          # nothing was launched
