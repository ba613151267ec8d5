"""Shared helpers of the GPU parity tests: run a workload through the C ABI
and compare with the CPU oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
import sparse_attention_serving_sfa_gb300 as sfa
import synth

LSE_ATOL = 1e-3
LSE_RTOL = 1e-4


def to_dev(d):
    """Device copies; a prefix-view value stays a view of the device key."""
    out = {"q": d["q"].cuda(), "k": d["k"].cuda(), "idx": d["idx"].cuda()}
    if d["v"].data_ptr() == d["k"].data_ptr():
        out["v"] = out["k"][..., : d["v"].shape[-1]]
    else:
        out["v"] = d["v"].cuda()
    return out


def run_gpu(case, dev, **opts):
    out, lse = sfa.sparse_flash_attention(dev["q"], dev["k"], dev["v"], dev["idx"], case.scale,
                                          case.layout, case.causal, return_lse=True, **opts)
    torch.cuda.synchronize()
    return out, lse


def check_full(case, d, out, lse):
    """Element-by-element comparison of every output row."""
    y, l = oracle.sfa(d["q"], d["k"], d["v"], d["idx"], case.scale, case.layout, case.causal)
    a = out.float().cpu().numpy()
    rep = oracle.precision_report(a, y, case.dtype)
    assert rep["passed"], rep
    lg = lse.cpu().numpy().astype(np.float64)
    masked = np.isneginf(l)
    assert np.array_equal(np.isneginf(lg), masked), "fully masked rows differ"
    np.testing.assert_allclose(lg[~masked], l[~masked], atol=LSE_ATOL, rtol=LSE_RTOL)
    # fully masked rows: exactly +0
    if masked.any():
        rows = a[masked] if case.layout == "BSND" else a[masked]
        assert np.all(rows == 0.0) and not np.signbit(rows).any()
    return rep


def sample_rows(case, n, seed=0):
    """n distinct (b, n1, s1) rows, always including the first and last."""
    total = case.B * case.N1 * case.S1
    rng = np.random.default_rng(seed)
    flat = np.unique(np.concatenate([[0, total - 1], rng.choice(total, size=min(n, total),
                                                                  replace=False)]))
    b = flat // (case.N1 * case.S1)
    n1 = (flat // case.S1) % case.N1
    s1 = flat % case.S1
    return np.stack([b, n1, s1], axis=1)


def check_rows(case, d, out, lse, rows):
    """Comparison on sampled rows the oracle computes one by one."""
    y, l = oracle.sfa_rows(d["q"], d["k"], d["v"], d["idx"], case.scale, rows, case.layout,
                           case.causal)
    o = out.cpu()
    lg = lse.cpu()
    if case.layout == "BSND":
        got = np.stack([o[b, s1, n1].float().numpy() for b, n1, s1 in rows])
        gl = np.array([float(lg[b, s1, n1]) for b, n1, s1 in rows])
    else:
        got = np.stack([o[b, n1, s1].float().numpy() for b, n1, s1 in rows])
        gl = np.array([float(lg[b, n1, s1]) for b, n1, s1 in rows])
    rep = oracle.precision_report(got, y, case.dtype)
    assert rep["passed"], rep
    masked = np.isneginf(l)
    assert np.array_equal(np.isneginf(gl), masked)
    np.testing.assert_allclose(gl[~masked], l[~masked], atol=LSE_ATOL, rtol=LSE_RTOL)
    if masked.any():
        assert np.all(got[masked] == 0.0) and not np.signbit(got[masked]).any()
    return rep
