"""Pins of the oracle's block-sparse mask and causal readings
("flashinfer.sparse", BlockSparseAttentionWrapper.plan(): mask (nnz, R, C),
packed_mask, causal), each against a dense brute force written here or an
exactly known result."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _dense_allowed(indptr, indices, M, N, R, C, mask=None, causal=False):
    """Dense (M, N) bool: stored blocks, then the per-element mask or causal."""
    allowed = np.zeros((M, N), dtype=bool)
    ip, ix = indptr.numpy(), indices.numpy()
    for br in range((M + R - 1) // R):
        r0, r1 = br * R, min(M, (br + 1) * R)
        for k in range(ip[br], ip[br + 1]):
            c0 = int(ix[k]) * C
            if mask is None:
                allowed[r0:r1, c0:c0 + C] = True
            else:
                allowed[r0:r1, c0:c0 + C] = mask[k][: r1 - r0]
    if mask is None and causal:
        i = np.arange(M)[:, None]
        j = np.arange(N)[None, :]
        allowed &= j <= i + (N - M)
    return allowed


def _dense_attention(q, k, v, allowed, scale):
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    M, Hq, d = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    y = np.zeros((M, Hq, d))
    lse = np.full((M, Hq), -np.inf)
    for h in range(Hq):
        s = qf[:, h, :] @ kf[:, h // G, :].T * scale
        s = np.where(allowed, s, -np.inf)
        for i in range(M):
            if not allowed[i].any():
                continue
            m = s[i].max()
            w = np.exp(s[i] - m)
            y[i, h] = (w / w.sum()) @ vf[:, h // G, :]
            lse[i, h] = m + np.log(w.sum())
    return y, lse


def _case(**kw):
    base = dict(name="m", M=96, N=128, R=16, C=32, Hq=4, Hkv=2, d=16, dtype="f16", p=0.5,
                sm_scale=0.25, seed=99)
    base.update(kw)
    return synth.BsrCase(**base)


def _inputs(case):
    return synth.make_bsr_inputs(case)


def test_full_mask_equals_no_mask():
    case = _case()
    x = _inputs(case)
    nnz = int(x["indptr"][-1])
    full = np.ones((nnz, case.R, case.C), dtype=bool)
    a = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N, case.R,
                   case.C, case.sm_scale)
    b = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N, case.R,
                   case.C, case.sm_scale, mask=full)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("M,N", [(128, 128), (96, 128), (100, 160)])
def test_causal_matches_dense_bottom_right(M, N):
    case = _case(M=M, N=N)
    x = _inputs(case)
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], M, N, case.R, case.C,
                        case.sm_scale, causal=True)
    allowed = _dense_allowed(x["indptr"], x["indices"], M, N, case.R, case.C, causal=True)
    ry, rl = _dense_attention(x["q"], x["k"], x["v"], allowed, case.sm_scale)
    np.testing.assert_allclose(y, ry, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("keep", [0.3, 0.9])
def test_mask_matches_dense(keep):
    case = _case(mask_keep=keep, M=100)
    x = _inputs(case)
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                        case.R, case.C, case.sm_scale, mask=x["mask"])
    allowed = _dense_allowed(x["indptr"], x["indices"], case.M, case.N, case.R, case.C,
                             mask=x["mask"])
    ry, rl = _dense_attention(x["q"], x["k"], x["v"], allowed, case.sm_scale)
    np.testing.assert_allclose(y, ry, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


def test_mask_overrides_causal():
    case = _case(mask_keep=0.5)
    x = _inputs(case)
    a = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N, case.R,
                   case.C, case.sm_scale, mask=x["mask"])
    b = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N, case.R,
                   case.C, case.sm_scale, mask=x["mask"], causal=True)
    np.testing.assert_array_equal(a[0], b[0])


def test_packed_bit_order_most_significant_first():
    """One stored block (1 x 8 elements), packed byte 0x40: only element 1
    (column 1) is allowed, so row 0 returns v[1] exactly."""
    q = torch.randn(1, 1, 8).half()
    k = torch.randn(8, 1, 8).half()
    v = torch.randn(8, 1, 8).half()
    indptr = torch.tensor([0, 1], dtype=torch.int32)
    indices = torch.tensor([0], dtype=torch.int32)
    y, _ = oracle.bsr(q, k, v, indptr, indices, 1, 8, 1, 8, 0.5,
                      packed_mask=np.array([0x40], dtype=np.uint8))
    np.testing.assert_array_equal(y[0, 0], v[1, 0].double().numpy())
    assert oracle.pack_mask(np.array([[[0, 1, 0, 0, 0, 0, 0, 0]]], dtype=bool))[0] == 0x40


def test_fully_masked_rows_zero():
    case = _case(mask_keep=0.5)
    x = _inputs(case)
    mask = x["mask"].copy()
    # rows 0 .. R-1 (block row 0) see nothing
    ip = x["indptr"].numpy()
    mask[ip[0]:ip[1]] = False
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                        case.R, case.C, case.sm_scale, mask=mask)
    assert np.all(y[: case.R] == 0.0)
    assert np.all(np.isneginf(lse[: case.R]))


def test_rows_entry_agrees_with_full():
    case = _case(mask_keep=0.6)
    x = _inputs(case)
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                        case.R, case.C, case.sm_scale, mask=x["mask"])
    rows = np.array([[0, 0], [17, 3], [95, 1]])
    yr, lr = oracle.bsr_rows(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M, case.N,
                             case.R, case.C, case.sm_scale, rows, mask=x["mask"])
    for n, (i, h) in enumerate(rows):
        np.testing.assert_array_equal(yr[n], y[i, h])
        assert lr[n] == lse[i, h]


@pytest.mark.parametrize("kind", ["plain", "causal", "mask"])
def test_work_counts_match_dense_allowed(kind):
    """The benchmark's useful-FLOP count is the number of allowed (row, key)
    pairs of the same dense mask the pins above use."""
    case = _case(M=100, N=160, causal=(kind == "causal"), mask_keep=(0.4 if kind == "mask" else 0))
    x = _inputs(case)
    counts = synth.bsr_counts(case, x["indptr"], x["indices"], x["mask"])
    allowed = _dense_allowed(x["indptr"], x["indices"], case.M, case.N, case.R, case.C,
                             mask=x["mask"], causal=case.causal)
    assert counts["allowed"] == int(allowed.sum())
    assert counts["flops"] == 4 * case.d * int(allowed.sum()) * case.Hq
