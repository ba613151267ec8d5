"""Pins of the oracle's logits soft cap ("flashinfer.sparse", plan()'s
logits_soft_cap in BlockSparseAttentionWrapper and
VariableBlockSparseAttentionWrapper: a logit x becomes cap * tanh(x / cap)),
each against a dense brute force written here or an exactly known limit."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.test_oracle_bsr_mask import _dense_allowed
from tests.test_oracle_varbsr import _element_mask


def _dense_capped(q, k, v, allowed, scale, cap):
    """NHD q (M,Hq,d), k/v (N,Hkv,d); allowed (M,N): masked softmax over the
    soft-capped scaled logits, fp64."""
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    M, Hq, d = qf.shape
    G = Hq // kf.shape[1]
    y = np.zeros((M, Hq, d))
    lse = np.full((M, Hq), -np.inf)
    for h in range(Hq):
        x = qf[:, h, :] @ kf[:, h // G, :].T * scale
        x = cap * np.tanh(x / cap)
        x = np.where(allowed, x, -np.inf)
        for i in range(M):
            if not allowed[i].any():
                continue
            m = x[i].max()
            w = np.exp(x[i] - m)
            y[i, h] = (w / w.sum()) @ vf[:, h // G, :]
            lse[i, h] = m + np.log(w.sum())
    return y, lse


def _case(**kw):
    base = dict(name="s", M=80, N=96, R=16, C=32, Hq=4, Hkv=2, d=16, dtype="f16", p=0.6,
                sm_scale=0.9, seed=71)
    base.update(kw)
    return synth.BsrCase(**base)


@pytest.mark.parametrize("variant", ["plain", "causal", "mask"])
@pytest.mark.parametrize("cap", [0.7, 5.0])
def test_bsr_matches_dense_brute_force(variant, cap):
    c = _case(causal=variant == "causal", mask_keep=0.5 if variant == "mask" else 0.0)
    x = synth.make_bsr_inputs(c)
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], c.M, c.N, c.R, c.C,
                        c.sm_scale, mask=x["mask"], causal=c.causal, softcap=cap)
    allowed = _dense_allowed(x["indptr"], x["indices"], c.M, c.N, c.R, c.C, x["mask"], c.causal)
    ye, le = _dense_capped(x["q"], x["k"], x["v"], allowed, c.sm_scale, cap)
    np.testing.assert_allclose(y, ye, rtol=1e-11, atol=1e-12)
    fin = np.isfinite(le)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], le[fin], rtol=1e-11)


def test_large_cap_is_no_cap():
    c = _case()
    x = synth.make_bsr_inputs(c)
    args = (x["q"], x["k"], x["v"], x["indptr"], x["indices"], c.M, c.N, c.R, c.C, c.sm_scale)
    y0, l0 = oracle.bsr(*args)
    y1, l1 = oracle.bsr(*args, softcap=1e9)
    np.testing.assert_allclose(y1, y0, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-9)


def test_tiny_cap_gives_mean_of_allowed_values():
    """cap -> 0: every capped logit is within cap of 0, so the weights are
    uniform over the allowed keys: y = mean of their values, lse = ln(count)."""
    c = _case(M=32, N=64, R=16, C=16, Hq=2, Hkv=1, d=8, p=0.5)
    x = synth.make_bsr_inputs(c)
    y, lse = oracle.bsr(x["q"], x["k"], x["v"], x["indptr"], x["indices"], c.M, c.N, c.R, c.C,
                        c.sm_scale, softcap=1e-12)
    allowed = _dense_allowed(x["indptr"], x["indices"], c.M, c.N, c.R, c.C)
    vf = x["v"].double().numpy()[:, 0, :]
    for i in range(c.M):
        n = int(allowed[i].sum())
        for h in range(c.Hq):
            np.testing.assert_allclose(y[i, h], vf[allowed[i]].mean(0), rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(lse[i, h], math.log(n), rtol=1e-9)


def test_rows_entry_matches_full():
    c = _case(causal=True)
    x = synth.make_bsr_inputs(c)
    args = (x["q"], x["k"], x["v"], x["indptr"], x["indices"], c.M, c.N, c.R, c.C, c.sm_scale)
    y, lse = oracle.bsr(*args, causal=True, softcap=2.0)
    rows = np.array([[0, 0], [17, 3], [c.M - 1, c.Hq - 1]])
    yr, lr = oracle.bsr_rows(*args, rows, causal=True, softcap=2.0)
    np.testing.assert_array_equal(yr, np.stack([y[i, h] for i, h in rows]))
    np.testing.assert_array_equal(lr, np.array([lse[i, h] for i, h in rows]))


@pytest.mark.parametrize("causal", [False, True])
def test_varbsr_matches_dense_brute_force(causal):
    c = synth.VarBsrCase("v", M=37, N=45, MB=5, NB=6, Hq=4, Hkv=2, d=16, dtype="bf16", p=0.5,
                         sm_scale=0.8, seed=73, causal=causal)
    x = synth.make_varbsr_inputs(c)
    y, lse = oracle.varbsr(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                           x["block_col_sz"], c.sm_scale, causal=causal, softcap=1.5)
    allowed = _element_mask(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"])
    G = c.Hq // c.Hkv
    for g in range(c.Hkv):
        a = allowed[g].copy()
        if causal:
            a &= np.arange(c.N)[None, :] <= np.arange(c.M)[:, None] + (c.N - c.M)
        # HND -> NHD slices of this kv head's qo heads
        qn = x["q"][g * G:(g + 1) * G].permute(1, 0, 2)
        kn = x["k"][g:g + 1].permute(1, 0, 2)
        vn = x["v"][g:g + 1].permute(1, 0, 2)
        ye, le = _dense_capped(qn, kn, vn, a, c.sm_scale, 1.5)
        np.testing.assert_allclose(y[g * G:(g + 1) * G], ye.transpose(1, 0, 2), rtol=1e-11,
                                   atol=1e-12)
        fin = np.isfinite(le.T)
        np.testing.assert_allclose(lse[g * G:(g + 1) * G][fin], le.T[fin], rtol=1e-11)
    yr, lr = oracle.varbsr_rows(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                                x["block_col_sz"], c.sm_scale, [0, 5, c.Hq * c.M - 1],
                                causal=causal, softcap=1.5)
    np.testing.assert_array_equal(yr, y.reshape(-1, c.d)[[0, 5, c.Hq * c.M - 1]])
