"""Pins of the oracle's variable block-sparse form ("flashinfer.sparse",
VariableBlockSparseAttentionWrapper: per-kv-head block mask map, per-kv-head
row and column block sizes, HND tensors), each against a dense brute force
written here, the page's worked example or an exactly known result."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.golden import fixtures


def _element_mask(mask_map, row_sz, col_sz):
    """(Hkv, M, N) bool: block (rb, cb) of kv head g spread over its rows and
    columns with np.repeat."""
    out = []
    for g in range(mask_map.shape[0]):
        m = np.repeat(np.asarray(mask_map[g], bool), np.asarray(row_sz[g]), axis=0)
        out.append(np.repeat(m, np.asarray(col_sz[g]), axis=1))
    return np.stack(out)


def _dense(q, k, v, allowed, scale, causal=False):
    """Masked softmax attention in fp64 over HND tensors; allowed (Hkv, M, N)."""
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    Hq, M, d = qf.shape
    Hkv, N = kf.shape[0], kf.shape[1]
    G = Hq // Hkv
    y = np.zeros((Hq, M, d))
    lse = np.full((Hq, M), -np.inf)
    for h in range(Hq):
        a = allowed[h // G].copy()
        if causal:
            a &= np.arange(N)[None, :] <= np.arange(M)[:, None] + (N - M)
        s = np.where(a, qf[h] @ kf[h // G].T * scale, -np.inf)
        for i in range(M):
            if not a[i].any():
                continue
            m = s[i].max()
            w = np.exp(s[i] - m)
            y[h, i] = (w / w.sum()) @ vf[h // G]
            lse[h, i] = m + np.log(w.sum())
    return y, lse


def _case(**kw):
    base = dict(name="v", M=37, N=45, MB=5, NB=6, Hq=4, Hkv=2, d=16, dtype="f16", p=0.5,
                sm_scale=0.3, seed=77)
    base.update(kw)
    return synth.VarBsrCase(**base)


def test_worked_example_expands_as_printed():
    """The page's example: the oracle's block expansion equals the dense mask
    expanded by hand from the plan() parameter definitions."""
    ex = fixtures.varbsr_example()
    S, d = ex["seq_len"], 16
    q = synth.normal(5, 0, (1, S, d), "f16")
    k = synth.normal(5, 1, (1, S, d), "f16")
    v = synth.normal(5, 2, (1, S, d), "f16")
    scale = 1.0 / math.sqrt(d)
    y, lse = oracle.varbsr(q, k, v, ex["block_mask_map"], ex["block_row_sz"], ex["block_col_sz"],
                           scale)
    ye, le = _dense(q, k, v, ex["mask"][None], scale)
    np.testing.assert_allclose(y, ye, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, le, rtol=1e-12, atol=1e-12)
    # the np.repeat expansion used by the other pins agrees with the hand expansion
    assert (_element_mask(ex["block_mask_map"], ex["block_row_sz"], ex["block_col_sz"])[0]
            == ex["mask"]).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matches_dense_brute_force(causal, dtype):
    c = _case(dtype=dtype, causal=causal)
    x = synth.make_varbsr_inputs(c)
    y, lse = oracle.varbsr(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                           x["block_col_sz"], c.sm_scale, causal=causal)
    allowed = _element_mask(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"])
    ye, le = _dense(x["q"], x["k"], x["v"], allowed, c.sm_scale, causal)
    np.testing.assert_allclose(y, ye, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, le, rtol=1e-11, atol=1e-12)


def test_kv_heads_keep_their_own_masks():
    """Two kv heads with complementary masks and different block sizes: qo
    heads 0, 1 read kv head 0 and heads 2, 3 kv head 1 (h / (Hq / Hkv))."""
    c = _case(M=12, N=10, MB=2, NB=2, Hq=4, Hkv=2)
    x = synth.make_varbsr_inputs(c)
    mm = np.array([[[1, 0], [0, 1]], [[0, 1], [1, 0]]], bool)
    rs = np.array([[5, 7], [9, 3]], np.int32)
    cs = np.array([[4, 6], [2, 8]], np.int32)
    y, _ = oracle.varbsr(x["q"], x["k"], x["v"], mm, rs, cs, c.sm_scale)
    ye, _ = _dense(x["q"], x["k"], x["v"], _element_mask(mm, rs, cs), c.sm_scale)
    np.testing.assert_allclose(y, ye, rtol=1e-11, atol=1e-12)
    # row 0 of qo head 0 sees only keys 0..3 (kv head 0, block (0, 0))
    vf = x["v"].double().numpy()
    s = x["q"][0, 0].double().numpy() @ x["k"][0, :4].double().numpy().T * c.sm_scale
    w = np.exp(s - s.max())
    np.testing.assert_allclose(y[0, 0], (w / w.sum()) @ vf[0, :4], rtol=1e-12, atol=1e-12)


def test_single_block_equals_dense_sdpa():
    """One block covering everything: plain (full or causal) attention."""
    for causal in (False, True):
        c = _case(M=20, N=20, MB=1, NB=1, Hq=2, Hkv=1, d=8, causal=causal)
        x = synth.make_varbsr_inputs(c)
        y, _ = oracle.varbsr(x["q"], x["k"], x["v"], np.ones((1, 1, 1), bool),
                             np.array([[20]], np.int32), np.array([[20]], np.int32), c.sm_scale,
                             causal=causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            x["q"].double()[None], x["k"].double().expand(2, -1, -1)[None],
            x["v"].double().expand(2, -1, -1)[None], is_causal=causal, scale=c.sm_scale)[0]
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_empty_blocks_and_fully_masked_rows():
    """Zero-size row and column blocks are allowed; a row whose row block has
    no set block gives y = 0 and lse = -inf."""
    c = _case(M=6, N=8, MB=3, NB=3, Hq=1, Hkv=1, d=8)
    x = synth.make_varbsr_inputs(c)
    mm = np.array([[[0, 0, 1], [1, 1, 1], [0, 0, 0]]], bool)
    rs = np.array([[2, 0, 4]], np.int32)
    cs = np.array([[3, 0, 5]], np.int32)
    y, lse = oracle.varbsr(x["q"], x["k"], x["v"], mm, rs, cs, c.sm_scale)
    assert (y[0, 2:] == 0).all() and np.isneginf(lse[0, 2:]).all()
    ye, le = _dense(x["q"], x["k"], x["v"], _element_mask(mm, rs, cs), c.sm_scale)
    np.testing.assert_allclose(y, ye, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse[0, :2], le[0, :2], rtol=1e-11)


def test_uniform_keys_give_mean_of_allowed_values():
    """Equal keys: the weights are uniform over the allowed columns, so y is the
    plain mean of those value rows (closed form)."""
    M, N, d = 4, 9, 8
    q = synth.normal(3, 0, (1, M, d), "f16")
    k = torch.ones((1, N, d), dtype=torch.float16)
    v = synth.normal(3, 2, (1, N, d), "f16")
    mm = np.array([[[1, 0, 1], [0, 1, 0]]], bool)
    rs = np.array([[1, 3]], np.int32)
    cs = np.array([[2, 3, 4]], np.int32)
    y, _ = oracle.varbsr(q, k, v, mm, rs, cs, 0.5)
    vf = v.double().numpy()[0]
    np.testing.assert_allclose(y[0, 0], vf[[0, 1, 5, 6, 7, 8]].mean(0), rtol=1e-12)
    np.testing.assert_allclose(y[0, 1:], np.broadcast_to(vf[2:5].mean(0), (3, d)), rtol=1e-12)


def test_rejects_sizes_that_do_not_sum():
    c = _case(M=6, N=6, MB=2, NB=2, Hq=1, Hkv=1, d=8)
    x = synth.make_varbsr_inputs(c)
    mm = np.ones((1, 2, 2), bool)
    with pytest.raises(oracle.OracleError):
        oracle.varbsr(x["q"], x["k"], x["v"], mm, np.array([[3, 2]], np.int32),
                      np.array([[3, 3]], np.int32), 0.5)
    with pytest.raises(oracle.OracleError):
        oracle.varbsr(x["q"], x["k"], x["v"], mm, np.array([[3, 3]], np.int32),
                      np.array([[7, -1]], np.int32), 0.5)


def test_rows_entry_equals_full_output():
    c = _case(causal=True, Hq=8, Hkv=2)
    x = synth.make_varbsr_inputs(c)
    args = (x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"], x["block_col_sz"],
            c.sm_scale)
    y, lse = oracle.varbsr(*args, causal=True)
    rows = np.array([0, 5, c.M - 1, c.M, 3 * c.M + 17, c.Hq * c.M - 1])
    yr, lr = oracle.varbsr_rows(*args, rows=rows, causal=True)
    np.testing.assert_array_equal(yr, y.reshape(-1, c.d)[rows])
    np.testing.assert_array_equal(lr, lse.reshape(-1)[rows])


def test_counts_match_dense_mask():
    for causal in (False, True):
        c = _case(causal=causal)
        x = synth.make_varbsr_inputs(c)
        allowed = _element_mask(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"])
        if causal:
            allowed &= np.arange(c.N)[None, None, :] <= np.arange(c.M)[None, :, None] + (c.N - c.M)
        n = synth.varbsr_counts(c, x["block_mask_map"], x["block_row_sz"], x["block_col_sz"])
        assert n["allowed"] == int(allowed.sum()) * (c.Hq // c.Hkv)
