"""Pins for the CPU oracle: each test checks it against something other than
itself -- the pages' worked examples, closed forms, a library routine on a
special case, or brute force with a different formulation."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests.golden import fixtures


# --------------------------------------------------------------------------
# helpers (independent of the oracle's code)

def small_case(**kw):
    base = dict(name="t", B=2, S1=3, S2=7, N1=4, N2=2, Dk=8, Dv=6, topK=5, dtype="f16",
                layout="BSND", causal=False, scale=0.3, seed=77)
    base.update(kw)
    return synth.SfaCase(**base)


def canon(t, layout):
    """Tensor in `layout` -> canonical [B, S, N, D] view."""
    return t if layout == "BSND" else t.permute(0, 2, 1, 3)


def with_replacement_indices(case, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, case.S2, (case.B, case.S1, case.N2, case.topK), generator=g,
                        dtype=torch.int32)
    return idx if case.layout == "BSND" else idx.permute(0, 2, 1, 3).contiguous()


def brute_force_multiset(q, k, v, idx, case):
    """Dense formulation over all S2 positions with multiplicities:
    y = sum_j c_j e^{l_j} v_j / sum_j c_j e^{l_j}, c_j = number of unmasked
    slots of the row holding position j.  Pure-Python loops, tiny shapes only."""
    Q = canon(q, case.layout).double()
    K = canon(k, case.layout).double()
    V = canon(v, case.layout).double()
    I = canon(idx, case.layout)
    G = case.N1 // case.N2
    y = np.zeros((case.B, case.S1, case.N1, case.Dv))
    lse = np.zeros((case.B, case.S1, case.N1))
    for b in range(case.B):
        for s1 in range(case.S1):
            for n1 in range(case.N1):
                n2 = n1 // G
                counts = [0] * case.S2
                for i in range(case.topK):
                    j = int(I[b, s1, n2, i])
                    if case.causal and j > s1 + case.S2 - case.S1:
                        continue
                    counts[j] += 1
                if sum(counts) == 0:
                    lse[b, s1, n1] = -math.inf
                    continue
                logits = [case.scale * sum(float(Q[b, s1, n1, d]) * float(K[b, j, n2, d])
                                           for d in range(case.Dk)) for j in range(case.S2)]
                mx = max(logits[j] for j in range(case.S2) if counts[j])
                w = [counts[j] * math.exp(logits[j] - mx) for j in range(case.S2)]
                z = sum(w)
                for e in range(case.Dv):
                    y[b, s1, n1, e] = sum(w[j] * float(V[b, j, n2, e]) for j in range(case.S2)) / z
                lse[b, s1, n1] = mx + math.log(z)
    if case.layout == "BNSD":
        return y.transpose(0, 2, 1, 3), lse.transpose(0, 2, 1)
    return y, lse


def run_oracle(d, case):
    return oracle.sfa(d["q"], d["k"], d["v"], d["idx"], case.scale, case.layout, case.causal)


def sdpa_dense(qc, kc, vc, scale, mask=None):
    """torch SDPA in float64 on canonical [B, S, N, D] tensors, GQA by
    repeating KV heads; returns [B, S1, N1, Dv]."""
    G = qc.shape[2] // kc.shape[2]
    qh = qc.double().permute(0, 2, 1, 3)
    kh = kc.double().permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = vc.double().permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    m = None if mask is None else torch.as_tensor(mask, dtype=torch.bool)
    o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=m, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


# --------------------------------------------------------------------------
# top-K form

@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_brute_force_multiset(layout, causal, dtype):
    case = small_case(layout=layout, causal=causal, dtype=dtype)
    d = synth.make_sfa_inputs(case)
    d["idx"] = with_replacement_indices(case, 5)      # duplicates included
    y, lse = run_oracle(d, case)
    yb, lb = brute_force_multiset(d["q"], d["k"], d["v"], d["idx"], case)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
@pytest.mark.parametrize("causal", [False, True])
def test_identity_indices_equal_dense_sdpa(layout, causal):
    """topK = S2 with slot i -> position i is dense attention (torch SDPA);
    with causal, dense attention under tril(diagonal = S2 - S1)."""
    case = small_case(B=2, S1=5, S2=9, N1=6, N2=2, Dk=16, Dv=8, topK=9, layout=layout,
                      causal=causal, scale=0.25)
    d = synth.make_sfa_inputs(case)
    ident = torch.arange(case.S2, dtype=torch.int32).expand(case.B, case.S1, case.N2, case.S2)
    d["idx"] = ident.contiguous() if layout == "BSND" else ident.permute(0, 2, 1, 3).contiguous()
    y, lse = run_oracle(d, case)
    mask = None
    if causal:
        mask = torch.tril(torch.ones(case.S1, case.S2, dtype=torch.bool), diagonal=case.S2 - case.S1)
    ref = sdpa_dense(canon(d["q"], layout), canon(d["k"], layout), canon(d["v"], layout),
                     case.scale, mask)
    np.testing.assert_allclose(canon(torch.from_numpy(y), layout).numpy(), ref, rtol=1e-10,
                               atol=1e-12)
    # lse against torch.logsumexp of the (masked) scaled logits
    qh = canon(d["q"], layout).double().permute(0, 2, 1, 3)
    kh = canon(d["k"], layout).double().permute(0, 2, 1, 3).repeat_interleave(case.G, dim=1)
    logits = torch.einsum("bhsd,bhtd->bhst", qh, kh) * case.scale
    if causal:
        logits = logits.masked_fill(~mask, -math.inf)
    ref_lse = torch.logsumexp(logits, dim=-1).permute(0, 2, 1).numpy()   # [B,S1,N1]
    got_lse = lse if layout == "BSND" else lse.transpose(0, 2, 1)
    np.testing.assert_allclose(got_lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_causal_mask_matches_printed_rule():
    """With q = 0 every visible slot has the same weight, and v = one-hot of
    the key position makes y the visibility indicator / count."""
    fx = fixtures.causal_bottom_right()
    S1, S2 = fx["qo_len"], fx["kv_len"]
    case = small_case(B=1, S1=S1, S2=S2, N1=1, N2=1, Dk=8, Dv=S2, topK=S2, causal=True)
    q = torch.zeros(1, S1, 1, 8, dtype=torch.float16)
    k = synth.normal(3, 1, (1, S2, 1, 8), "f16")
    v = torch.eye(S2, dtype=torch.float16).reshape(1, S2, 1, S2)
    idx = torch.arange(S2, dtype=torch.int32).expand(1, S1, 1, S2).contiguous()
    y, lse = oracle.sfa(q, k, v, idx, case.scale, "BSND", True)
    mask = fx["mask"]
    for s1 in range(S1):
        n = mask[s1].sum()
        np.testing.assert_array_equal(y[0, s1, 0], mask[s1] / n)
        assert lse[0, s1, 0] == pytest.approx(math.log(n), abs=1e-15)


def test_fully_masked_rows_are_zero():
    case = small_case(B=1, S1=3, S2=8, N1=2, N2=1, Dk=8, Dv=8, topK=4, causal=True)
    d = synth.make_sfa_inputs(case)
    # row s1 = 0 sees positions <= 5: choose only 6 and 7 -> fully masked.
    idx = d["idx"].clone()
    idx[0, 0, 0] = torch.tensor([6, 7, 7, 6], dtype=torch.int32)
    d["idx"] = idx
    y, lse = run_oracle(d, case)
    assert np.all(y[0, 0] == 0.0) and not np.signbit(y[0, 0]).any()
    assert np.all(np.isneginf(lse[0, 0]))
    assert np.all(np.isfinite(lse[0, 1:]))


def test_single_slot_closed_form():
    """topK = 1: the softmax weight is 1, so y = v[idx] and lse = scale * q.k[idx]."""
    case = small_case(topK=1, Dk=16, Dv=16)
    d = synth.make_sfa_inputs(case)
    y, lse = run_oracle(d, case)
    Q, K, V, I = (canon(d[n], "BSND") for n in ("q", "k", "v", "idx"))
    for b in range(case.B):
        for s1 in range(case.S1):
            for n1 in range(case.N1):
                n2 = n1 // case.G
                j = int(I[b, s1, n2, 0])
                np.testing.assert_array_equal(y[b, s1, n1], V[b, j, n2].double().numpy())
                dot = float(np.dot(Q[b, s1, n1].double().numpy(), K[b, j, n2].double().numpy()))
                assert lse[b, s1, n1] == pytest.approx(case.scale * dot, rel=1e-14, abs=1e-14)


def test_uniform_scores_give_mean():
    """q = 0: every slot scores 0, so y is the mean of the gathered value rows
    and lse = ln(topK)."""
    case = small_case(topK=5)
    d = synth.make_sfa_inputs(case)
    d["q"] = torch.zeros_like(d["q"])
    y, lse = run_oracle(d, case)
    V, I = canon(d["v"], "BSND").double(), canon(d["idx"], "BSND").long()
    for b in range(case.B):
        for s1 in range(case.S1):
            for n1 in range(case.N1):
                n2 = n1 // case.G
                ref = V[b, I[b, s1, n2], n2].mean(dim=0).numpy()
                np.testing.assert_allclose(y[b, s1, n1], ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(case.topK), rtol=1e-14)


def test_gqa_equals_repeated_kv_heads():
    case = small_case(N1=6, N2=2, S2=11, topK=6, causal=True, S1=4)
    d = synth.make_sfa_inputs(case)
    y, lse = run_oracle(d, case)
    G = case.G
    rep = case.replace(N2=case.N1)
    d2 = {"q": d["q"], "k": d["k"].repeat_interleave(G, dim=2).contiguous(),
          "v": d["v"].repeat_interleave(G, dim=2).contiguous(),
          "idx": d["idx"].repeat_interleave(G, dim=2).contiguous()}
    y2, lse2 = run_oracle(d2, rep)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(lse, lse2)


def test_bsnd_equals_bnsd_after_permute():
    a = small_case(layout="BSND", causal=True, S1=4, S2=9)
    b = a.replace(layout="BNSD")
    da, db = synth.make_sfa_inputs(a), synth.make_sfa_inputs(b)
    for n in ("q", "k", "v", "idx"):
        assert torch.equal(da[n].permute(0, 2, 1, 3), db[n])
    ya, la = run_oracle(da, a)
    yb, lb = run_oracle(db, b)
    np.testing.assert_array_equal(ya.transpose(0, 2, 1, 3), yb)
    np.testing.assert_array_equal(la.transpose(0, 2, 1), lb)


def test_slot_order_invariance():
    case = small_case(topK=7, S2=12, causal=True, S1=5)
    d = synth.make_sfa_inputs(case)
    y, lse = run_oracle(d, case)
    perm = torch.from_numpy(np.random.default_rng(0).permutation(case.topK))
    d2 = dict(d, idx=d["idx"][..., perm].contiguous())
    y2, lse2 = run_oracle(d2, case)
    np.testing.assert_allclose(y, y2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13)


def test_duplicate_slot_counts_twice():
    """Two slots holding the same position: same y as one slot, lse + ln 2."""
    case = small_case(topK=1)
    d = synth.make_sfa_inputs(case)
    y1, l1 = run_oracle(d, case)
    d2 = dict(d, idx=d["idx"].repeat(1, 1, 1, 2).contiguous())
    y2, l2 = run_oracle(d2, case.replace(topK=2))
    np.testing.assert_allclose(y1, y2, rtol=1e-15, atol=0)
    np.testing.assert_allclose(l2, l1 + math.log(2.0), rtol=1e-14)


@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
def test_value_prefix_view_equals_copy(layout):
    case = small_case(Dk=16, Dv=8, layout=layout, value_is_key_prefix=True)
    d = synth.make_sfa_inputs(case)
    assert d["v"].data_ptr() == d["k"].data_ptr() and not d["v"].is_contiguous()
    y, lse = run_oracle(d, case)
    y2, lse2 = run_oracle(dict(d, v=d["v"].contiguous()), case)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(lse, lse2)


def test_rows_entry_matches_full():
    case = small_case(causal=True, S1=4, S2=9, layout="BNSD")
    d = synth.make_sfa_inputs(case)
    y, lse = run_oracle(d, case)
    rows = np.array([[b, n1, s1] for b in range(case.B) for n1 in range(case.N1)
                     for s1 in range(case.S1)])
    yr, lr = oracle.sfa_rows(d["q"], d["k"], d["v"], d["idx"], case.scale, rows, case.layout, True)
    for r, (b, n1, s1) in enumerate(rows):
        np.testing.assert_array_equal(yr[r], y[b, n1, s1])
        assert lr[r] == lse[b, n1, s1]


def test_out_of_range_index_is_an_error():
    case = small_case()
    d = synth.make_sfa_inputs(case)
    d["idx"] = d["idx"].clone()
    d["idx"][0, 0, 0, 0] = case.S2
    with pytest.raises(oracle.OracleError):
        run_oracle(d, case)


# --------------------------------------------------------------------------
# block-sparse form

def bsr_sdpa(q, k, v, mask, scale):
    """Dense masked attention via torch SDPA (float64) on NHD tensors."""
    G = q.shape[1] // k.shape[1]
    qh = q.double().permute(1, 0, 2)
    kh = k.double().permute(1, 0, 2).repeat_interleave(G, dim=0)
    vh = v.double().permute(1, 0, 2).repeat_interleave(G, dim=0)
    o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=torch.as_tensor(mask), scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_bsr_worked_example():
    fx = fixtures.bsr_3x3_example()
    M, N, Hq, Hkv, d = fx["M"], fx["N"], fx["num_qo_heads"], fx["num_kv_heads"], fx["head_dim"]
    q = synth.normal(11, 0, (M, Hq, d), "f16")
    k = synth.normal(11, 1, (N, Hkv, d), "f16")
    v = synth.normal(11, 2, (N, Hkv, d), "f16")
    indptr = torch.tensor(fx["indptr"], dtype=torch.int32)
    indices = torch.tensor(fx["indices"], dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    y, lse = oracle.bsr(q, k, v, indptr, indices, M, N, fx["R"], fx["C"], scale)
    ref = bsr_sdpa(q, k, v, fx["mask"], scale)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("R,C,M,N", [(3, 2, 10, 8), (4, 4, 12, 16), (1, 3, 5, 9)])
def test_bsr_equals_block_expanded_mask(R, C, M, N):
    MB, NB = -(-M // R), N // C
    indptr, indices = synth.bsr_pattern(99 + R, MB, NB, 0.4)
    dense_blocks = np.zeros((MB, NB), dtype=np.int64)
    for i in range(MB):
        dense_blocks[i, indices[indptr[i]:indptr[i + 1]]] = 1
    mask = np.kron(dense_blocks, np.ones((R, C), dtype=np.int64))[:M].astype(bool)
    live = mask.any(axis=1)                # rows with at least one stored block
    mask_sdpa = mask.copy()
    mask_sdpa[~live] = True                # keep SDPA finite on rows checked separately
    Hq, Hkv, d = 4, 2, 8
    q = synth.normal(5, 0, (M, Hq, d), "bf16")
    k = synth.normal(5, 1, (N, Hkv, d), "bf16")
    v = synth.normal(5, 2, (N, Hkv, d), "bf16")
    y, lse = oracle.bsr(q, k, v, torch.from_numpy(indptr), torch.from_numpy(indices), M, N, R,
                        C, 0.4)
    ref = bsr_sdpa(q, k, v, mask_sdpa, 0.4)
    np.testing.assert_allclose(y[live], ref[live], rtol=1e-10, atol=1e-12)
    assert np.all(y[~live] == 0.0) and np.all(np.isneginf(lse[~live]))
    G = Hq // Hkv
    kh = k.double().repeat_interleave(G, dim=1)
    logits = torch.einsum("mhd,nhd->hmn", q.double(), kh) * 0.4
    logits = logits.masked_fill(~torch.from_numpy(mask), -math.inf)
    np.testing.assert_allclose(lse[live], torch.logsumexp(logits, -1).T.numpy()[live], rtol=1e-12)


def test_bsr_empty_block_row_is_zero():
    M, N, R, C = 6, 6, 2, 3
    indptr = torch.tensor([0, 1, 1, 2], dtype=torch.int32)    # block row 1 empty
    indices = torch.tensor([0, 1], dtype=torch.int32)
    q = synth.normal(1, 0, (M, 2, 8), "f16")
    k = synth.normal(1, 1, (N, 1, 8), "f16")
    v = synth.normal(1, 2, (N, 1, 8), "f16")
    y, lse = oracle.bsr(q, k, v, indptr, indices, M, N, R, C, 0.5)
    assert np.all(y[2:4] == 0.0) and np.all(np.isneginf(lse[2:4]))
    assert np.all(np.isfinite(lse[:2])) and np.all(np.isfinite(lse[4:]))


def test_bsr_rows_entry_matches_full():
    M, N, R, C = 10, 8, 3, 2
    indptr, indices = synth.bsr_pattern(3, 4, 4, 0.5)
    q = synth.normal(2, 0, (M, 4, 8), "f16")
    k = synth.normal(2, 1, (N, 2, 8), "f16")
    v = synth.normal(2, 2, (N, 2, 8), "f16")
    ip, ix = torch.from_numpy(indptr), torch.from_numpy(indices)
    y, lse = oracle.bsr(q, k, v, ip, ix, M, N, R, C, 0.3)
    rows = np.array([[i, h] for i in range(M) for h in range(4)])
    yr, lr = oracle.bsr_rows(q, k, v, ip, ix, M, N, R, C, 0.3, rows)
    np.testing.assert_array_equal(yr, y.reshape(-1, 8))
    np.testing.assert_array_equal(lr, lse.reshape(-1))


def test_bsr_bad_block_column_is_an_error():
    q = synth.normal(1, 0, (4, 1, 8), "f16")
    k = synth.normal(1, 1, (4, 1, 8), "f16")
    with pytest.raises(oracle.OracleError):
        oracle.bsr(q, k, k, torch.tensor([0, 1, 2], dtype=torch.int32),
                   torch.tensor([0, 2], dtype=torch.int32), 4, 4, 2, 2, 1.0)


# --------------------------------------------------------------------------
# precision standard

def test_precision_report_closed_forms():
    g = np.linspace(0.5, 2.0, 101)
    rep = oracle.precision_report(g * (1 + 2.0 ** -12), g, "f16", round_golden=False)
    assert rep["mere"] == pytest.approx(2.0 ** -12, rel=1e-6)
    assert rep["passed"]
    rep = oracle.precision_report(g * (1 + 2.0 ** -9), g, "f16", round_golden=False)
    assert rep["mere"] == pytest.approx(2.0 ** -9, rel=1e-6) and not rep["passed"]
    # near-zero golden: a small absolute error is tolerated by the cap only
    g2 = np.array([1e-6, 1.0])
    a2 = np.array([5e-3, 1.0])
    rep = oracle.precision_report(a2, g2, "f16", round_golden=False)
    assert rep["mare"] > 10 * 2.0 ** -10 and rep["mare_capped"] == 0.0
    assert not oracle.precision_report(np.array([np.nan]), np.array([1.0]), "bf16")["passed"]
