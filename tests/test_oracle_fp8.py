"""Pins of the oracle's FP8 path: the E4M3 / E5M2 decoders and run()'s
per-head dequantisation scales ("flashinfer.sparse",
BlockSparseAttentionWrapper plan() q_data_type / kv_data_type, run()
scale_q / scale_k / scale_v; the two formats are the ones the operator page's
precision table, §4 精度要求, names).  CPU only.

What pins what:
  - every one of the 256 codes of each format against torch's own float8
    types (an independent implementation of the formats), and closed forms
    (largest finite value, smallest subnormal, one, NaN / infinity codes);
    E5M2 also as the high byte of an IEEE binary16;
  - FP8 inputs with unit scales against the 16-bit oracle on the same values
    (every E4M3 / E5M2 value is exact in fp16);
  - each scale against the closed form it stands for: scale_v multiplies the
    output of its kv head's rows and leaves lse alone; scale_k of kv head g
    and scale_q of qo head h act as a factor on sm_scale for exactly the rows
    they reach;
  - a dense brute force in numpy (decoding through torch, masks expanded
    with np.kron) for mixed (fp16 q, FP8 k / v) and pure FP8 inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

F8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _torch_decode(codes, fmt):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(F8[fmt])
    return t.to(torch.float64).numpy()


def _same_with_nan(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)],
                                                                       b[~np.isnan(b)])


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode(codes, "e4m3")
    assert _same_with_nan(got, _torch_decode(codes, "e4m3"))
    # signs of zero
    assert not np.signbit(got[0]) and np.signbit(got[0x80])


def test_e5m2_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    assert _same_with_nan(oracle.decode(codes, "e5m2"), _torch_decode(codes, "e5m2"))


def test_e5m2_is_the_high_byte_of_f16():
    codes = np.arange(256, dtype=np.uint16)
    as_f16 = oracle.decode(codes << 8, "f16")
    assert _same_with_nan(oracle.decode(codes.astype(np.uint8), "e5m2"), as_f16)


def test_fp8_closed_forms():
    e4 = oracle.decode(np.array([0x7E, 0x01, 0x08, 0x38, 0x7F, 0xFF, 0xFE, 0x07], np.uint8), "e4m3")
    assert e4[0] == 448.0 and e4[1] == 2.0 ** -9 and e4[2] == 2.0 ** -6 and e4[3] == 1.0
    assert np.isnan(e4[4]) and np.isnan(e4[5]) and e4[6] == -448.0 and e4[7] == 7 * 2.0 ** -9
    e5 = oracle.decode(np.array([0x7B, 0x7C, 0x01, 0x3C, 0x7D, 0xFC, 0x04], np.uint8), "e5m2")
    assert e5[0] == 57344.0 and e5[1] == np.inf and e5[2] == 2.0 ** -16 and e5[3] == 1.0
    assert np.isnan(e5[4]) and e5[5] == -np.inf and e5[6] == 2.0 ** -14


# ---------------------------------------------------------------------------
# block-sparse attention with FP8 inputs and per-head scales

def _case(fmt_q, fmt_kv, M=48, N=64, R=16, C=16, Hq=4, Hkv=2, d=32, seed=5):
    """Inputs whose FP8 codes are N(0,1) samples converted by torch, one
    random scale per head, and a random block pattern."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(M, Hq, d, generator=g)
    k = torch.randn(N, Hkv, d, generator=g) * 3
    v = torch.randn(N, Hkv, d, generator=g)
    cast = {"f16": torch.float16, "bf16": torch.bfloat16, **F8}
    MB, NB = -(-M // R), N // C
    indptr, indices = synth.bsr_pattern(seed, MB, NB, 0.5)
    return {"q": q.to(cast[fmt_q]), "k": k.to(cast[fmt_kv]), "v": v.to(cast[fmt_kv]),
            "indptr": torch.from_numpy(indptr), "indices": torch.from_numpy(indices.copy()),
            "M": M, "N": N, "R": R, "C": C, "Hq": Hq, "Hkv": Hkv, "d": d,
            "scale_q": 0.5 + torch.rand(Hq, generator=g).numpy(),
            "scale_k": 0.5 + torch.rand(Hkv, generator=g).numpy(),
            "scale_v": 0.5 + torch.rand(Hkv, generator=g).numpy()}


def _run(x, scale, **kw):
    return oracle.bsr_scaled(x["q"], x["k"], x["v"], x["indptr"], x["indices"], x["M"], x["N"],
                             x["R"], x["C"], scale, **kw)


def test_fp8_equals_the_16bit_run_on_the_same_values():
    for fmt in ("e4m3", "e5m2"):
        x = _case(fmt, fmt)
        y8, l8 = _run(x, 0.2)
        x16 = dict(x, q=x["q"].to(torch.float16), k=x["k"].to(torch.float16),
                   v=x["v"].to(torch.float16))
        y16, l16 = oracle.bsr(x16["q"], x16["k"], x16["v"], x["indptr"], x["indices"], x["M"],
                              x["N"], x["R"], x["C"], 0.2)
        np.testing.assert_array_equal(y8, y16)
        np.testing.assert_array_equal(l8, l16)


def test_scale_v_scales_the_output_only():
    x = _case("e4m3", "e4m3")
    y0, l0 = _run(x, 0.2)
    sv = np.array([3.0, 0.25])
    y1, l1 = _run(x, 0.2, scale_v=sv)
    G = x["Hq"] // x["Hkv"]
    for h in range(x["Hq"]):
        np.testing.assert_allclose(y1[:, h], y0[:, h] * sv[h // G], rtol=1e-12, atol=0)
    np.testing.assert_array_equal(l1, l0)


def test_scale_k_is_a_per_group_sm_scale():
    x = _case("e4m3", "e4m3")
    sk = np.array([1.7, 1.0])
    y1, l1 = _run(x, 0.2, scale_k=sk)
    y_s, l_s = _run(x, 0.2 * 1.7)
    y_1, l_1 = _run(x, 0.2)
    G = x["Hq"] // x["Hkv"]
    np.testing.assert_allclose(y1[:, :G], y_s[:, :G], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(l1[:, :G], l_s[:, :G], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(y1[:, G:], y_1[:, G:], rtol=1e-12, atol=0)


def test_scale_q_is_a_per_head_sm_scale():
    x = _case("e5m2", "e5m2")
    sq = np.ones(x["Hq"])
    sq[1] = 0.3
    y1, l1 = _run(x, 0.2, scale_q=sq)
    y_s, l_s = _run(x, 0.2 * 0.3)
    y_1, _ = _run(x, 0.2)
    np.testing.assert_allclose(y1[:, 1], y_s[:, 1], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(l1[:, 1], l_s[:, 1], rtol=1e-10, atol=1e-13)
    others = [h for h in range(x["Hq"]) if h != 1]
    np.testing.assert_allclose(y1[:, others], y_1[:, others], rtol=1e-12, atol=0)


@pytest.mark.parametrize("fmt_kv", ["e4m3", "e5m2"])
@pytest.mark.parametrize("fmt_q", ["f16", "same"])
def test_matches_dense_brute_force(fmt_kv, fmt_q):
    fq = fmt_kv if fmt_q == "same" else fmt_q
    x = _case(fq, fmt_kv)
    M, N, R, C, Hq, Hkv, d = (x[k] for k in ("M", "N", "R", "C", "Hq", "Hkv", "d"))
    scale = 1.0 / math.sqrt(d)
    y, lse = _run(x, scale, scale_q=x["scale_q"], scale_k=x["scale_k"], scale_v=x["scale_v"])
    # brute force: torch decodes, per-head scales multiply, dense masked softmax
    q = x["q"].to(torch.float64).numpy() * x["scale_q"][None, :, None]
    k = x["k"].to(torch.float64).numpy() * x["scale_k"][None, :, None]
    v = x["v"].to(torch.float64).numpy() * x["scale_v"][None, :, None]
    blocks = np.zeros((-(-M // R), N // C), bool)
    ip, ix = x["indptr"].numpy(), x["indices"].numpy()
    for br in range(blocks.shape[0]):
        blocks[br, ix[ip[br]:ip[br + 1]]] = True
    allowed = np.kron(blocks, np.ones((R, C), bool))[:M]
    G = Hq // Hkv
    for h in range(Hq):
        s = q[:, h] @ k[:, h // G].T * scale
        s = np.where(allowed, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        finite = np.isfinite(mx[:, 0])
        p = np.where(allowed, np.exp(s - np.where(np.isfinite(mx), mx, 0)), 0.0)
        l = p.sum(axis=1)
        want = np.where(finite[:, None], p @ v[:, h // G] / np.where(l > 0, l, 1)[:, None], 0.0)
        np.testing.assert_allclose(y[:, h], want, rtol=1e-9, atol=1e-12)
        wl = np.where(finite, mx[:, 0] + np.log(np.where(l > 0, l, 1)), -np.inf)
        np.testing.assert_allclose(lse[:, h], wl, rtol=1e-9, atol=1e-12)


def test_rows_entry_equals_the_whole_output():
    x = _case("e4m3", "e4m3")
    y, lse = _run(x, 0.3, scale_q=x["scale_q"], scale_k=x["scale_k"], scale_v=x["scale_v"])
    rows = np.array([[0, 0], [5, 3], [x["M"] - 1, 2], [17, 1]])
    yr, lr = _run(x, 0.3, scale_q=x["scale_q"], scale_k=x["scale_k"], scale_v=x["scale_v"],
                  rows=rows)
    np.testing.assert_array_equal(yr, y[rows[:, 0], rows[:, 1]])
    np.testing.assert_array_equal(lr, lse[rows[:, 0], rows[:, 1]])
