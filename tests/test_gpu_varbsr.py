"""GPU parity of the variable block-sparse path (VariableBlockSparseAttentionWrapper)
against the CPU oracle, and the plan's key tile lists checked exactly."""
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


def run_varbsr(x, Hq, Hkv, d, scale, dtype, causal=False, plan=None):
    if plan is None:
        plan = sfa.varbsr_plan(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"], Hq, Hkv,
                               d, causal=causal, sm_scale=scale, dtype=dtype)
    q = x["q"].cuda()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    sfa.varbsr_run(plan, q, x["k"].cuda(), x["v"].cuda(), out, lse)
    torch.cuda.synchronize()
    assert sfa.sfa_get_last_error() == sfa.SFA_OK
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


def oracle_of(x, scale, causal=False):
    return oracle.varbsr(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                         x["block_col_sz"], scale, causal=causal)


def test_worked_example():
    ex = fixtures.varbsr_example()
    S, d = ex["seq_len"], ex["head_dim"]
    x = {"q": synth.normal(12, 0, (1, S, d), "f16"), "k": synth.normal(12, 1, (1, S, d), "f16"),
         "v": synth.normal(12, 2, (1, S, d), "f16"), "block_mask_map": ex["block_mask_map"],
         "block_row_sz": ex["block_row_sz"], "block_col_sz": ex["block_col_sz"]}
    scale = 1 / math.sqrt(d)
    out, lse = run_varbsr(x, 1, 1, d, scale, "f16")
    y, l = oracle_of(x, scale)
    compare(out, lse, y, l, "f16")


SHAPES = [
    # M, N, MB, NB, Hq, Hkv, d, dtype, p, causal
    (300, 500, 7, 9, 8, 2, 128, "f16", 0.4, False),      # G = 4
    (300, 500, 7, 9, 8, 2, 128, "bf16", 0.4, True),      # causal, qo_len < kv_len
    (256, 256, 64, 64, 4, 4, 64, "f16", 0.3, False),     # G = 1, many tiny and empty blocks
    (257, 257, 5, 3, 16, 2, 128, "bf16", 0.6, True),     # G = 8, causal, qo_len == kv_len
    (100, 700, 3, 20, 16, 1, 64, "f16", 0.5, False),     # G = 16
    (513, 130, 9, 4, 2, 1, 128, "f16", 0.7, True),       # causal, qo_len > kv_len: empty rows
]


@pytest.mark.parametrize("M,N,MB,NB,Hq,Hkv,d,dtype,p,causal", SHAPES)
def test_shapes(M, N, MB, NB, Hq, Hkv, d, dtype, p, causal):
    c = synth.VarBsrCase("t", M=M, N=N, MB=MB, NB=NB, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, p=p,
                         sm_scale=1 / math.sqrt(d), seed=91, causal=causal)
    x = synth.make_varbsr_inputs(c)
    out, lse = run_varbsr(x, Hq, Hkv, d, c.sm_scale, dtype, causal)
    y, l = oracle_of(x, c.sm_scale, causal)
    compare(out, lse, y, l, dtype)


def _plan_lists(plan, Hkv, MB):
    """(lists, windows (n, 6), items (m, 4)) read back from the plan's
    workspace (each part starts on a 16-byte boundary)."""
    ws = plan.int_ws.cpu().view(torch.int32).numpy()
    nl = Hkv * MB
    lists = ws[: nl + 1]
    off = (nl + 1 + 3) // 4 * 4
    nt = int(lists[-1])
    tiles = ws[off: off + 6 * nt].reshape(nt, 6)
    return lists, tiles, ws[off + (6 * nt + 3) // 4 * 4:]


@pytest.mark.parametrize("causal", [False, True])
def test_plan_tiles_cover_exactly_the_allowed_keys(causal):
    c = synth.VarBsrCase("p", M=700, N=900, MB=11, NB=13, Hq=8, Hkv=2, d=128, dtype="f16",
                         p=0.5, sm_scale=0.1, seed=93, causal=causal)
    x = synth.make_varbsr_inputs(c)
    plan = sfa.varbsr_plan(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"], c.Hq, c.Hkv,
                           c.d, causal=causal, sm_scale=c.sm_scale, dtype="f16")
    torch.cuda.synchronize()
    assert (plan.qo_len, plan.kv_len) == (c.M, c.N)
    lists, tiles, items = _plan_lists(plan, c.Hkv, c.MB)
    rows_covered = np.zeros((c.Hkv, c.M), np.int64)
    for g in range(c.Hkv):
        r0 = 0
        cstart = np.concatenate([[0], np.cumsum(x["block_col_sz"][g])])
        for rb in range(c.MB):
            s = int(x["block_row_sz"][g][rb])
            want = np.zeros(c.N, bool)
            for cb in np.nonzero(x["block_mask_map"][g][rb])[0]:
                want[cstart[cb]:cstart[cb + 1]] = True
            if causal:
                want[max(0, r0 + s - 1 + c.N - c.M + 1):] = False
            got = np.zeros(c.N, bool)
            lst = g * c.MB + rb
            prev_end = -1
            for t in tiles[lists[lst]:lists[lst + 1]]:
                # four 16-key quarters: starts t[0..3], mask t[5]:t[4] with
                # bits 16 q .. 16 q + 15 for quarter q; a last window is
                # completed with empty quarters at key N
                m64 = int(np.uint32(t[4])) | (int(np.uint32(t[5])) << 32)
                for q in range(4):
                    start, mask = int(t[q]), (m64 >> (16 * q)) & 0xFFFF
                    if mask == 0:
                        assert start == c.N                    # a padding quarter
                        continue
                    assert start >= prev_end and mask & 1      # disjoint, starts on an allowed key
                    for j in range(16):
                        if (mask >> j) & 1:
                            assert start + j < c.N
                            got[start + j] = True
                    prev_end = start + 16
            if s > 0:
                assert np.array_equal(got, want), (g, rb)
            else:
                assert lists[lst + 1] == lists[lst]
            r0 += s
    # work items: every row of every kv head exactly once
    assert len(items) % 4 == 0
    rows_per = 2 * (128 // (c.Hq // c.Hkv))
    for lst, row0, g, row_end in items.reshape(-1, 4):
        rows_covered[g, row0: min(row0 + rows_per, row_end)] += 1
    assert (rows_covered == 1).all()


def test_plan_reuse_and_empty_rows():
    c = synth.VarBsrCase("r", M=200, N=300, MB=4, NB=5, Hq=8, Hkv=2, d=64, dtype="bf16", p=0.5,
                         sm_scale=0.125, seed=94)
    x = synth.make_varbsr_inputs(c)
    mm = x["block_mask_map"].copy()
    mm[1, 2, :] = False                    # kv head 1, row block 2: no key
    x["block_mask_map"] = mm
    plan = sfa.varbsr_plan(mm, x["block_row_sz"], x["block_col_sz"], c.Hq, c.Hkv, c.d,
                           sm_scale=c.sm_scale, dtype="bf16")
    r0 = int(x["block_row_sz"][1][:2].sum())
    r1 = r0 + int(x["block_row_sz"][1][2])
    for seed in (1, 2):
        x["q"] = synth.normal(seed, 0, (c.Hq, c.M, c.d), "bf16")
        out, lse = run_varbsr(x, c.Hq, c.Hkv, c.d, c.sm_scale, "bf16", plan=plan)
        y, l = oracle_of(x, c.sm_scale)
        compare(out, lse, y, l, "bf16")
        assert torch.all(out[4:8, r0:r1] == 0) and torch.all(torch.isneginf(lse[4:8, r0:r1]))


def test_large_scores_rescale():
    """Scores spanning a wide range exercise the conditional O rescale."""
    c = synth.VarBsrCase("s", M=128, N=640, MB=2, NB=3, Hq=4, Hkv=1, d=128, dtype="f16", p=1.0,
                         sm_scale=0.0884, seed=95)
    x = synth.make_varbsr_inputs(c)
    x["q"] = (x["q"].float() * 3).half()
    x["k"] = (x["k"].float() * torch.linspace(0.2, 4.0, c.N).view(1, c.N, 1)).half()
    out, lse = run_varbsr(x, c.Hq, c.Hkv, c.d, c.sm_scale, "f16")
    y, l = oracle_of(x, c.sm_scale)
    compare(out, lse, y, l, "f16")


@pytest.mark.slow
def test_full_workload_sampled():
    c = synth.VARBSR
    x = synth.make_varbsr_inputs(c)
    out, lse = run_varbsr(x, c.Hq, c.Hkv, c.d, c.sm_scale, c.dtype, c.causal)
    rng = np.random.default_rng(3)
    # the edges of the work items: items take 2 * 128 / G rows of one
    # (kv head, row block) in two M-tiles; rows at offsets 0, 31, 32, 63, 64
    # and the last row of every row block of kv heads 0 and Hkv - 1, and the
    # first and last row of every row block of the others (one qo head each)
    G = c.Hq // c.Hkv
    tr = 128 // G
    edge = []
    for g in range(c.Hkv):
        starts = np.concatenate([[0], np.cumsum(x["block_row_sz"][g])[:-1]])
        for rb, (r0, sz) in enumerate(zip(starts, x["block_row_sz"][g])):
            if sz == 0:
                continue
            offs = ((0, tr - 1, tr, 2 * tr - 1, 2 * tr, sz - 1) if g in (0, c.Hkv - 1)
                    else (0, sz - 1))
            h = g * G + rb % G
            edge += [h * c.M + r0 + o for o in set(offs) if o < sz]
    rows = np.concatenate([rng.integers(0, c.Hq * c.M, 64), edge, [0, c.Hq * c.M - 1]])
    assert len(rows) > 2000
    y, l = oracle.varbsr_rows(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                              x["block_col_sz"], c.sm_scale, rows, causal=c.causal)
    got = out.reshape(-1, c.d)[rows]
    gl = lse.reshape(-1)[rows]
    compare(got, gl, y, l, c.dtype)
    assert torch.isfinite(out.float()).all()
