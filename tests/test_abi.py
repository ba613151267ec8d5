"""The C ABI without a GPU: the library builds, loads, exports every entry
point declared in include/*.h, and rejects bad arguments on the host before
any launch."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest
import torch

import sparse_attention_serving_sfa_gb300 as sfa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sfa.build()
    return sfa.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"sfa_run", "sfa_run_ex", "bsr_plan", "bsr_run", "bsr_plan_destroy"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(sfa.EXPORTS) <= names


def test_status_strings(lib):
    for st in range(7):
        assert sfa.status_string(st)


FAKE = 1 << 20     # aligned non-null address; never dereferenced by rejected calls


def call_run(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE + 4096, idx=FAKE, B=1, S1=4, S2=64, N1=4, N2=1, Dk=64, Dv=64,
             topK=16, scale=0.125, layout=0, causal=0, dtype=0, out=FAKE, lse=None)
    a.update(over)
    return sfa.sfa_run(a["q"], a["k"], a["v"], a["idx"], a["B"], a["S1"], a["S2"], a["N1"],
                       a["N2"], a["Dk"], a["Dv"], a["topK"], a["scale"], a["layout"], a["causal"],
                       a["dtype"], a["out"], a["lse"], None, check=False)


@pytest.mark.parametrize("over,status", [
    (dict(N1=6, N2=4), sfa.SFA_ERR_INVALID_ARG),            # N1 % N2 != 0
    (dict(Dv=128, Dk=64), sfa.SFA_ERR_INVALID_ARG),         # Dv > Dk
    (dict(Dk=96, Dv=64), sfa.SFA_ERR_INVALID_ARG),          # Dk not 64-aligned
    (dict(Dv=32), sfa.SFA_ERR_INVALID_ARG),                 # Dv not 64-aligned
    (dict(topK=65), sfa.SFA_ERR_INVALID_ARG),               # topK > S2
    (dict(topK=0), sfa.SFA_ERR_INVALID_ARG),
    (dict(causal=1, S1=65), sfa.SFA_ERR_INVALID_ARG),       # causal needs S1 <= S2
    (dict(layout=2), sfa.SFA_ERR_INVALID_ARG),
    (dict(dtype=7), sfa.SFA_ERR_INVALID_ARG),
    (dict(q=None), sfa.SFA_ERR_INVALID_ARG),
    (dict(idx=None), sfa.SFA_ERR_INVALID_ARG),
    (dict(out=None), sfa.SFA_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), sfa.SFA_ERR_INVALID_ARG),            # misaligned
    (dict(lse=FAKE + 1), sfa.SFA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), sfa.SFA_ERR_INVALID_ARG),
    (dict(B=0), sfa.SFA_ERR_INVALID_ARG),
    (dict(Dk=640, Dv=64), sfa.SFA_ERR_UNSUPPORTED),         # beyond this build's limits
    (dict(Dk=640, Dv=576), sfa.SFA_ERR_UNSUPPORTED),
])
def test_sfa_run_rejects(lib, over, status):
    assert call_run(**over) == status


def test_prefix_flag_requires_alias(lib):
    st = sfa.sfa_run_ex(FAKE, FAKE, FAKE + 4096, FAKE, 1, 4, 64, 4, 1, 128, 64, 16, 0.1, 0, 0, 0,
                        FAKE, None, None, value_is_key_prefix=True, check=False)
    assert st == sfa.SFA_ERR_INVALID_ARG


def test_workspace_size(lib):
    n = sfa.sfa_workspace_size(16, 1, 32, 8, 128, 128, 1024)
    assert n >= 16 * 32 * 2 * (128 + 2) * 4
    assert sfa.sfa_workspace_size(1, 1, 1, 1, 64, 64, 16, num_splits=1) == 0
    # fixed counter head (16384 ints) + split partials
    assert sfa.sfa_workspace_size(2, 3, 4, 2, 64, 64, 64, num_splits=4) == 65536 + 2 * 3 * 4 * 4 * 66 * 4
    with pytest.raises(sfa.SfaError):
        sfa.sfa_workspace_size(0, 1, 1, 1, 64, 64, 16)


def bsr_call(indptr, indices, M, N, R, C, Hq=4, Hkv=2, d=64, causal=0, ws_bytes=1 << 20):
    handle = ctypes.c_void_p(0)
    ip = torch.tensor(indptr, dtype=torch.int32)
    ix = torch.tensor(indices if indices else [0], dtype=torch.int32)
    st = sfa.load().bsr_plan(ip.data_ptr(), ix.data_ptr(), M, N, R, C, Hq, Hkv, d, causal, 0.0, 0,
                             FAKE, ws_bytes, None, 0, None, ctypes.byref(handle))
    assert not handle.value
    return st


@pytest.mark.parametrize("args,status", [
    (([0, 1, 2], [0, 1], 4, 5, 2, 2), sfa.SFA_ERR_INVALID_ARG),        # N % C != 0
    (([1, 1, 2], [0, 1], 4, 4, 2, 2), sfa.SFA_ERR_INVALID_ARG),        # indptr[0] != 0
    (([0, 2, 1], [0, 1], 4, 4, 2, 2), sfa.SFA_ERR_INVALID_ARG),        # decreasing indptr
    (([0, 1, 2], [0, 2], 4, 4, 2, 2), sfa.SFA_ERR_INVALID_ARG),        # block column >= NB
    (([0, 2, 2], [1, 1], 4, 4, 2, 2), sfa.SFA_ERR_INVALID_ARG),        # repeated block
    (([0, 1, 2], [0, 1], 4, 4, 2, 2, 3, 2), sfa.SFA_ERR_INVALID_ARG),  # Hq % Hkv != 0
    (([0, 1, 2], [0, 1], 4, 4, 2, 2, 4, 2, 96), sfa.SFA_ERR_INVALID_ARG),   # head_dim % 64
    (([0, 1, 2], [0, 1], 4, 4, 2, 2, 4, 2, 320), sfa.SFA_ERR_UNSUPPORTED),  # head_dim > 256
])
def test_bsr_plan_rejects(lib, args, status):
    assert bsr_call(*args) == status


def test_bsr_plan_workspace_too_small(lib):
    assert bsr_call([0, 1, 2], [0, 1], 4, 4, 2, 2, ws_bytes=8) == sfa.SFA_ERR_WORKSPACE


def test_bsr_int_workspace_size(lib):
    ip = torch.tensor([0, 1, 3, 5], dtype=torch.int32)
    n = sfa.bsr_plan_int_workspace_size(ip, 3, 3, 1, 1, 32, 8, 128)
    # indptr (4) + indices (5 -> 8) + 3 tiles x 4 ints
    assert n == 4 * (4 + 8 + 12)


def test_bsr_causal_plan_passes_validation(lib):
    # causal is supported: validation passes and only the workspace is checked
    assert bsr_call([0, 1, 2], [0, 1], 4, 4, 2, 2, causal=1, ws_bytes=8) == sfa.SFA_ERR_WORKSPACE


def test_bsr_masked_int_workspace_size(lib):
    ip = torch.tensor([0, 1, 3, 5], dtype=torch.int32)
    base = sfa.bsr_plan_int_workspace_size(ip, 48, 48, 16, 16, 32, 8, 128)
    assert sfa.bsr_plan_masked_int_workspace_size(ip, 48, 48, 16, 16, 32, 8, 128, False) == base
    # 5 blocks x 16 x 16 bits = 160 bytes (a multiple of 16)
    assert sfa.bsr_plan_masked_int_workspace_size(ip, 48, 48, 16, 16, 32, 8, 128, True) == base + 160
    ip1 = torch.tensor([0, 1], dtype=torch.int32)
    base1 = sfa.bsr_plan_int_workspace_size(ip1, 3, 3, 3, 3, 4, 2, 64)
    # 9 bits -> 2 bytes -> rounded up to 16
    assert sfa.bsr_plan_masked_int_workspace_size(ip1, 3, 3, 3, 3, 4, 2, 64, True) == base1 + 16


def test_bsr_masked_plan_needs_room_for_the_mask(lib):
    handle = ctypes.c_void_p(0)
    ip = torch.tensor([0, 1, 2], dtype=torch.int32)
    ix = torch.tensor([0, 1], dtype=torch.int32)
    mask = sfa.pack_block_mask(torch.ones(2, 2, 2, dtype=torch.bool))
    base = sfa.bsr_plan_int_workspace_size(ip, 4, 4, 2, 2, 4, 2, 64)
    st = sfa.load().bsr_plan_masked(ip.data_ptr(), ix.data_ptr(), mask.ctypes.data, 4, 4, 2, 2, 4,
                                    2, 64, 0, 0.0, 0, FAKE, base, None, 0, None,
                                    ctypes.byref(handle))
    assert st == sfa.SFA_ERR_WORKSPACE and not handle.value


def test_pack_block_mask_bit_order():
    m = torch.zeros(1, 2, 8, dtype=torch.bool)
    m[0, 0, 1] = True
    m[0, 1, 7] = True
    assert list(sfa.pack_block_mask(m)) == [0x40, 0x01]


# ---- variable block-sparse plan (host logic only) ----

def _varbsr_example():
    mm = np.array([[[0, 0, 1], [1, 0, 1], [0, 1, 1]]], dtype=np.uint8)
    rs = np.array([[1, 2, 3]], dtype=np.int32)
    cs = np.array([[3, 1, 2]], dtype=np.int32)
    return mm, rs, cs


def test_varbsr_int_workspace_size(lib):
    mm, rs, cs = _varbsr_example()
    # 3 lists (offsets: 4 ints) + 3 key windows x 6 ints (rounded up to 20)
    # + 3 items x 4 ints
    assert sfa.varbsr_plan_int_workspace_size(mm, rs, cs, 1, 1, 128) == 4 * (4 + 20 + 12)
    # causal (qo_len == kv_len == 6): row block 0 (row 0) sees no allowed key
    # (its set block holds keys 4, 5), so one window fewer
    assert sfa.varbsr_plan_int_workspace_size(mm, rs, cs, 1, 1, 128, causal=True) == 4 * (4 + 12 + 12)
    # four 16-key quarters per window: one set block of 130 keys needs 9
    # quarters, 3 windows (18 ints, rounded up to 20)
    n = sfa.varbsr_plan_int_workspace_size(np.ones((1, 1, 1), np.uint8), [[10]], [[130]], 4, 1, 64)
    assert n == 4 * (4 + 20 + 4)


@pytest.mark.parametrize("rs,cs,Hq,Hkv,d,status", [
    ([[1, 2, 3]], [[3, 1, 2]], 3, 2, 128, sfa.SFA_ERR_INVALID_ARG),     # Hq % Hkv != 0
    ([[1, 2, 3]], [[3, 1, 2]], 3, 1, 128, sfa.SFA_ERR_UNSUPPORTED),     # 128 % G != 0
    ([[1, 2, 3]], [[3, 1, 2]], 1, 1, 96, sfa.SFA_ERR_UNSUPPORTED),      # head_dim not 64 / 128
    ([[1, -2, 3]], [[3, 1, 2]], 1, 1, 128, sfa.SFA_ERR_INVALID_ARG),    # negative size
    ([[0, 0, 0]], [[3, 1, 2]], 1, 1, 128, sfa.SFA_ERR_INVALID_ARG),     # qo_len 0
])
def test_varbsr_plan_rejects(lib, rs, cs, Hq, Hkv, d, status):
    mm = np.ones((1, 3, 3), np.uint8)
    with pytest.raises(sfa.SfaError) as e:
        sfa.varbsr_plan_int_workspace_size(mm, rs, cs, Hq, Hkv, d)
    assert e.value.status == status


def test_varbsr_heads_must_agree_on_lengths(lib):
    mm = np.ones((2, 2, 2), np.uint8)
    with pytest.raises(sfa.SfaError) as e:
        sfa.varbsr_plan_int_workspace_size(mm, [[2, 2], [1, 2]], [[3, 3], [3, 3]], 2, 2, 64)
    assert e.value.status == sfa.SFA_ERR_INVALID_ARG


def test_varbsr_plan_workspace_too_small(lib):
    mm, rs, cs = _varbsr_example()
    handle = ctypes.c_void_p(0)
    st = sfa.load().varbsr_plan(mm.ctypes.data, rs.ctypes.data, cs.ctypes.data, 3, 3, 1, 1, 128, 0,
                                0.0, 0, FAKE, 8, None, ctypes.byref(handle))
    assert st == sfa.SFA_ERR_WORKSPACE and not handle.value


def test_soft_cap_setters_reject_bad_arguments(lib):
    assert lib.bsr_plan_set_logits_soft_cap(None, 1.0) == sfa.SFA_ERR_INVALID_ARG
    assert lib.varbsr_plan_set_logits_soft_cap(None, 1.0) == sfa.SFA_ERR_INVALID_ARG
    # (making a plan needs a device; the NaN / inf checks run in test_gpu_softcap.py)


def test_kv_layout_setter_rejects_bad_arguments(lib):
    assert lib.bsr_plan_set_kv_layout(None, 0) == sfa.SFA_ERR_INVALID_ARG
    assert lib.bsr_plan_set_kv_layout(None, 1) == sfa.SFA_ERR_INVALID_ARG
    # a plan with a layout value outside the enum: checked on the GPU machine
    # (making a plan uploads its work list)


def test_gather_probe_rejects_bad_arguments(lib):
    # host-side checks only (null pointers, sizes, alignment): no GPU needed
    assert lib.sfa_gather_probe(None, FAKE, FAKE, 1, 1, 8, 1, 64, 64, 4, 0, FAKE, 4096,
                                None) == sfa.SFA_ERR_INVALID_ARG
    assert lib.sfa_gather_probe(FAKE, FAKE, FAKE, 1, 1, 8, 1, 64, 64, 9, 0, FAKE, 4096,
                                None) == sfa.SFA_ERR_INVALID_ARG     # topK > S2
    assert lib.sfa_gather_probe(FAKE, FAKE, FAKE, 1, 1, 8, 1, 64, 128, 4, 0, FAKE, 4096,
                                None) == sfa.SFA_ERR_INVALID_ARG     # Dv > Dk
    assert lib.sfa_gather_probe(FAKE, FAKE, FAKE + 8, 1, 1, 8, 1, 64, 64, 4, 0, FAKE, 4096,
                                None) == sfa.SFA_ERR_INVALID_ARG     # unaligned indices


def test_tma_gather_probe_rejects_bad_arguments(lib):
    assert lib.sfa_gather_probe_tma(None, FAKE, FAKE, 1, 1, 8, 1, 64, 64, 4, 0,
                                    None) == sfa.SFA_ERR_INVALID_ARG
    assert lib.sfa_gather_probe_tma(FAKE, FAKE, FAKE, 1, 1, 8, 1, 64, 64, 9, 0,
                                    None) == sfa.SFA_ERR_INVALID_ARG     # topK > S2
    assert lib.sfa_gather_probe_tma(FAKE, FAKE, FAKE, 1, 1, 8, 1, 96, 64, 4, 0,
                                    None) == sfa.SFA_ERR_INVALID_ARG     # Dk % 64
    assert lib.sfa_gather_probe_tma(FAKE, FAKE, FAKE, 1, 1, 8, 1, 64, 64, 4, 2,
                                    None) == sfa.SFA_ERR_INVALID_ARG     # layout
    assert lib.sfa_gather_probe_tma(FAKE, FAKE, FAKE, 1 << 16, 1, 1 << 14, 8, 64, 64, 4, 0,
                                    None) == sfa.SFA_ERR_UNSUPPORTED     # 2^33 rows


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(sfa, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sfa, "_lib", None)
    with pytest.raises(RuntimeError):
        sfa.load()


def _varbsr_expected_bytes(mm, rs, cs, Hq, Hkv, causal):
    """Workspace bytes from an independent count: per (kv head, row block) the
    fewest 16-key quarters covering the allowed keys (greedy from the first
    uncovered key), four to a window of 6 ints (a last window padded), and
    ceil(rows / (2 * 128 / G)) work items per non-empty row block; each part
    starts on a 16-byte boundary."""
    Hkv_, MB, NB = mm.shape
    M, N = int(rs[0].sum()), int(cs[0].sum())
    rows_per = 2 * (128 // (Hq // Hkv))
    ntiles = nitems = 0
    for g in range(Hkv_):
        cstart = np.concatenate([[0], np.cumsum(cs[g])])
        r0 = 0
        for rb in range(MB):
            s = int(rs[g][rb])
            if s > 0:
                keys = np.zeros(N, bool)
                for cb in np.nonzero(mm[g][rb])[0]:
                    keys[cstart[cb]:cstart[cb + 1]] = True
                if causal:
                    keys[max(0, r0 + s - 1 + N - M + 1):] = False
                j = quarters = 0
                while j < N:
                    if keys[j]:
                        quarters += 1
                        j += 16
                    else:
                        j += 1
                ntiles += -(-quarters // 4)
                nitems += -(-s // rows_per)
            r0 += s
    nlists = Hkv_ * MB
    return 4 * (((nlists + 1 + 3) // 4) * 4 + (6 * ntiles + 3) // 4 * 4 + 4 * nitems)


@pytest.mark.parametrize("seed,causal,Hq,Hkv", [(1, False, 8, 2), (2, True, 8, 2),
                                               (3, False, 16, 1), (4, True, 4, 4)])
def test_varbsr_workspace_matches_independent_tiling(lib, seed, causal, Hq, Hkv):
    import synth
    c = synth.VarBsrCase("w", M=900, N=1300, MB=13, NB=17, Hq=Hq, Hkv=Hkv, d=128, dtype="f16",
                         p=0.4, sm_scale=0.1, seed=seed, causal=causal)
    rng = np.random.Generator(np.random.PCG64(seed))
    rs = synth.block_sizes(rng, Hkv, c.MB, c.M)
    cs = synth.block_sizes(rng, Hkv, c.NB, c.N)
    mm = rng.random((Hkv, c.MB, c.NB)) < c.p
    got = sfa.varbsr_plan_int_workspace_size(mm, rs, cs, Hq, Hkv, 128, causal=causal)
    assert got == _varbsr_expected_bytes(mm.astype(np.uint8), rs, cs, Hq, Hkv, causal)
