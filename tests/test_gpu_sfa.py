"""GPU parity of the top-K path: the CUDA library (through the C ABI) against
the CPU oracle on the same seeded inputs, element by element at small sizes
and on sampled rows at the full workload sizes."""
import math

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


def small(**kw):
    base = dict(name="s", B=2, S1=3, S2=300, N1=8, N2=2, Dk=128, Dv=128, topK=100, dtype="bf16",
                layout="BSND", causal=False, scale=0.09, seed=4321)
    base.update(kw)
    return synth.SfaCase(**base)


def run_and_check(case, **opts):
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out, lse = T.run_gpu(case, dev, **opts)
    return T.check_full(case, d, out, lse)


def test_tiny_workload():
    run_and_check(synth.TINY)


@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_layouts_dtypes_causal(layout, dtype, causal):
    run_and_check(small(layout=layout, dtype=dtype, causal=causal, S2=120 if causal else 300))


@pytest.mark.parametrize("G,N2", [(1, 3), (4, 2), (8, 1), (16, 1), (128, 1)])
def test_gqa_groups(G, N2):
    run_and_check(small(N1=G * N2, N2=N2, S1=2, topK=70))


@pytest.mark.parametrize("Dk,Dv,prefix", [(64, 64, False), (192, 128, True), (256, 64, False),
                                          (576, 512, True), (512, 512, False)])
def test_head_dims(Dk, Dv, prefix):
    run_and_check(small(Dk=Dk, Dv=Dv, value_is_key_prefix=prefix, N1=4, N2=1, topK=77, S1=2))


@pytest.mark.parametrize("topK", [1, 2, 31, 32, 33, 64, 65, 257])
def test_ragged_topk(topK):
    run_and_check(small(topK=topK, S2=max(topK, 300)))


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_splits_agree(splits):
    case = small(topK=224, causal=True, S2=240)
    run_and_check(case, num_splits=splits)


def test_fully_masked_rows_exact_zero():
    """causal, indices of some rows entirely above the diagonal; those rows
    must be exactly +0 with lse = -inf, also when the row is split."""
    case = small(causal=True, S1=16, S2=64, topK=20, index_kind="causal_mix", masked_frac=0.1,
                 full_masked_rows=5)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for splits in (1, 3):
        out, lse = T.run_gpu(case, dev, num_splits=splits)
        T.check_full(case, d, out, lse)
        assert torch.all(out[0, :5] == 0) and torch.all(torch.isneginf(lse[0, :5]))


def test_identity_indices_equal_dense_attention():
    """topK = S2 with identity indices is dense attention (also checked by the
    oracle pins); here against the oracle on the GPU path."""
    case = small(S1=5, S2=96, topK=96, causal=True)
    d = synth.make_sfa_inputs(case)
    ident = torch.arange(case.S2, dtype=torch.int32).expand(case.B, case.S1, case.N2, case.S2)
    d["idx"] = ident.contiguous()
    out, lse = T.run_gpu(case, T.to_dev(d))
    T.check_full(case, d, out, lse)


def test_duplicate_indices_count_per_slot():
    case = small(topK=40, S2=50)
    d = synth.make_sfa_inputs(case)
    g = torch.Generator().manual_seed(3)
    d["idx"] = torch.randint(0, 10, d["idx"].shape, generator=g, dtype=torch.int32)
    out, lse = T.run_gpu(case, T.to_dev(d))
    T.check_full(case, d, out, lse)


def test_prefix_view_equals_separate_value():
    case = small(Dk=192, Dv=128, value_is_key_prefix=True)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out1, lse1 = T.run_gpu(case, dev)
    dev2 = dict(dev, v=dev["v"].contiguous())
    out2, lse2 = T.run_gpu(case.replace(value_is_key_prefix=False), dev2)
    T.check_full(case, d, out1, lse1)
    assert torch.allclose(out1.float(), out2.float(), atol=1e-2, rtol=0)


def test_caller_workspace_and_too_small():
    case = small(topK=256, S2=300)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    need = sfa.sfa_workspace_size(case.B, case.S1, case.N1, case.N2, case.Dk, case.Dv, case.topK,
                                  num_splits=4)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out, lse = T.run_gpu(case, dev, workspace=ws, num_splits=4)
    T.check_full(case, d, out, lse)
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(sfa.SfaError) as e:
        T.run_gpu(case, dev, workspace=small_ws, num_splits=4)
    assert e.value.status == sfa.SFA_ERR_WORKSPACE


def test_out_of_range_indices_masked_and_reported():
    case = small(topK=16, S2=64)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    assert sfa.sfa_get_last_error() == sfa.SFA_OK
    bad = dev["idx"].clone()
    bad[0, 0, 0, :4] = torch.tensor([-1, 64, 1 << 30, -(1 << 30)], dtype=torch.int32)
    out, lse = T.run_gpu(case, dict(dev, idx=bad), validate_indices=True)
    assert sfa.sfa_get_last_error() == sfa.SFA_ERR_INDEX_RANGE
    assert sfa.sfa_get_last_error() == sfa.SFA_OK        # cleared by the read
    # the bad slots behave as masked: equal to the oracle with those slots dropped
    keep = d["idx"][0, 0, 0, 4:].clone()
    G = case.G
    ds = {"q": d["q"][:1, :1, :G].contiguous(), "k": d["k"][:1, :, :1].contiguous(),
          "v": d["v"][:1, :, :1].contiguous(), "idx": keep.reshape(1, 1, 1, 12).contiguous()}
    y, l = oracle.sfa(ds["q"], ds["k"], ds["v"], ds["idx"], case.scale, "BSND", False)
    got = out[0, 0, :case.G].float().cpu().numpy()
    assert oracle.precision_report(got, y[0, 0, :case.G], case.dtype)["passed"]


def test_guard_bytes_untouched():
    """Writes stay inside out / lse: canaries around both survive."""
    case = small(topK=64, S2=100)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    n_out = case.B * case.S1 * case.N1 * case.Dv
    n_lse = case.B * case.S1 * case.N1
    big = torch.full((n_out + 2048,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbig = torch.full((n_lse + 256,), 7.0, dtype=torch.float32, device="cuda")
    out = big[1024:1024 + n_out]
    lse = lbig[128:128 + n_lse]
    sfa.sfa_run(dev["q"], dev["k"], dev["v"], dev["idx"], case.B, case.S1, case.S2, case.N1,
                case.N2, case.Dk, case.Dv, case.topK, case.scale, case.layout, case.causal,
                case.dtype, out, lse)
    torch.cuda.synchronize()
    assert torch.all(big[:1024] == 7.0) and torch.all(big[1024 + n_out:] == 7.0)
    assert torch.all(lbig[:128] == 7.0) and torch.all(lbig[128 + n_lse:] == 7.0)


def test_stream_argument():
    case = small()
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = sfa.sparse_flash_attention(dev["q"], dev["k"], dev["v"], dev["idx"], case.scale,
                                              case.layout, case.causal, return_lse=True, stream=s)
    s.synchronize()
    T.check_full(case, d, out, lse)


# ---------------------------------------------------------------------------
# full-size workloads, sampled rows

@pytest.mark.parametrize("name", ["gqa_decode", "mla_decode", "mla_mtp", "call_example"])
def test_full_workload_every_row(name):
    """The full-size workloads whose oracle finishes in seconds: every output
    row compared element by element (so every stream-K range boundary, split
    index list and cluster of the launch bench.py times is covered)."""
    case = synth.SFA_WORKLOADS[name]
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out, lse = T.run_gpu(case, dev)
    T.check_full(case, d, out, lse)
    assert torch.isfinite(out.float()).all()


def aligned_range_boundary_rows(case, ctas_options):
    """(b, n1, s1) rows of the first and last index list of every CTA's range
    when whole index lists are dealt out in equal contiguous ranges to `ctas`
    CTAs (list u = (b * N2 + n2) * S1 + s1), for each grid size given; the
    first and last query head of each such list."""
    units = case.B * case.N2 * case.S1
    lists = set()
    for ctas in ctas_options:
        for c in range(ctas):
            lo, hi = c * units // ctas, (c + 1) * units // ctas - 1
            if hi >= lo:
                lists.update((lo, hi))
    rows = []
    for u in sorted(lists):
        s1, n2, b = u % case.S1, (u // case.S1) % case.N2, u // (case.S1 * case.N2)
        rows += [[b, n2 * case.G, s1], [b, n2 * case.G + case.G - 1, s1]]
    return np.array(rows, dtype=np.int64)


def test_full_workload_sampled_prefill():
    """Sparse prefill (the oracle needs ~1.7 ms per row): random rows, the
    fully masked rows (b = 0, s1 < 8), the last rows, and the first and last
    index list of every persistent CTA's range for one and two CTAs per SM."""
    case = synth.PREFILL
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out, lse = T.run_gpu(case, dev)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = T.sample_rows(case, 64)
    extra = np.array([[0, n1, s1] for n1 in (0, 63) for s1 in (0, 7, 8)] +
                     [[1, 5, 2047], [1, 63, 2046]])
    rows = np.unique(np.concatenate([rows, extra,
                                     aligned_range_boundary_rows(case, (sms, 2 * sms))]), axis=0)
    assert len(rows) > 500
    T.check_rows(case, d, out, lse, rows)
    assert torch.isfinite(out.float()).all()
    assert torch.all(out[0, :8] == 0)


# ---------------------------------------------------------------------------
# small-group decode path (G <= 8, Dk == Dv, G * Dk <= 512)

@pytest.mark.parametrize("D,G,N2", [(64, 1, 2), (64, 2, 2), (64, 4, 1), (64, 8, 2), (128, 1, 3),
                                    (128, 2, 2), (128, 4, 2), (256, 1, 1), (256, 2, 2)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_path_shapes(D, G, N2, dtype):
    run_and_check(small(Dk=D, Dv=D, N1=G * N2, N2=N2, S1=2, topK=150, S2=400, dtype=dtype,
                        causal=True, layout="BNSD"))


@pytest.mark.parametrize("splits", [1, 2, 5, 16])
def test_decode_multi_chunk_online_softmax(splits):
    """Several 64-slot chunks per CTA (online rescaling across chunks)."""
    case = small(Dk=128, Dv=128, N1=16, N2=4, S1=1, topK=1000, S2=3000, causal=True,
                 index_kind="sorted")
    run_and_check(case, num_splits=splits)


def test_decode_fully_masked_rows():
    case = small(Dk=128, Dv=128, N1=8, N2=2, S1=12, S2=64, topK=40, causal=True,
                 index_kind="causal_mix", masked_frac=0.2, full_masked_rows=6)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for splits in (1, 2):
        out, lse = T.run_gpu(case, dev, num_splits=splits)
        T.check_full(case, d, out, lse)
        assert torch.all(out[0, :6] == 0) and torch.all(torch.isneginf(lse[0, :6]))


@pytest.mark.parametrize("B,S1,N2,topK,S2", [(8, 64, 4, 64, 256),     # one chunk per index list
                                             (4, 50, 4, 150, 400),    # ranges span several lists
                                             (1, 1, 1, 1000, 3000),   # one list over many CTAs
                                             (3, 7, 2, 1, 9),         # topK = 1
                                             (8, 400, 2, 128, 512)])  # many lists: whole lists per CTA
def test_decode_stream_k_partitions(B, S1, N2, topK, S2):
    """The persistent decode kernel's contiguous chunk ranges: lists written
    directly by one CTA, lists split across CTAs (merged by the combine), and
    CTAs whose ranges cross list boundaries."""
    case = small(B=B, S1=S1, N1=4 * N2, N2=N2, Dk=128, Dv=128, topK=topK, S2=S2, causal=True,
                 layout="BSND", dtype="f16")
    run_and_check(case)


@pytest.mark.parametrize("schedule", ["cluster", "stream_k", "many_lists"])
def test_inputs_ready_back_to_back(schedule):
    """sfa_options.inputs_ready: four calls on different inputs issued back to
    back on one stream with no synchronisation, so each call's gather may run
    while the previous call is still writing; the four outputs must all equal
    the oracle's.  Schedules: lists cut into segments merged in a cluster;
    ranges that split lists, merged through the library workspace's counters
    (which a call may touch only once the previous one is done); whole lists
    per CTA."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if schedule == "many_lists":
        case = small(B=4, S1=320, N1=8, N2=2, topK=100, S2=600, causal=True, seed=41)
        opts = {}
    else:
        B = max(1, (2 * sms) // 2 // 4)
        case = small(B=B, S1=2, N1=8, N2=2, topK=512, S2=900, causal=True, layout="BNSD", seed=42)
        opts = {} if schedule == "cluster" else {"num_ctas": 7}
    inputs = [synth.make_sfa_inputs(case.replace(seed=case.seed + t)) for t in range(4)]
    devs = [T.to_dev(d) for d in inputs]
    torch.cuda.synchronize()
    results = [sfa.sparse_flash_attention(dv["q"], dv["k"], dv["v"], dv["idx"], case.scale,
                                          case.layout, case.causal, return_lse=True,
                                          inputs_ready=True, **opts) for dv in devs]
    torch.cuda.synchronize()
    for d, (out, lse) in zip(inputs, results):
        T.check_full(case, d, out, lse)
    assert sfa.sfa_get_last_error() == sfa.SFA_OK


@pytest.mark.parametrize("seg,topK,mix", [(2, 1024, False), (3, 1000, True), (5, 1000, False),
                                          (7, 700, True), (8, 450, False), (8, 300, True)])
def test_decode_cluster_merge(seg, topK, mix):
    """Fewer index lists than resident CTAs (two per SM at these dims): each
    list is cut into `seg` segments that run as one thread-block cluster and
    merge through distributed shared memory -- ragged segments where the chunk
    count is no multiple of seg, fewer segments than asked where a list holds
    fewer chunks (topK = 300: 5 chunks), and, with `mix`, slots and whole
    lists masked by the causal rule (empty partials in the merge).  The same
    shape with the grid size forced takes the merge through the workspace;
    both must match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N2, S1 = 2, 2
    B = max(1, (2 * sms) // seg // (N2 * S1))
    kw = dict(index_kind="causal_mix", masked_frac=0.3, full_masked_rows=1) if mix else {}
    case = small(B=B, S1=S1, N1=4 * N2, N2=N2, Dk=128, Dv=128, topK=topK, S2=topK + 300,
                 causal=True, layout="BSND", dtype="bf16", seed=900 + seg, **kw)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for opts in ({}, {"num_ctas": B * S1 * N2 * seg}):
        out, lse = T.run_gpu(case, dev, **opts)
        T.check_full(case, d, out, lse)
        if mix:
            assert torch.all(out[0, 0] == 0) and torch.all(torch.isneginf(lse[0, 0]))
    assert sfa.sfa_get_last_error() == sfa.SFA_OK


def test_workspace_shared_across_shapes():
    """Calls of different shapes and paths share the library-owned workspace:
    split partials of the generic path must never land in the arrival
    counters of the decode path (and the counters must be left at zero)."""
    cases = [small(N1=16, N2=1, topK=200, S2=300),                       # generic, splits
             small(B=4, S1=50, N1=16, N2=4, topK=150, S2=400, causal=True),   # decode, stream-K merge
             small(N1=32, N2=2, topK=300, S2=300, S1=1),                 # generic again
             small(B=2, S1=3, N1=8, N2=2, topK=900, S2=1000)]            # decode again
    for rep in range(2):
        for case in cases:
            run_and_check(case)


# ---------------------------------------------------------------------------
# many index lists (at least four per CTA) of small groups: 9 to 16 query
# heads per list (Dv = 128, Dk in {128, 192, 256}) take the tensor-core kernel
# (slots on the MMA's M side in 128-slot chunks, whole lists per CTA), up to 8
# the warp-MMA kernel's whole-list schedule.  num_ctas shrinks the grid so
# that small shapes take these schedules.

def tc_case(**kw):
    base = dict(name="tc", B=2, S1=24, S2=600, N1=24, N2=2, Dk=128, Dv=128, topK=300,
                dtype="bf16", layout="BSND", causal=True, scale=0.09, seed=5151)
    base.update(kw)
    return synth.SfaCase(**base)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 9, 12, 16])
@pytest.mark.parametrize("Dk,prefix", [(128, False), (128, True), (192, True), (256, False),
                                       (256, True)])
def test_group_tc_shapes(G, Dk, prefix):
    case = tc_case(N1=2 * G, Dk=Dk, value_is_key_prefix=prefix, dtype="f16" if G % 2 else "bf16",
                   seed=5200 + G)
    run_and_check(case, num_ctas=8)


@pytest.mark.parametrize("topK,S2", [(1, 30), (100, 300), (128, 128), (129, 400), (255, 256),
                                     (640, 2000)])
def test_group_tc_ragged_topk(topK, S2):
    """Partial last chunks (slots past topK zero-filled and masked), a single
    slot, exactly one chunk, and topK = S2."""
    run_and_check(tc_case(topK=topK, S2=S2, N1=32, N2=2, seed=5300 + topK), num_ctas=6)


@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_group_tc_layouts_dtypes(layout, dtype, causal):
    run_and_check(tc_case(layout=layout, dtype=dtype, causal=causal, S1=40, S2=200, topK=170),
                  num_ctas=10)


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 0])
def test_group_tc_grid_sizes(num_ctas):
    """Ranges of whole index lists: one CTA for everything, ragged ranges
    (lists % CTAs != 0), and the default one-per-SM grid (640 lists)."""
    case = tc_case(B=4, S1=80, N1=20, N2=2, topK=200, S2=500, seed=5400 + num_ctas)
    run_and_check(case, num_ctas=num_ctas)


def test_group_tc_masked_rows_and_rescale():
    """Whole lists above the causal diagonal (+0 rows, lse = -inf) and a large
    scale: scores grow across chunks by far more than the lazy-rescale
    threshold, so O is rescaled many times."""
    case = tc_case(S1=40, S2=700, topK=600, N1=32, N2=2, index_kind="causal_mix",
                   masked_frac=0.3, full_masked_rows=5, scale=1.5)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out, lse = T.run_gpu(case, dev, num_ctas=8)
    T.check_full(case, d, out, lse)
    assert torch.all(out[0, :5] == 0) and torch.all(torch.isneginf(lse[0, :5]))


def test_group_tc_out_of_range_indices():
    case = tc_case(topK=200, S2=400, S1=20)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    bad = dev["idx"].clone()
    bad[1, 3, 1, 5:9] = torch.tensor([-1, 400, 1 << 30, -(1 << 30)], dtype=torch.int32)
    out, lse = T.run_gpu(case, dict(dev, idx=bad), validate_indices=True, num_ctas=5)
    assert sfa.sfa_get_last_error() == sfa.SFA_ERR_INDEX_RANGE
    # the bad slots of list (b 1, s1 3, n2 1) act as masked: the same as slots
    # whose index lies above that list's causal diagonal (s1 + S2 - S1 = 383)
    d2 = dict(d)
    d2["idx"] = d["idx"].clone()
    d2["idx"][1, 3, 1, 5:9] = 399
    T.check_full(case, d2, out, lse)


def test_group_tc_and_cuda_core_kernels_agree_with_oracle():
    """The same many-list shape of 16 heads per list on the tensor-core kernel
    and on the CUDA-core kernel (a forced split count selects the latter)."""
    case = tc_case(S1=40, N1=64, N2=4, topK=256, S2=512, dtype="f16")
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for opts in ({"num_ctas": 8}, {"num_splits": 2}):
        out, lse = T.run_gpu(case, dev, **opts)
        T.check_full(case, d, out, lse)


# ---------------------------------------------------------------------------
# MLA tensor-core path (128 heads per index list, Dk = 576, Dv = 512, value =
# key prefix): 2-CTA clusters, stream-K with in-kernel merge

def mla(**kw):
    base = dict(name="mla", B=2, S1=2, S2=700, N1=128, N2=1, Dk=576, Dv=512, topK=300,
                dtype="bf16", layout="BSND", causal=False, scale=1 / math.sqrt(576),
                value_is_key_prefix=True, seed=777)
    base.update(kw)
    return synth.SfaCase(**base)


@pytest.mark.parametrize("layout", ["BSND", "BNSD"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_mla_path_layouts_dtypes(layout, dtype, causal):
    run_and_check(mla(layout=layout, dtype=dtype, causal=causal))


def test_mla_two_kv_heads():
    run_and_check(mla(B=3, S1=1, N1=256, N2=2, topK=200, S2=500, causal=True))


@pytest.mark.parametrize("topK", [1, 63, 64, 65, 129])
def test_mla_ragged_topk(topK):
    run_and_check(mla(topK=topK, S2=max(topK, 150), S1=3, causal=True, index_kind="sorted"))


def test_mla_fully_masked_rows():
    case = mla(B=2, S1=6, S2=90, topK=70, causal=True, index_kind="causal_mix",
               masked_frac=0.3, full_masked_rows=3)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    out, lse = T.run_gpu(case, dev)
    T.check_full(case, d, out, lse)
    assert torch.all(out[0, :3] == 0) and torch.all(torch.isneginf(lse[0, :3]))


@pytest.mark.parametrize("num_ctas", [2, 6, 20, 0])
def test_mla_cluster_schedules(num_ctas):
    """One cluster walking every unit; a few clusters whose ranges split
    units (merged in-kernel by the last to finish); the resident-cluster
    default where most units are split.  Each case runs twice: the merge
    counters must be back at zero after a call."""
    case = mla(B=5, S1=3, topK=260, S2=600, causal=True)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for _ in range(2):
        out, lse = T.run_gpu(case, dev, num_ctas=num_ctas)
        T.check_full(case, d, out, lse)


@pytest.mark.parametrize("B,S1,causal,dtype,layout", [(32, 1, False, "bf16", "BSND"),
                                                       (1, 32, True, "bf16", "BSND"),
                                                       (1, 32, True, "f16", "BNSD")])
def test_mla_two_range_units_merge_in_cluster(B, S1, causal, dtype, layout):
    """32 index lists of 128 heads with 4 chunks each: with 64-127 resident
    CTA pairs every list is cut into two ranges whose pairs run as one 4-CTA
    cluster and merge in distributed shared memory -- one kernel launch per
    call, no merge kernel.  The MLA decode batch shape (B = 32, one query
    row), and 32 causal query rows of one batch whose first two rows select
    only keys above the diagonal (+0, lse -inf after the merge)."""
    extra = dict(index_kind="causal_mix", masked_frac=0.1, full_masked_rows=2) if causal else {}
    case = mla(B=B, S1=S1, S2=2048, topK=256, causal=causal, dtype=dtype, layout=layout, **extra)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    for _ in range(2):
        before = sfa.sfa_kernel_launches()
        out, lse = T.run_gpu(case, dev)
        assert sfa.sfa_kernel_launches() - before == 1
        T.check_full(case, d, out, lse)
    if causal:
        rows_out = out[0, :2] if layout == "BSND" else out[0, :, :2]
        rows_lse = lse[0, :2] if layout == "BSND" else lse[0, :, :2]
        assert torch.all(rows_out == 0) and torch.all(torch.isneginf(rows_lse))


@pytest.mark.parametrize("schedule", ["cluster_merge", "merge_kernel", "whole_lists"])
def test_mla_inputs_ready_back_to_back(schedule):
    """sfa_options.inputs_ready on the MLA path: four calls on different inputs
    issued back to back with no synchronisation (each may gather while the
    previous call still runs); every output must equal the oracle's.
    Schedules: two ranges per list merged in a 4-CTA cluster; ranges merged by
    the merge kernel (forced CTA count); whole lists per pair."""
    if schedule == "whole_lists":
        case = mla(B=2, S1=24, S2=600, topK=64, causal=True, seed=31)   # 48 one-chunk lists
        opts = {}
    else:
        case = mla(B=32, S1=1, S2=1024, topK=256, seed=32)
        opts = {} if schedule == "cluster_merge" else {"num_ctas": 10}
    inputs = [synth.make_sfa_inputs(case.replace(seed=case.seed + t)) for t in range(4)]
    devs = [T.to_dev(d) for d in inputs]
    torch.cuda.synchronize()
    results = [sfa.sparse_flash_attention(dv["q"], dv["k"], dv["v"], dv["idx"], case.scale,
                                          case.layout, case.causal, return_lse=True,
                                          inputs_ready=True, **opts) for dv in devs]
    torch.cuda.synchronize()
    for d, (out, lse) in zip(inputs, results):
        T.check_full(case, d, out, lse)


def test_mla_out_of_range_indices_masked_and_reported():
    """Indices outside [0, S2) act as masked slots and set the error word."""
    case = mla(B=1, S1=2, topK=130, S2=400)
    d = synth.make_sfa_inputs(case)
    dev = T.to_dev(d)
    bad = dev["idx"].clone()
    bad_slots = {0: [0, 1, 2, 3, 4], 1: [7, 100]}
    bad[0, 0, 0, :5] = -1
    bad[0, 1, 0, 7] = 400
    bad[0, 1, 0, 100] = 1 << 30
    assert sfa.sfa_get_last_error() == sfa.SFA_OK
    out, lse = T.run_gpu(case, dict(dev, idx=bad), validate_indices=True)
    assert sfa.sfa_get_last_error() == sfa.SFA_ERR_INDEX_RANGE
    for s1, drop in bad_slots.items():
        keep = np.delete(d["idx"][0, s1, 0].numpy(), drop)
        sub = {"q": d["q"][:, s1:s1 + 1].contiguous(), "k": d["k"],
               "idx": torch.from_numpy(keep).reshape(1, 1, 1, -1).contiguous()}
        sub["v"] = sub["k"][..., :case.Dv]
        y, l = oracle.sfa(sub["q"], sub["k"], sub["v"], sub["idx"], case.scale, "BSND", False)
        got = out[0, s1].float().cpu().numpy()
        rep = oracle.precision_report(got, y[0, 0], case.dtype)
        assert rep["passed"], rep
        np.testing.assert_allclose(lse[0, s1].cpu().numpy(), l[0, 0], atol=T.LSE_ATOL,
                                   rtol=T.LSE_RTOL)
