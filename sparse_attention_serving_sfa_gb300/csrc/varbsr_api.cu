// C ABI of the variable block-sparse path ("flashinfer.sparse",
// VariableBlockSparseAttentionWrapper): plan() turns each kv head's block
// mask map and block sizes into key window lists and a work list, uploads them
// into the caller's int workspace; run() launches the tensor-core BSR kernel
// in its variable mode with that plan.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct varbsr_plan_s {
    int M, N, MB, NB, Hq, Hkv, d;
    sfa_dtype dtype;
    float scale;
    int causal;
    float softcap_log2 = 0.f;       // logits_soft_cap * log2(e); 0 = none
    int nlists, ntiles, nitems;
    const int32_t* d_lists;
    const int32_t* d_tiles;
    const void* d_items;
    std::vector<int32_t> staging;   // host copy kept alive for the async upload
};

namespace {

constexpr int kTileKeys = 64;   // keys of a window (four 16-key quarters)
constexpr int kQuarterKeys = 16;
constexpr int kWindowInts = 6;  // first key of each quarter, then the 64-bit mask (low word first)

size_t round4(size_t n) { return (n + 3) & ~size_t(3); }

struct Built {
    int M = 0, N = 0;
    std::vector<int32_t> lists;     // nlists + 1 offsets into tiles
    std::vector<int32_t> tiles;     // kWindowInts ints per key window
    std::vector<int32_t> items;     // 4 ints each: list, row0, kv head, row end
};

sfa_status check_args(const uint8_t* mm, const int32_t* rs, const int32_t* cs, int MB, int NB,
                      int Hq, int Hkv, int d) {
    if (!mm || !rs || !cs) return SFA_ERR_INVALID_ARG;
    if (MB < 1 || NB < 1 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0) return SFA_ERR_INVALID_ARG;
    if ((int64_t)Hkv * MB * NB > (int64_t)INT32_MAX) return SFA_ERR_UNSUPPORTED;
    // the tensor-core kernel: head_dim 64 or 128, Hq / Hkv divides 128
    if (!sfa::bsr_tc_supported(d, kTileKeys, Hq, Hkv)) return SFA_ERR_UNSUPPORTED;
    return SFA_OK;
}

// Key windows of one (kv head, row block): the allowed key columns (set
// blocks, and with causal only keys <= limit) covered greedily by 16-key
// quarters, each starting at the first allowed key not yet covered (the
// fewest quarters that cover the set), four in order to a 64-key window:
// {first key of quarters 0..3, mask low word, mask high word}, bit 16 q + j of
// the mask = key j of quarter q allowed.  A last window with fewer than four
// quarters is completed with empty ones at key n_keys (rows past the end of
// the keys: read as zeros, all masked).
void tile_row_block(const uint8_t* mrow, const int32_t* cs, int NB, int64_t limit,
                    int64_t n_keys, std::vector<int32_t>& tiles) {
    int64_t key0 = -1;                  // the quarter being filled
    uint32_t bits = 0;
    int64_t wkey[4] = {0, 0, 0, 0};     // the window being filled
    uint64_t wmask = 0;
    int nq = 0;
    auto emit_quarter = [&](int64_t k, uint32_t m) {
        wkey[nq] = k;
        wmask |= (uint64_t)m << (16 * nq);
        if (++nq < 4) return;
        for (int q = 0; q < 4; ++q) tiles.push_back((int32_t)wkey[q]);
        tiles.push_back((int32_t)(uint32_t)wmask);
        tiles.push_back((int32_t)(uint32_t)(wmask >> 32));
        nq = 0;
        wmask = 0;
    };
    auto flush = [&] {
        if (key0 >= 0) emit_quarter(key0, bits);
        key0 = -1;
        bits = 0;
    };
    int64_t c0 = 0;
    for (int cb = 0; cb < NB; ++cb) {
        int64_t a = c0;
        const int64_t b = std::min(c0 + cs[cb], limit + 1);
        c0 += cs[cb];
        if (!mrow[cb]) continue;
        while (a < b) {
            if (key0 < 0 || a >= key0 + kQuarterKeys) {
                flush();
                key0 = a;
            }
            const int64_t e = std::min(b, key0 + kQuarterKeys);
            const int o0 = (int)(a - key0), n = (int)(e - a);
            bits |= ((1u << n) - 1u) << o0;         // n <= 16
            a = e;
        }
    }
    flush();
    const int pad = nq > 0 ? 4 - nq : 0;
    for (int i = 0; i < pad; ++i) emit_quarter(n_keys, 0u);
}

sfa_status build(const uint8_t* mm, const int32_t* rs, const int32_t* cs, int MB, int NB, int Hq,
                 int Hkv, int causal, Built& out) {
    // every kv head's row sizes sum to the same qo_len, column sizes to kv_len
    int64_t M = -1, N = -1;
    for (int g = 0; g < Hkv; ++g) {
        int64_t sr = 0, sc = 0;
        for (int b = 0; b < MB; ++b) {
            if (rs[(int64_t)g * MB + b] < 0) return SFA_ERR_INVALID_ARG;
            sr += rs[(int64_t)g * MB + b];
        }
        for (int b = 0; b < NB; ++b) {
            if (cs[(int64_t)g * NB + b] < 0) return SFA_ERR_INVALID_ARG;
            sc += cs[(int64_t)g * NB + b];
        }
        if (g == 0) {
            M = sr;
            N = sc;
        } else if (sr != M || sc != N) {
            return SFA_ERR_INVALID_ARG;
        }
    }
    if (M < 1 || N < 1) return SFA_ERR_INVALID_ARG;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return SFA_ERR_UNSUPPORTED;
    out.M = (int)M;
    out.N = (int)N;
    const int rows_per = sfa::bsr_tc_rows_per_item(Hq, Hkv);
    out.lists.assign(1, 0);
    out.tiles.clear();
    out.items.clear();
    for (int g = 0; g < Hkv; ++g) {
        int64_t r0 = 0;
        for (int rb = 0; rb < MB; ++rb) {
            const int s = rs[(int64_t)g * MB + rb];
            const int list = (int)out.lists.size() - 1;
            if (s > 0) {
                const int64_t limit = causal ? r0 + s - 1 + (N - M) : N - 1;
                tile_row_block(mm + ((int64_t)g * MB + rb) * NB, cs + (int64_t)g * NB, NB, limit, N,
                               out.tiles);
                for (int x = 0; x < s; x += rows_per) {
                    out.items.push_back(list);
                    out.items.push_back((int32_t)(r0 + x));
                    out.items.push_back(g);
                    out.items.push_back((int32_t)(r0 + s));
                }
            }
            if (out.tiles.size() / kWindowInts > (size_t)INT32_MAX) return SFA_ERR_UNSUPPORTED;
            out.lists.push_back((int32_t)(out.tiles.size() / kWindowInts));
            r0 += s;
        }
    }
    // kv head by kv head (CTAs resident at one time share one head's K / V,
    // kept in L2 while q and out stream through), heaviest items first within
    // a head
    const size_t ni = out.items.size() / 4;
    std::vector<int> order(ni);
    for (size_t i = 0; i < ni; ++i) order[i] = (int)i;
    auto weight = [&](int i) {
        const int l = out.items[4 * (size_t)i];
        return out.lists[l + 1] - out.lists[l];
    };
    auto head = [&](int i) { return out.items[4 * (size_t)i + 2]; };
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (head(a) != head(b)) return head(a) < head(b);
        return weight(a) > weight(b);
    });
    std::vector<int32_t> sorted(out.items.size());
    for (size_t i = 0; i < ni; ++i)
        std::copy(out.items.begin() + 4 * (size_t)order[i], out.items.begin() + 4 * (size_t)order[i] + 4,
                  sorted.begin() + 4 * i);
    out.items.swap(sorted);
    return SFA_OK;
}

size_t ws_bytes(const Built& b) {
    // lists, windows and items each start on a 16-byte boundary
    return 4 * (round4(b.lists.size()) + round4(b.tiles.size()) + b.items.size());
}

}  // namespace

extern "C" {

sfa_status varbsr_plan_int_workspace_size(const uint8_t* block_mask_map_host,
                                          const int32_t* block_row_sz_host,
                                          const int32_t* block_col_sz_host, int MB, int NB,
                                          int num_qo_heads, int num_kv_heads, int head_dim,
                                          int causal, size_t* bytes) {
    if (!bytes) return SFA_ERR_INVALID_ARG;
    sfa_status st = check_args(block_mask_map_host, block_row_sz_host, block_col_sz_host, MB, NB,
                               num_qo_heads, num_kv_heads, head_dim);
    if (st != SFA_OK) return st;
    Built b;
    st = build(block_mask_map_host, block_row_sz_host, block_col_sz_host, MB, NB, num_qo_heads,
               num_kv_heads, causal, b);
    if (st != SFA_OK) return st;
    *bytes = ws_bytes(b);
    return SFA_OK;
}

sfa_status varbsr_plan(const uint8_t* block_mask_map_host, const int32_t* block_row_sz_host,
                       const int32_t* block_col_sz_host, int MB, int NB, int num_qo_heads,
                       int num_kv_heads, int head_dim, int causal, float sm_scale,
                       sfa_dtype dtype, void* int_ws, size_t int_ws_bytes, sfa_stream_t stream,
                       varbsr_plan_t* plan_out) {
    if (!plan_out) return SFA_ERR_INVALID_ARG;
    *plan_out = nullptr;
    sfa_status st = check_args(block_mask_map_host, block_row_sz_host, block_col_sz_host, MB, NB,
                               num_qo_heads, num_kv_heads, head_dim);
    if (st != SFA_OK) return st;
    if (dtype != SFA_DTYPE_F16 && dtype != SFA_DTYPE_BF16) return SFA_ERR_INVALID_ARG;
    if (!isfinite(sm_scale)) return SFA_ERR_INVALID_ARG;
    varbsr_plan_s* plan = new (std::nothrow) varbsr_plan_s();
    if (!plan) return SFA_ERR_INVALID_ARG;
    Built b;
    st = build(block_mask_map_host, block_row_sz_host, block_col_sz_host, MB, NB, num_qo_heads,
               num_kv_heads, causal, b);
    if (st != SFA_OK) {
        delete plan;
        return st;
    }
    const size_t need = ws_bytes(b);
    if (!int_ws || int_ws_bytes < need) {
        delete plan;
        return SFA_ERR_WORKSPACE;
    }
    if (reinterpret_cast<uintptr_t>(int_ws) & 15u) {
        delete plan;
        return SFA_ERR_INVALID_ARG;
    }
    plan->M = b.M;
    plan->N = b.N;
    plan->MB = MB;
    plan->NB = NB;
    plan->Hq = num_qo_heads;
    plan->Hkv = num_kv_heads;
    plan->d = head_dim;
    plan->dtype = dtype;
    plan->scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)head_dim);
    plan->causal = causal ? 1 : 0;
    plan->nlists = (int)b.lists.size() - 1;
    plan->ntiles = (int)(b.tiles.size() / kWindowInts);
    plan->nitems = (int)(b.items.size() / 4);
    const size_t n_lists = round4(b.lists.size()), n_tiles = round4(b.tiles.size());
    plan->staging.assign(need / 4, 0);
    std::copy(b.lists.begin(), b.lists.end(), plan->staging.begin());
    std::copy(b.tiles.begin(), b.tiles.end(), plan->staging.begin() + n_lists);
    std::copy(b.items.begin(), b.items.end(), plan->staging.begin() + n_lists + n_tiles);
    int32_t* base = static_cast<int32_t*>(int_ws);
    plan->d_lists = base;
    plan->d_tiles = base + n_lists;
    plan->d_items = base + n_lists + n_tiles;
    cudaError_t err = cudaMemcpyAsync(int_ws, plan->staging.data(), need, cudaMemcpyHostToDevice,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) {
        delete plan;
        return SFA_ERR_CUDA;
    }
    *plan_out = plan;
    return SFA_OK;
}

sfa_status varbsr_plan_dims(varbsr_plan_t plan, int* qo_len, int* kv_len) {
    if (!plan || !qo_len || !kv_len) return SFA_ERR_INVALID_ARG;
    *qo_len = plan->M;
    *kv_len = plan->N;
    return SFA_OK;
}

sfa_status varbsr_run(varbsr_plan_t plan, const void* q, const void* k, const void* v, void* out,
                      float* lse, sfa_stream_t stream) {
    if (!plan || !q || !k || !v || !out) return SFA_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return SFA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SFA_ERR_INVALID_ARG;
    sfa::BsrParams p{};
    p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse;
    p.indptr = plan->d_lists;
    p.indices = plan->d_tiles;
    p.M = plan->M; p.N = plan->N; p.R = 1; p.C = kTileKeys;
    p.Hq = plan->Hq; p.Hkv = plan->Hkv; p.d = plan->d;
    p.scale_log2 = plan->scale * sfa::kLog2e;
    p.mask_mode = 3;
    p.causal = plan->causal;
    p.softcap_log2 = plan->softcap_log2;
    int* ew = sfa::device_error_word();
    if (!ew) return SFA_ERR_CUDA;
    cudaError_t err = sfa::launch_bsr_tc_wide(p, plan->d_items, plan->nitems, ew, plan->dtype,
                                              reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

sfa_status varbsr_plan_set_logits_soft_cap(varbsr_plan_t plan, float logits_soft_cap) {
    if (!plan || !isfinite(logits_soft_cap)) return SFA_ERR_INVALID_ARG;
    plan->softcap_log2 = logits_soft_cap > 0.f ? logits_soft_cap * sfa::kLog2e : 0.f;
    return SFA_OK;
}

void varbsr_plan_destroy(varbsr_plan_t plan) { delete plan; }

}  // extern "C"
