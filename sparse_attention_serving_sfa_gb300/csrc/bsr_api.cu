// C ABI of the block-sparse path ("flashinfer.sparse",
// BlockSparseAttentionWrapper): plan() validates the BSR pattern on the host
// and uploads it with a row-tile work list into the caller's int workspace;
// run() launches the kernels with that plan.
#include <math.h>

#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct bsr_plan_s {
    int M, N, R, C, Hq, Hkv, d;
    sfa_dtype dtype;
    float scale;
    int MB, NB, nnz, ntiles;
    bool tc;                        // tensor-core path (work items) vs generic (row tiles)
    int mask_mode;                  // 0 none, 1 causal, 2 per-element bits
    float softcap_log2 = 0.f;       // logits_soft_cap * log2(e); 0 = none
    int kv_layout = SFA_KV_LAYOUT_NHD;
    // plan()'s q_data_type / kv_data_type / o_data_type (all `dtype` unless set)
    sfa_dtype q_dtype, kv_dtype, o_dtype;
    const int32_t* d_indptr;
    const int32_t* d_indices;
    const void* d_work;             // BsrTile list (generic) or 4-int items (tensor cores)
    const uint8_t* d_mask;          // packed element mask (mode 2)
    std::vector<int32_t> staging;   // host copy kept alive for the async upload
};

namespace {

constexpr int kTileRows = 64;

size_t round4(size_t n) { return (n + 3) & ~size_t(3); }

// Row tiles of `rows_per` rows (never crossing a block row).
int count_tiles(int M, int R, int rows_per = kTileRows) {
    const int MB = (M + R - 1) / R;
    int n = 0;
    for (int rb = 0; rb < MB; ++rb) {
        const int rows = std::min(R, M - rb * R);
        n += (rows + rows_per - 1) / rows_per;
    }
    return n;
}

// Work entries of either path (4 ints each).
int count_work(int M, int R, int C, int Hq, int Hkv, int d) {
    if (sfa::bsr_tc_supported(d, C, Hq, Hkv))
        return count_tiles(M, R, sfa::bsr_tc_rows_per_item(Hq, Hkv)) * Hkv;
    return count_tiles(M, R);
}

sfa_status check_shape(int M, int N, int R, int C, int Hq, int Hkv, int d) {
    if (M < 1 || N < 1 || R < 1 || C < 1 || Hq < 1 || Hkv < 1 || d < 1) return SFA_ERR_INVALID_ARG;
    if (N % C != 0) return SFA_ERR_INVALID_ARG;        // NB = N / C, N divisible by C
    if (Hq % Hkv != 0) return SFA_ERR_INVALID_ARG;     // qo heads a multiple of kv heads
    if (d % 64 != 0) return SFA_ERR_INVALID_ARG;
    if (d > 256) return SFA_ERR_UNSUPPORTED;
    return SFA_OK;
}

size_t int_ws_bytes(int MB, int nnz, int ntiles) {
    return 4 * (round4((size_t)MB + 1) + round4((size_t)nnz) + 4 * (size_t)ntiles);
}

// Bytes of the packed element mask: nnz * R * C bits, rounded up to 16.
size_t mask_bytes(int nnz, int R, int C) {
    const size_t bits = (size_t)nnz * (size_t)R * (size_t)C;
    return (((bits + 7) / 8) + 15) & ~size_t(15);
}

}  // namespace

extern "C" {

sfa_status bsr_plan_int_workspace_size(const int32_t* indptr_host, int M, int N, int R, int C,
                                       int num_qo_heads, int num_kv_heads, int head_dim,
                                       size_t* bytes) {
    if (!indptr_host || !bytes) return SFA_ERR_INVALID_ARG;
    sfa_status st = check_shape(M, N, R, C, num_qo_heads, num_kv_heads, head_dim);
    if (st != SFA_OK) return st;
    const int MB = (M + R - 1) / R;
    const int nnz = indptr_host[MB];
    if (nnz < 0) return SFA_ERR_INVALID_ARG;
    *bytes = int_ws_bytes(MB, nnz, count_work(M, R, C, num_qo_heads, num_kv_heads, head_dim));
    return SFA_OK;
}

sfa_status bsr_plan_masked_int_workspace_size(const int32_t* indptr_host, int M, int N, int R,
                                              int C, int num_qo_heads, int num_kv_heads,
                                              int head_dim, int with_mask, size_t* bytes) {
    sfa_status st = bsr_plan_int_workspace_size(indptr_host, M, N, R, C, num_qo_heads,
                                                num_kv_heads, head_dim, bytes);
    if (st != SFA_OK || !with_mask) return st;
    const int MB = (M + R - 1) / R;
    *bytes += mask_bytes(indptr_host[MB], R, C);
    return SFA_OK;
}

sfa_status bsr_plan(const int32_t* indptr_host, const int32_t* indices_host, int M, int N,
                    int R, int C, int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                    float sm_scale, sfa_dtype dtype, void* int_ws, size_t int_ws_bytes_given,
                    void* float_ws, size_t float_ws_bytes, sfa_stream_t stream,
                    bsr_plan_t* plan_out) {
    return bsr_plan_masked(indptr_host, indices_host, nullptr, M, N, R, C, num_qo_heads,
                           num_kv_heads, head_dim, causal, sm_scale, dtype, int_ws,
                           int_ws_bytes_given, float_ws, float_ws_bytes, stream, plan_out);
}

sfa_status bsr_plan_masked(const int32_t* indptr_host, const int32_t* indices_host,
                           const uint8_t* packed_mask_host, int M, int N, int R, int C,
                           int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                           float sm_scale, sfa_dtype dtype, void* int_ws,
                           size_t int_ws_bytes_given, void* float_ws, size_t float_ws_bytes,
                           sfa_stream_t stream, bsr_plan_t* plan_out) {
    (void)float_ws;
    (void)float_ws_bytes;
    if (!plan_out || !indptr_host) return SFA_ERR_INVALID_ARG;
    *plan_out = nullptr;
    sfa_status st = check_shape(M, N, R, C, num_qo_heads, num_kv_heads, head_dim);
    if (st != SFA_OK) return st;
    if (dtype != SFA_DTYPE_F16 && dtype != SFA_DTYPE_BF16) return SFA_ERR_INVALID_ARG;
    if (!isfinite(sm_scale)) return SFA_ERR_INVALID_ARG;
    const int MB = (M + R - 1) / R, NB = N / C;
    // indptr: starts at 0, non-decreasing
    if (indptr_host[0] != 0) return SFA_ERR_INVALID_ARG;
    for (int i = 0; i < MB; ++i)
        if (indptr_host[i + 1] < indptr_host[i]) return SFA_ERR_INVALID_ARG;
    const int nnz = indptr_host[MB];
    if (nnz > 0 && !indices_host) return SFA_ERR_INVALID_ARG;
    // indices: each block column in [0, NB), at most once per block row
    {
        std::vector<unsigned char> seen((size_t)NB, 0);
        for (int i = 0; i < MB; ++i) {
            for (int j = indptr_host[i]; j < indptr_host[i + 1]; ++j) {
                const int c = indices_host[j];
                if (c < 0 || c >= NB || seen[(size_t)c]) return SFA_ERR_INVALID_ARG;
                seen[(size_t)c] = 1;
            }
            for (int j = indptr_host[i]; j < indptr_host[i + 1]; ++j) seen[(size_t)indices_host[j]] = 0;
        }
    }
    // masked elements: the per-element mask wins over causal (plan() applies
    // causal only without a mask); its bit index must fit an int
    const int mask_mode = packed_mask_host ? 2 : (causal ? 1 : 0);
    if (mask_mode == 2 && (int64_t)nnz * R * C > (int64_t)INT32_MAX) return SFA_ERR_UNSUPPORTED;
    // causal: blocks entirely above the bottom-right diagonal drop out (no
    // element of them is visible); the kernels test the others per element
    std::vector<int32_t> f_indptr(indptr_host, indptr_host + MB + 1);
    std::vector<int32_t> f_indices(indices_host ? indices_host : indptr_host,
                                   indices_host ? indices_host + nnz : indptr_host);
    if (mask_mode == 1) {
        f_indptr[0] = 0;
        f_indices.clear();
        for (int i = 0; i < MB; ++i) {
            const int64_t last_row = std::min((int64_t)(i + 1) * R, (int64_t)M) - 1;
            for (int j = indptr_host[i]; j < indptr_host[i + 1]; ++j)
                if ((int64_t)indices_host[j] * C <= last_row + (N - M)) f_indices.push_back(indices_host[j]);
            f_indptr[i + 1] = (int32_t)f_indices.size();
        }
    }
    const int f_nnz = f_indptr[MB];
    const bool tc = sfa::bsr_tc_supported(head_dim, C, num_qo_heads, num_kv_heads);
    const int ntiles = count_work(M, R, C, num_qo_heads, num_kv_heads, head_dim);
    const size_t base_bytes = int_ws_bytes(MB, f_nnz, ntiles);
    const size_t need = base_bytes + (mask_mode == 2 ? mask_bytes(nnz, R, C) : 0);
    if (!int_ws || int_ws_bytes_given < need) return SFA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(int_ws) & 15u) return SFA_ERR_INVALID_ARG;

    bsr_plan_s* plan = new (std::nothrow) bsr_plan_s();
    if (!plan) return SFA_ERR_INVALID_ARG;
    plan->M = M; plan->N = N; plan->R = R; plan->C = C;
    plan->Hq = num_qo_heads; plan->Hkv = num_kv_heads; plan->d = head_dim;
    plan->dtype = dtype;
    plan->q_dtype = plan->kv_dtype = plan->o_dtype = dtype;
    plan->scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)head_dim);
    plan->MB = MB; plan->NB = NB; plan->nnz = f_nnz; plan->ntiles = ntiles;
    plan->tc = tc;
    plan->mask_mode = mask_mode;

    // Work list: generic row tiles of <= 64 rows (the kernel's grid.y spans
    // the qo heads), heaviest block rows first, or tensor-core items of
    // (block row, first row, kv head).
    std::vector<sfa::BsrTile> tiles;
    tiles.reserve((size_t)ntiles);
    const int rows_per = tc ? sfa::bsr_tc_rows_per_item(num_qo_heads, num_kv_heads) : kTileRows;
    for (int rb = 0; rb < MB; ++rb) {
        const int rows = std::min(R, M - rb * R);
        for (int r0 = 0; r0 < rows; r0 += rows_per) {
            if (tc) {
                for (int h = 0; h < num_kv_heads; ++h) tiles.push_back({rb, rb * R + r0, h, 0});
            } else {
                tiles.push_back({rb, rb * R + r0, std::min(kTileRows, rows - r0), 0});
            }
        }
    }
    // tensor-core items go kv head by kv head (the third int), so that the
    // CTAs resident at one time share one head's K / V (a few MB, kept in L2
    // while q and out stream through), heaviest block rows first within a
    // head
    std::stable_sort(tiles.begin(), tiles.end(), [&](const sfa::BsrTile& a, const sfa::BsrTile& b) {
        if (tc && a.nrows != b.nrows) return a.nrows < b.nrows;
        return (f_indptr[a.rb + 1] - f_indptr[a.rb]) > (f_indptr[b.rb + 1] - f_indptr[b.rb]);
    });

    const size_t n_indptr = round4((size_t)MB + 1), n_indices = round4((size_t)f_nnz);
    plan->staging.assign(need / 4, 0);
    std::copy(f_indptr.begin(), f_indptr.end(), plan->staging.begin());
    if (f_nnz) std::copy(f_indices.begin(), f_indices.end(), plan->staging.begin() + n_indptr);
    std::copy(reinterpret_cast<const int32_t*>(tiles.data()),
              reinterpret_cast<const int32_t*>(tiles.data()) + 4 * tiles.size(),
              plan->staging.begin() + n_indptr + n_indices);
    if (mask_mode == 2) {
        const size_t mbits = (size_t)nnz * R * C;
        std::memcpy(reinterpret_cast<unsigned char*>(plan->staging.data()) + base_bytes,
                    packed_mask_host, (mbits + 7) / 8);
    }
    int32_t* base = static_cast<int32_t*>(int_ws);
    plan->d_indptr = base;
    plan->d_indices = base + n_indptr;
    plan->d_work = base + n_indptr + n_indices;
    plan->d_mask = mask_mode == 2 ? reinterpret_cast<const uint8_t*>(
                                        static_cast<unsigned char*>(int_ws) + base_bytes)
                                  : nullptr;
    cudaError_t err = cudaMemcpyAsync(int_ws, plan->staging.data(), need, cudaMemcpyHostToDevice,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) {
        delete plan;
        return SFA_ERR_CUDA;
    }
    *plan_out = plan;
    return SFA_OK;
}

sfa_status bsr_run_scaled(bsr_plan_t plan, const void* q, const void* k, const void* v,
                          const float* scale_q, const float* scale_k, const float* scale_v,
                          void* out, float* lse, sfa_stream_t stream) {
    if (!plan || !q || !k || !v || !out) return SFA_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return SFA_ERR_INVALID_ARG;
    if ((lse && !a4(lse)) || (scale_q && !a4(scale_q)) || (scale_k && !a4(scale_k)) ||
        (scale_v && !a4(scale_v)))
        return SFA_ERR_INVALID_ARG;
    const bool f8 = plan->kv_dtype == SFA_DTYPE_E4M3 || plan->kv_dtype == SFA_DTYPE_E5M2;
    // per-head scales are the FP8 path's (run(): "for FP8 quantisation")
    if (!f8 && (scale_q || scale_k || scale_v)) return SFA_ERR_UNSUPPORTED;
    if (f8 && plan->softcap_log2 > 0.f) return SFA_ERR_UNSUPPORTED;
    sfa::BsrParams p{};
    p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse;
    p.indptr = plan->d_indptr;
    p.indices = plan->d_indices;
    p.tiles = static_cast<const sfa::BsrTile*>(plan->d_work);
    p.ntiles = plan->ntiles;
    p.M = plan->M; p.N = plan->N; p.R = plan->R; p.C = plan->C;
    p.Hq = plan->Hq; p.Hkv = plan->Hkv; p.d = plan->d;
    p.scale_log2 = plan->scale * sfa::kLog2e;
    p.mask_mode = plan->mask_mode;
    p.mask = plan->d_mask;
    p.softcap_log2 = plan->softcap_log2;
    p.kv_hnd = plan->kv_layout == SFA_KV_LAYOUT_HND ? 1 : 0;
    p.f8 = !f8 ? 0 : (plan->kv_dtype == SFA_DTYPE_E4M3 ? 1 : 2);
    p.scale_q = scale_q;
    p.scale_k = scale_k;
    p.scale_v = scale_v;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (f8) {
        int* ew = sfa::device_error_word();
        if (!ew) return SFA_ERR_CUDA;
        // the 128-key tensor-core kernel's FP8 instantiations; `dtype` = out's
        err = sfa::launch_bsr_tc_wide(p, plan->d_work, plan->ntiles, ew, plan->o_dtype, s);
    } else if (plan->tc) {
        int* ew = sfa::device_error_word();
        if (!ew) return SFA_ERR_CUDA;
        // per-element mask: 64-key blocks (measured faster); otherwise 128-key steps
        err = plan->mask_mode == 2
                  ? sfa::launch_bsr_tc(p, plan->d_work, plan->ntiles, ew, plan->dtype, s)
                  : sfa::launch_bsr_tc_wide(p, plan->d_work, plan->ntiles, ew, plan->dtype, s);
    } else {
        err = sfa::launch_bsr_generic(p, plan->dtype, s);
    }
    return err == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

sfa_status bsr_run(bsr_plan_t plan, const void* q, const void* k, const void* v, void* out,
                   float* lse, sfa_stream_t stream) {
    return bsr_run_scaled(plan, q, k, v, nullptr, nullptr, nullptr, out, lse, stream);
}

sfa_status bsr_plan_set_data_types(bsr_plan_t plan, sfa_dtype q_dtype, sfa_dtype kv_dtype,
                                   sfa_dtype o_dtype) {
    auto known = [](int t) { return t >= SFA_DTYPE_F16 && t <= SFA_DTYPE_E5M2; };
    if (!plan || !known(q_dtype) || !known(kv_dtype) || !known(o_dtype))
        return SFA_ERR_INVALID_ARG;
    const bool wide16 = o_dtype == SFA_DTYPE_F16 || o_dtype == SFA_DTYPE_BF16;
    if (q_dtype == kv_dtype && kv_dtype == o_dtype && wide16) {
        if (o_dtype != plan->dtype) return SFA_ERR_UNSUPPORTED;   // the plan's own kernels
    } else {
        // FP8: q and k / v of one 8-bit format, 16-bit out, on the 128-key
        // tensor-core kernel (head_dim 128, plain or causal blocks)
        const bool f8 = kv_dtype == SFA_DTYPE_E4M3 || kv_dtype == SFA_DTYPE_E5M2;
        if (!f8 || q_dtype != kv_dtype || !wide16) return SFA_ERR_UNSUPPORTED;
        if (!plan->tc || plan->d != 128 || plan->mask_mode == 2) return SFA_ERR_UNSUPPORTED;
    }
    plan->q_dtype = q_dtype;
    plan->kv_dtype = kv_dtype;
    plan->o_dtype = o_dtype;
    return SFA_OK;
}

sfa_status bsr_plan_set_logits_soft_cap(bsr_plan_t plan, float logits_soft_cap) {
    if (!plan || !isfinite(logits_soft_cap)) return SFA_ERR_INVALID_ARG;
    plan->softcap_log2 = logits_soft_cap > 0.f ? logits_soft_cap * sfa::kLog2e : 0.f;
    return SFA_OK;
}

sfa_status bsr_plan_set_kv_layout(bsr_plan_t plan, sfa_kv_layout kv_layout) {
    if (!plan || (kv_layout != SFA_KV_LAYOUT_NHD && kv_layout != SFA_KV_LAYOUT_HND))
        return SFA_ERR_INVALID_ARG;
    plan->kv_layout = kv_layout;
    return SFA_OK;
}

void bsr_plan_destroy(bsr_plan_t plan) { delete plan; }

}  // extern "C"
