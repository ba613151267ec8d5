// Block-sparse (BSR) attention with plan()'s per-element block mask, on the
// 5th-generation tensor cores (tcgen05), in 64-key blocks.
//
// "flashinfer.sparse", BlockSparseAttentionWrapper: query row i attends to
// key column j iff block (i / R, j / C) is stored and the mask element of
// (i, j) inside that block is set; qo head h reads kv head h / (Hq / Hkv).
// This path takes C a multiple of 64 and head_dim 64 or 128: every stored
// block is a run of dense 64-key blocks of K and V.  (Plain, causal and
// variable blocks run in the 128-key kernel, bsr_tc_wide.cu; with the
// per-element mask this 64-key kernel measured faster.)
//
// CTA = one kv head x 2 M-tiles of 128 query vectors (TR = 128 / G rows of
// one block row x the G qo heads that share the kv head), 9 warps:
//   - control warp (one thread): TMA tiled loads of the two Q tiles and of
//     each 64-key K and V block (128-byte swizzle, three-stage ring), and the
//     tcgen05.mma issue: S_t = Q_t K^T into tensor memory, then O_t += P_t V
//     (P in shared memory, V as an MN-major operand), the two tiles half a
//     block apart (PV(b,0) QK(b+1,0) PV(b,1) QK(b+1,1)) so the tensor core
//     works on one tile while the other tile's softmax runs;
//   - two softmax warpgroups, one per M-tile: thread r owns row r of its tile
//     (TMEM lane r): it loads S, masks the scores whose element bit is clear
//     (-inf; the row's 64 bits of the next block are loaded one block ahead),
//     keeps the online-softmax max / sum in registers, rescales O in tensor
//     memory only when the running max grows by more than 2^8 (otherwise the
//     stale max is kept: same softmax, exponentials bounded by 256), and
//     writes P = exp2(s - m) as a 16-bit high part plus a 16-bit remainder,
//     so that P.V carries P to ~fp32 accuracy.
// One CTA per SM (all 512 TMEM columns: S and O of both tiles).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace sfa {
namespace {

constexpr int kTileM = 128;
constexpr int kKeys = 64;           // keys per K/V block (N of Q.K^T, K of P.V)
constexpr int kStages = 3;
constexpr int kSoftWarps = 8;
constexpr int kThreads = kSoftWarps * 32 + 32;
constexpr int kTmemCols = 512;
constexpr int kTileCols = 256;      // TMEM columns per M-tile: S [0, 64), O [64, 64 + D)
constexpr int kOCol = 64;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct TcSmem {
    static constexpr int panels = D / 64;
    static constexpr int qTile = kTileM * D * 2;          // panels x 128 rows x 128 B
    static constexpr int kvTile = kKeys * D * 2;          // panels x 64 rows x 128 B
    static constexpr int pTile = kTileM * kKeys * 2;      // 128 rows x 128 B
    static constexpr int q = 0;
    static constexpr int kv = q + 2 * qTile;              // [stage][K, V]
    static constexpr int p = kv + kStages * 2 * kvTile;   // [tile][hi, lo]
    static constexpr int bars = p + 4 * pTile;
    static constexpr int tmem_slot = bars + 16 * 8;      // TMEM base address
    static constexpr int abort = tmem_slot + 4;          // a wait timed out
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;            // room to align the base to 1024
    static_assert(alloc <= 232448, "dynamic shared memory per block");
};

// barrier indices
enum {
    B_Q = 0,
    B_KV_FULL = 1,
    B_KV_FREE = B_KV_FULL + kStages,
    B_S_FULL = B_KV_FREE + kStages,
    B_P_FULL = B_S_FULL + 2,
    B_O_DONE = B_P_FULL + 2,
    B_DRAIN = B_O_DONE + 2,
    B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT <= 16, "barrier slots");

struct BsrTcItem {
    int rb, row0, kvh, pad;
};

struct BsrTcParams {
    void* out;
    float* lse;
    const int32_t* indptr;
    const int32_t* indices;
    const BsrTcItem* items;
    int* err_word;
    int M, N, R, C, Hq, G, TR;
    float scale_log2;
    const uint8_t* mask;    // per-element bits, most significant first
    float capl2, inv_capl2; // logits soft cap in log2 units (CAP instantiations)
    int kv_hnd;             // K / V maps over (Hkv, N, d)
};

// The 64-bit word whose bit j is element j of the 64 mask elements held,
// most significant bit first, by the 8 bytes `raw` was loaded from.
__device__ __forceinline__ uint64_t mask_bits64(uint64_t raw) {
    const uint64_t rev = __brevll(raw);     // bit j of byte t now at bit 8 (7 - t) + j
    const uint32_t lo = (uint32_t)rev, hi = (uint32_t)(rev >> 32);
    return ((uint64_t)__byte_perm(lo, 0, 0x0123) << 32) | __byte_perm(hi, 0, 0x0123);
}

template <class E, int D, bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
bsr_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const BsrTcParams p) {
    using T = typename E::T;
    using L = TcSmem<D>;
    constexpr bool kBf16 = std::is_same<E, BF16>::value;
    constexpr uint32_t kIdescQK = idesc_f16(kTileM, kKeys, kBf16, false, false);
    constexpr uint32_t kIdescPV = idesc_f16(kTileM, D, kBf16, false, true);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return sbase + L::bars + 8 * i; };

    const BsrTcItem item = p.items[blockIdx.x];
    const int blk0 = p.indptr[item.rb];
    const int sub = p.C / kKeys;
    const int nb = (p.indptr[item.rb + 1] - blk0) * sub;
    const int row_end = min((item.rb + 1) * p.R, p.M);

    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::abort);
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar(B_Q), 1);
        mbar_init(bar(B_DRAIN), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_FREE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_S_FULL + t), 1);
            mbar_init(bar(B_P_FULL + t), 128);
            mbar_init(bar(B_O_DONE + t), 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(sbase + L::tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::tmem_slot);

    if (warp == kSoftWarps) {
        // ============================ control ============================
        if (lane == 0 && nb > 0) {
            tma_prefetch_map(&mq);
            tma_prefetch_map(&mk);
            tma_prefetch_map(&mv);
            mbar_arrive_expect_tx(bar(B_Q), 2 * L::qTile);
            for (int t = 0; t < 2; ++t)
                for (int pn = 0; pn < L::panels; ++pn)
                    tma_load_3d(sbase + L::q + t * L::qTile + pn * (kTileM * 128), &mq, pn * 64,
                                item.kvh * p.G, item.row0 + t * p.TR, bar(B_Q));
            auto load_kv = [&](int b) {
                const int s = b % kStages;
                const int col = p.indices[blk0 + b / sub] * p.C + (b % sub) * kKeys;
                const uint32_t dst = sbase + L::kv + s * 2 * L::kvTile;
                mbar_arrive_expect_tx(bar(B_KV_FULL + s), 2 * L::kvTile);
                // NHD maps take (dim, kv head, key), HND maps (dim, key, kv head)
                const int y = p.kv_hnd ? col : item.kvh, z = p.kv_hnd ? item.kvh : col;
                for (int pn = 0; pn < L::panels; ++pn) {
                    tma_load_3d(dst + pn * (kKeys * 128), &mk, pn * 64, y, z, bar(B_KV_FULL + s));
                    tma_load_3d(dst + L::kvTile + pn * (kKeys * 128), &mv, pn * 64, y, z,
                                bar(B_KV_FULL + s));
                }
            };
            for (int b = 0; b < min(kStages, nb); ++b) load_kv(b);
            int loaded = min(kStages, nb) - 1, waited = -1;     // K/V blocks issued / landed
            // S_t = Q_t K_b^T
            auto qk = [&](int b, int t) {
                const uint32_t kbase = sbase + L::kv + (b % kStages) * 2 * L::kvTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    const uint64_t ad = sdesc_sw128(
                        sbase + L::q + t * L::qTile + (kk >> 2) * (kTileM * 128) + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * (kKeys * 128) + off, 16, 1024);
                    tc_mma_f16(tmem + t * kTileCols, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(B_S_FULL + t));
            };
            // O_t += P_t V_b (high part, then remainder)
            auto pv = [&](int b, int t) {
                const uint32_t vbase = sbase + L::kv + (b % kStages) * 2 * L::kvTile + L::kvTile;
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk) {
                        const uint64_t ad = sdesc_sw128(
                            sbase + L::p + (2 * t + part) * L::pTile + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(vbase + kk * 16 * 128, kKeys * 128, 1024);
                        const uint32_t acc = (b > 0 || part > 0 || kk > 0) ? 1u : 0u;
                        tc_mma_f16(tmem + t * kTileCols + kOCol, ad, bd, kIdescPV, acc);
                    }
                tc_commit(bar(B_O_DONE + t));
            };
            bool ok = mbar_wait(bar(B_Q), 0, p.err_word, abort_flag);
            // The two M-tiles run half a block apart: while the softmax of
            // one tile runs, the tensor core does the other tile's P.V and
            // its next Q.K^T.  Order: PV(b,0) QK(b+1,0) PV(b,1) QK(b+1,1).
            if (ok && nb > 0) {
                ok = mbar_wait(bar(B_KV_FULL), 0, p.err_word, abort_flag);
                if (ok) {
                    waited = 0;
                    tc_fence_after();
                    qk(0, 0);
                    qk(0, 1);
                }
            }
            for (int b = 0; b < nb && ok; ++b) {
                ok = mbar_wait(bar(B_P_FULL + 0), b & 1, p.err_word, abort_flag);
                if (!ok) break;
                tc_fence_after();
                pv(b, 0);
                // refill the stage that block b - 1 used (its last P.V ran on
                // the tensor core before Q.K^T of block b, which the softmax
                // of P(b,0) waited for, so this wait is short)
                const int nxt = b - 1 + kStages;
                if (b >= 1 && nxt < nb) {
                    ok = mbar_wait(bar(B_KV_FREE + (b - 1) % kStages), ((b - 1) / kStages) & 1,
                                   p.err_word, abort_flag);
                    if (!ok) break;
                    load_kv(nxt);
                    loaded = nxt;
                }
                if (b + 1 < nb) {
                    ok = mbar_wait(bar(B_KV_FULL + (b + 1) % kStages), ((b + 1) / kStages) & 1,
                                   p.err_word, abort_flag);
                    if (!ok) break;
                    waited = b + 1;
                    tc_fence_after();
                    qk(b + 1, 0);
                }
                ok = mbar_wait(bar(B_P_FULL + 1), b & 1, p.err_word, abort_flag);
                if (!ok) break;
                tc_fence_after();
                pv(b, 1);
                tc_commit(bar(B_KV_FREE + b % kStages));
                if (b + 1 < nb) qk(b + 1, 1);
            }
            if (!ok) {
                // a wait gave up (the abort flag is set): let every MMA and
                // copy this thread issued finish (bounded) before leaving
                tc_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0, nullptr, nullptr, 100000000ull);
                mbar_wait(bar(B_Q), 0, nullptr, nullptr, 100000000ull);
                for (int bb = waited + 1; bb <= loaded; ++bb)
                    mbar_wait(bar(B_KV_FULL + bb % kStages), (bb / kStages) & 1, nullptr, nullptr,
                              100000000ull);
            }
        }
    } else {
        // ============================ softmax ============================
        const int t = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;                       // row of the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16) + t * kTileCols;
        unsigned char* p_hi = smem + L::p + (2 * t) * L::pTile;
        unsigned char* p_lo = p_hi + L::pTile;
        float m_used = -INFINITY, l = 0.f;
        // per-element mask: this row's 64 bits of block b + 1 are loaded while
        // block b is processed (8 bytes per row and 64-key block)
        uint64_t mask_next = 0;
        auto mask_word = [&](int bb) -> uint64_t {
            const int i = item.row0 + t * p.TR + r / p.G;
            if (!(i < row_end && r / p.G < p.TR)) return 0;
            const int64_t e0 = ((int64_t)(blk0 + bb / sub) * p.R + (i - item.rb * p.R)) * p.C +
                               (bb % sub) * kKeys;
            return __ldg(reinterpret_cast<const unsigned long long*>(p.mask + (e0 >> 3)));
        };
        if (nb > 0) mask_next = mask_word(0);
        for (int b = 0; b < nb; ++b) {
            mbar_wait(bar(B_S_FULL + t), b & 1, p.err_word, abort_flag);
            tc_fence_after();
            uint32_t sv[64];
            tmem_ld32(lane_base, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(lane_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_wait_ld();
            // allowed keys of this 64-key block for this row (bit j = key j)
            uint64_t am = ~0ull;
            {
                const int i = item.row0 + t * p.TR + r / p.G;     // query row of this thread
                if (i < row_end && r / p.G < p.TR) am = mask_bits64(mask_next);
            }
            // masked keys: scores -inf before the max; without a soft cap
            // (which would map -inf to a finite value) that is the whole
            // mask, exp2(-inf - m) being 0
            if (am != ~0ull) {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (!((am >> j) & 1ull)) sv[j] = __float_as_uint(-INFINITY);
            }
            if (b + 1 < nb) mask_next = mask_word(b + 1);
            // block max in four independent chains, scaled once (the scale is
            // positive and rounding monotonic, so this equals the max of the
            // scaled scores)
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sv[j]));
            float bmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
            // the soft cap is increasing too: capped max = max of capped
            if constexpr (CAP)
                if (bmax != -INFINITY) bmax = soft_cap_log2(bmax, p.capl2, p.inv_capl2);
            const float m_new = fmaxf(m_used, bmax);
            const bool need = m_new > m_used + kRescaleThreshold;
            if (b > 0) {
                // P.V of block b - 1 must be done before P and O are touched
                mbar_wait(bar(B_O_DONE + t), (b - 1) & 1, p.err_word, abort_flag);
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
                    const float f = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(lane_base + kOCol + 32 * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                        tmem_st32(lane_base + kOCol + 32 * c, ov);
                    }
                    tmem_wait_st();
                    l *= f;
                }
            }
            if (need) m_used = m_new;
            // P = exp2(s - m): high and low 16-bit parts, swizzled rows (a row
            // that has seen no allowed key has m = -inf and only -inf scores:
            // subtracting 0 gives P = 0 instead of NaN)
            const float m_sub = (!CAP && m_used == -INFINITY) ? 0.f : m_used;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};     // row sum in four chains
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float u0 = __uint_as_float(sv[8 * c + 2 * e]) * p.scale_log2;
                    float u1 = __uint_as_float(sv[8 * c + 2 * e + 1]) * p.scale_log2;
                    if constexpr (CAP) {
                        u0 = soft_cap_log2(u0, p.capl2, p.inv_capl2);
                        u1 = soft_cap_log2(u1, p.capl2, p.inv_capl2);
                    }
                    float p0 = fast_exp2(u0 - m_sub);
                    float p1 = fast_exp2(u1 - m_sub);
                    if constexpr (CAP) {
                        // capped masked keys give 0, also while the row has
                        // seen none (m = -inf)
                        if (!((am >> (8 * c + 2 * e)) & 1ull)) p0 = 0.f;
                        if (!((am >> (8 * c + 2 * e + 1)) & 1ull)) p1 = 0.f;
                    }
                    ls[e] += p0 + p1;
                    hw[e] = E::pack2(p0, p1);
                    const float2 h = E::unpack2(hw[e]);
                    lw[e] = E::pack2(p0 - h.x, p1 - h.y);
                }
                const int pos = r * 128 + ((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(p_hi + pos) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(p_lo + pos) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + t));
        }
        // ---- epilogue: O / l for the rows of this tile ----
        const int i = item.row0 + t * p.TR + r / p.G;
        const int h = item.kvh * p.G + r % p.G;
        const bool valid_row = i < row_end && r / p.G < p.TR;
        if (nb > 0) {
            mbar_wait(bar(B_O_DONE + t), (nb - 1) & 1, p.err_word, abort_flag);
            tc_fence_after();
        }
        const bool empty = !(l > 0.f);
        const float inv = empty ? 0.f : 1.f / l;
        const int64_t orow_idx = (int64_t)i * p.Hq + h;
        T* orow = static_cast<T*>(p.out) + orow_idx * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            if (nb > 0) {
                tmem_ld32(lane_base + kOCol + 32 * c, ov);
                tmem_wait_ld();
            }
            if (valid_row) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 w;
                    w.x = empty ? 0u : E::pack2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
                    w.y = empty ? 0u : E::pack2(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
                    w.z = empty ? 0u : E::pack2(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv);
                    w.w = empty ? 0u : E::pack2(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + 32 * c + j) = w;
                }
            }
        }
        if (valid_row && p.lse)
            p.lse[orow_idx] = empty ? -INFINITY : (m_used + __log2f(l)) * kLn2;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// ---- host: tensor maps (shared with the 128-key kernel) ------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                            &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }
}  // namespace

// 3-D map over a [rows][heads][dim] tensor: box = 64 dims x hb heads x rb rows,
// 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, bool bf16, int dim, int heads, int rows,
              int hb, int rb) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)dim * heads * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)hb, (cuuint32_t)rb};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over a [heads][rows][dim] (HND) tensor: box = 64 dims x rb rows x
// hb heads, 128-byte swizzle.
bool make_map_hnd(CUtensorMap* map, const void* base, bool bf16, int dim, int rows, int heads,
                  int rb, int hb) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)dim * rows * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rb, (cuuint32_t)hb};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 8-bit elements: 3-D maps as above, box 128 elements (128 bytes) wide.
bool make_map8(CUtensorMap* map, const void* base, int dim, int heads, int rows, int hb, int rb) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim, (cuuint64_t)dim * heads};
    const cuuint32_t box[3] = {128, (cuuint32_t)hb, (cuuint32_t)rb};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gdim, gstride,
                    box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map8_hnd(CUtensorMap* map, const void* base, int dim, int rows, int heads, int rb,
                   int hb) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim, (cuuint64_t)dim * rows};
    const cuuint32_t box[3] = {128, (cuuint32_t)rb, (cuuint32_t)hb};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gdim, gstride,
                    box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over `rows` rows of `width` 16-bit elements, `row_stride`
// elements apart: box = box_w elements x 1 row, no swizzle (the row-gather
// form: each tile::gather4 copy moves four such boxes of four rows).
bool make_rows_map(CUtensorMap* map, const void* base, bool bf16, int width, int64_t rows,
                   int64_t row_stride, int box_w) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_w, 1};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

template <class E, int D, bool CAP>
cudaError_t launch_tc_t(const BsrParams& bp, const BsrTcParams& tp, int nitems, cudaStream_t stream) {
    using L = TcSmem<D>;
    const bool bf16 = std::is_same<E, BF16>::value;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, bp.q, bf16, D, bp.Hq, bp.M, tp.G, tp.TR))
        return cudaErrorInvalidValue;
    if (bp.kv_hnd ? (!make_map_hnd(&mk, bp.k, bf16, D, bp.N, bp.Hkv, kKeys, 1) ||
                     !make_map_hnd(&mv, bp.v, bf16, D, bp.N, bp.Hkv, kKeys, 1))
                  : (!make_map(&mk, bp.k, bf16, D, bp.Hkv, bp.N, 1, kKeys) ||
                     !make_map(&mv, bp.v, bf16, D, bp.Hkv, bp.N, 1, kKeys)))
        return cudaErrorInvalidValue;
    auto kern = bsr_tc_kernel<E, D, CAP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
    if (err != cudaSuccess) return err;
    kern<<<nitems, kThreads, L::alloc, stream>>>(mq, mk, mv, tp);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool bsr_tc_supported(int head_dim, int C, int Hq, int Hkv) {
    const int G = Hq / Hkv;
    return (head_dim == 64 || head_dim == 128) && C % kKeys == 0 && G >= 1 && G <= kTileM &&
           kTileM % G == 0;
}

int bsr_tc_rows_per_item(int Hq, int Hkv) { return 2 * (kTileM / (Hq / Hkv)); }

cudaError_t launch_bsr_tc(const BsrParams& bp, const void* items, int nitems, int* err_word,
                          sfa_dtype dtype, cudaStream_t stream) {
    if (nitems == 0) return cudaSuccess;
    if (bp.mask_mode != 2) return cudaErrorInvalidValue;   // the per-element mask mode only
    BsrTcParams tp{};
    tp.out = bp.out;
    tp.lse = bp.lse;
    tp.indptr = bp.indptr;
    tp.indices = bp.indices;
    tp.items = static_cast<const BsrTcItem*>(items);
    tp.err_word = err_word;
    tp.M = bp.M;
    tp.N = bp.N;
    tp.mask = bp.mask;
    tp.R = bp.R;
    tp.C = bp.C;
    tp.Hq = bp.Hq;
    tp.G = bp.Hq / bp.Hkv;
    tp.kv_hnd = bp.kv_hnd;
    tp.TR = kTileM / tp.G;
    tp.scale_log2 = bp.scale_log2;
    const bool cap = bp.softcap_log2 > 0.f;
    tp.capl2 = cap ? bp.softcap_log2 : 0.f;
    tp.inv_capl2 = cap ? 1.f / bp.softcap_log2 : 0.f;
    const bool bf16 = dtype == SFA_DTYPE_BF16;
#define SFA_BSR_TC_CAP(CAP_)                                                                     \
    if (cap == CAP_) {                                                                           \
        if (bp.d == 128)                                                                         \
            return bf16 ? launch_tc_t<BF16, 128, CAP_>(bp, tp, nitems, stream)                   \
                        : launch_tc_t<F16, 128, CAP_>(bp, tp, nitems, stream);                   \
        if (bp.d == 64)                                                                          \
            return bf16 ? launch_tc_t<BF16, 64, CAP_>(bp, tp, nitems, stream)                    \
                        : launch_tc_t<F16, 64, CAP_>(bp, tp, nitems, stream);                    \
    }
    SFA_BSR_TC_CAP(false)
    SFA_BSR_TC_CAP(true)
#undef SFA_BSR_TC_CAP
    return cudaErrorInvalidValue;
}

}  // namespace sfa
