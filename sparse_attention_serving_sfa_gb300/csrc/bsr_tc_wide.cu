// Block-sparse (BSR) attention on the tensor cores in steps of 128 keys.
//
// "flashinfer.sparse", BlockSparseAttentionWrapper: query row i attends to
// key column j iff block (i / R, j / C) is stored; qo head h reads kv head
// h / (Hq / Hkv).  Same work items, support (head_dim 64 or 128, C % 64 == 0,
// Hq / Hkv dividing 128) and warp roles as the 64-key kernel (bsr_tc.cu,
// which serves plan()'s per-element block mask), for plain blocks (mode 0),
// bottom-right causal (mode 1) and VariableBlockSparseAttentionWrapper's
// variable blocks over HND tensors (mode 3: per (kv head, row block) a list
// of 64-key windows, each four 16-key quarters at their own start keys and a
// 64-bit mask of allowed keys).  Each step takes two 64-key blocks (or windows), so the per-step
// round trip (Q.K^T -> softmax -> P.V and the barriers between them) is paid
// once per 128 keys:
//   - control warp (one thread): TMA loads of the two Q tiles and of two
//     64-key K / V blocks per step into a two-stage ring (a step with one
//     block left loads rows past the end, which TMA fills with zeros), and
//     the tcgen05.mma issue: S_t = Q_t K^T
//     (N = 128) into tensor memory, then O_t += P_t V with P read from tensor
//     memory (written over S) and V an MN-major shared-memory operand (in the
//     causal and variable modes in two halves: keys 64..127 of both tiles as
//     soon as the softmax has written them, then keys 0..63);
//   - two softmax warpgroups, thread r = row r of its tile (TMEM lane r):
//     the step's max over 128 scores, the conditional O rescale (only when the
//     running max grows by more than 2^8), and P = exp2(s - m) as a 16-bit
//     high part plus the 16-bit rounding of the remainder, stored over S,
//     keys 64..127 first (still in registers from the max pass).
// TMEM per tile: S / P in columns [0, 128), O in [128, 128 + D).
//
// FP8 instantiations (F8 = 1: E4M3, 2: E5M2; plan() q_data_type /
// kv_data_type, run() scale_q / scale_k / scale_v of "flashinfer.sparse"):
// q, k and v hold 8-bit codes, both contractions run as
// tcgen05.mma.kind::f8f6f4 (32 keys or dims per instruction), the
// dequantisation scales scale_q[h] * scale_k[g] multiply each row's scores and
// scale_v[g] its output.  P = exp2(s - m + 8) (kept below the format's largest
// value by rescaling O whenever the running max grows by more than 0.5) goes
// to the tensor core in V's format as a high part plus the rounding of the
// remainder, four keys per TMEM column; out is fp16 or bf16.
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace sfa {
namespace {

constexpr int kTileM = 128;
constexpr int kBlk = 64;            // keys per K/V block
constexpr int kStep = 2 * kBlk;     // keys per step
constexpr int kStages = 2;
constexpr int kSoftWarps = 8;
constexpr int kThreads = kSoftWarps * 32 + 32;
// The variable mode's block: two softmax warpgroups and a control warpgroup
// (one working warp) that gives registers back, so that a softmax thread
// holds a whole 128-key step of scores and reads them from tensor memory in
// one round trip: launched with kRegsLaunch registers a thread, then control
// kRegsControl, softmax kRegsSoftmax.  (Measured on the other modes it ran
// 3-8% slower than one 64-key half at a time with kThreads threads.)
constexpr int kThreadsSplit = kSoftWarps * 32 + 128;
constexpr int kRegsLaunch = 168, kRegsControl = 80, kRegsSoftmax = 208;
static_assert(kRegsSoftmax * kSoftWarps * 32 + kRegsControl * 128 <= kRegsLaunch * kThreadsSplit,
              "the register split fits what the block was launched with");
static_assert(2 * 32 * kRegsSoftmax + 32 * kRegsControl <= 16384,
              "the register split fits each SM sub-partition (two softmax warps and one control warp)");
constexpr int kTmemCols = 512;
constexpr int kTileCols = 256;      // TMEM columns per M-tile
constexpr int kOCol = 128;          // O after the 128 S / P columns
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D, int EB>                                  // EB: bytes per element
struct WideSmem {
    static constexpr int rowBytes = D * EB;
    static constexpr int panels = rowBytes / 128;
    static constexpr int qTile = kTileM * rowBytes;       // panels x 128 rows x 128 B
    static constexpr int kPanel = kStep * 128;            // 128 keys x 128 B
    static constexpr int kvHalf = kBlk * 128;             // one block's rows of a panel
    static constexpr int kvTile = panels * kPanel;        // K (or V) of one step
    static constexpr int q = 0;
    static constexpr int kv = q + 2 * qTile;              // [stage][K, V]
    static constexpr int bars = kv + kStages * 2 * kvTile;
    static constexpr int tmem_slot = bars + 16 * 8;
    static constexpr int abort = tmem_slot + 4;
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;            // room to align the base to 1024
    static_assert(alloc <= 232448, "dynamic shared memory per block");
};

// P_HALF(t): P of keys 64..127 of tile t written; P_FULL(t): all of P written
enum {
    B_Q = 0,
    B_KV_FULL = 1,
    B_KV_FREE = 3,
    B_S_FULL = 5,
    B_P_FULL = 7,
    B_O_DONE = 9,
    B_P_HALF = 11,
    B_DRAIN = 13
};

struct WideItem {
    int rb, row0, kvh, pad;
};

// Mode 3 key window: four 16-key quarters, keys [key[q], key[q] + 16) in
// rows 16 q .. 16 q + 15 of the 64-key block; bit j of the mask (hi:lo) =
// row j allowed.
struct alignas(8) WideWindow {
    int key[4];
    unsigned lo, hi;
};
constexpr int kQuarter = kBlk / 4;

struct WideParams {
    void* out;
    float* lse;
    const int32_t* indptr;
    const int32_t* indices;
    const WideItem* items;
    int* err_word;
    int M, N, R, C, Hq, G, TR;
    float scale_log2;
    int causal;             // mode 3: bottom-right causal on top of the windows
    float capl2, inv_capl2; // logits soft cap in log2 units (CAP instantiations)
    int kv_hnd;             // modes 0 / 1: K / V maps over (Hkv, N, d)
    // FP8 instantiations: per-head dequantisation scales (NULL = 1)
    const float* scale_q;   // [Hq]
    const float* scale_k;   // [Hkv]
    const float* scale_v;   // [Hkv]
};

// Keys j <= lim allowed among the 64 of a block (lim relative to its first key).
__device__ __forceinline__ uint64_t causal_bits64(int64_t lim) {
    return lim < 0 ? 0ull : (lim >= 63 ? ~0ull : ((2ull << lim) - 1ull));
}
// The same among the 16 keys of a quarter window.
__device__ __forceinline__ uint32_t causal_bits16(int64_t lim) {
    return lim < 0 ? 0u : (lim >= 15 ? 0xffffu : ((2u << lim) - 1u));
}

// Per mode (measured): the causal and variable modes hand P to the tensor
// core in two halves and skip a second M-tile that has no rows of the item
// (row blocks of any size); plain blocks do neither (both measured slower
// there: 647 -> 666 / 702 us).
template <int MODE>
struct WideSchedule {
    static constexpr bool split_p = MODE != 0;
    static constexpr bool tile_skip = MODE != 0;
    static constexpr bool split_regs = MODE == 3;
    static constexpr int threads = split_regs ? kThreadsSplit : kThreads;
};

template <class E, int D, int MODE, bool CAP, int F8>
__global__ void __launch_bounds__(WideSchedule<MODE>::threads, 1)
bsr_tc_wide_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const WideParams p) {
    // E: element type of q / k / v / out, or of out alone with F8
    constexpr int EB = F8 ? 1 : 2;
    static_assert(!F8 || D == 128, "8-bit rows of 128 bytes");
    using L = WideSmem<D, EB>;
    constexpr bool kBf16 = std::is_same<E, BF16>::value;
    constexpr bool kE5 = F8 == 2;
    constexpr uint32_t kIdescQK = F8 ? idesc_f8(kTileM, kStep, kE5, false, false)
                                     : idesc_f16(kTileM, kStep, kBf16, false, false);
    constexpr uint32_t kIdescPV = F8 ? idesc_f8(kTileM, D, kE5, false, true)
                                     : idesc_f16(kTileM, D, kBf16, false, true);
    constexpr int KK = 32 / EB;              // keys (or dims) per MMA instruction
    constexpr int KQ = kBlk / KK;            // instructions per 64-key half
    constexpr int PC = 16 * EB;              // P columns of one part (high or low) of a half
    constexpr int kCol0 = 128 / EB;          // TMA coordinate step between 128-byte panels
    // log2 of the factor P carries (8-bit P is kept in the format's normal range)
    constexpr float kPShift = F8 ? 8.f : 0.f;
    constexpr float kThresh = F8 ? 0.5f : kRescaleThreshold;
    auto mma_ss = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (F8) tc_mma_f8(d, a, b, id, acc);
        else tc_mma_f16(d, a, b, id, acc);
    };
    auto mma_ts = [](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (F8) tc_mma_f8_ts(d, a, b, id, acc);
        else tc_mma_f16_ts(d, a, b, id, acc);
    };

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return sbase + L::bars + 8 * i; };

    const WideItem item = p.items[blockIdx.x];
    const int blk0 = p.indptr[item.rb];
    const int sub = p.C / kBlk;
    const int nb = (p.indptr[item.rb + 1] - blk0) * sub;     // 64-key blocks
    const int ns = (nb + 1) / 2;                              // steps
    // mode 3: rb = key window list, pad = end of the row block
    const int row_end = MODE == 3 ? item.pad : min((item.rb + 1) * p.R, p.M);
    // M-tiles with rows of this item: the second only when the row block
    // extends past the first tile's TR rows
    const int ntl = (WideSchedule<MODE>::tile_skip && item.row0 + p.TR >= row_end) ? 1 : 2;
    const WideWindow* wins = reinterpret_cast<const WideWindow*>(p.indices);
    // first key of 64-key block b
    auto block_key0 = [&](int b) -> int {
        if constexpr (MODE == 3) return wins[blk0 + b].key[0];
        return p.indices[blk0 + b / sub] * p.C + (b % sub) * kBlk;
    };

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
            mbar_init(bar(B_P_HALF + t), 128);
            mbar_init(bar(B_O_DONE + t), 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(sbase + L::tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::tmem_slot);

    constexpr bool kSplitRegs = WideSchedule<MODE>::split_regs;
    if (warp >= kSoftWarps) {
        if constexpr (kSplitRegs) regs_release<kRegsControl>();
        // ============================ control ============================
        if (warp == kSoftWarps && lane == 0 && ns > 0) {
            tma_prefetch_map(&mq);
            tma_prefetch_map(&mk);
            tma_prefetch_map(&mv);
            mbar_arrive_expect_tx(bar(B_Q), ntl * L::qTile);
            for (int t = 0; t < ntl; ++t)
                for (int pn = 0; pn < L::panels; ++pn) {
                    if constexpr (MODE == 3)
                        tma_load_3d(sbase + L::q + t * L::qTile + pn * (kTileM * 128), &mq,
                                    pn * kCol0, item.row0 + t * p.TR, item.kvh * p.G, bar(B_Q));
                    else
                        tma_load_3d(sbase + L::q + t * L::qTile + pn * (kTileM * 128), &mq,
                                    pn * kCol0, item.kvh * p.G, item.row0 + t * p.TR, bar(B_Q));
                }
            // step st: blocks 2 st and 2 st + 1; a missing second block reads
            // rows N.. (all outside the tensor: zeros, full byte count)
            auto load_step = [&](int st) {
                const int s = st % kStages;
                const uint32_t dst = sbase + L::kv + s * 2 * L::kvTile;
                mbar_arrive_expect_tx(bar(B_KV_FULL + s), 2 * L::kvTile);
                for (int h = 0; h < 2; ++h) {
                    const int b = 2 * st + h;
                    if constexpr (MODE == 3) {
                        // a window's four 16-key quarters, 16-row boxes at
                        // rows key[q] .. key[q] + 15 (a missing window: rows
                        // past the end, zeros)
                        const WideWindow w =
                            b < nb ? wins[blk0 + b] : WideWindow{{p.N, p.N, p.N, p.N}, 0u, 0u};
                        for (int pn = 0; pn < L::panels; ++pn) {
                            const uint32_t kd = dst + pn * L::kPanel + h * L::kvHalf;
                            const uint32_t vd = kd + L::kvTile;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                tma_load_3d(kd + q * kQuarter * 128, &mk, pn * kCol0, w.key[q], item.kvh,
                                            bar(B_KV_FULL + s));
                                tma_load_3d(vd + q * kQuarter * 128, &mv, pn * kCol0, w.key[q], item.kvh,
                                            bar(B_KV_FULL + s));
                            }
                        }
                        continue;
                    }
                    const int col = b < nb ? block_key0(b) : p.N;
                    for (int pn = 0; pn < L::panels; ++pn) {
                        const uint32_t kd = dst + pn * L::kPanel + h * L::kvHalf;
                        const uint32_t vd = kd + L::kvTile;
                        if (MODE == 3 || p.kv_hnd) {
                            tma_load_3d(kd, &mk, pn * kCol0, col, item.kvh, bar(B_KV_FULL + s));
                            tma_load_3d(vd, &mv, pn * kCol0, col, item.kvh, bar(B_KV_FULL + s));
                        } else {
                            tma_load_3d(kd, &mk, pn * kCol0, item.kvh, col, bar(B_KV_FULL + s));
                            tma_load_3d(vd, &mv, pn * kCol0, item.kvh, col, bar(B_KV_FULL + s));
                        }
                    }
                }
            };
            for (int st = 0; st < min(kStages, ns); ++st) load_step(st);
            int loaded = min(kStages, ns) - 1, waited = -1;     // steps issued / landed
            bool ok = mbar_wait(bar(B_Q), 0, p.err_word, abort_flag);
            for (int st = 0; st < ns && ok; ++st) {
                const int s = st % kStages;
                ok = mbar_wait(bar(B_KV_FULL + s), (st / kStages) & 1, p.err_word, abort_flag);
                if (!ok) break;
                waited = st;
                tc_fence_after();
                const uint32_t kbase = sbase + L::kv + s * 2 * L::kvTile;
                // S_t = Q_t K^T, 128 keys
                for (int t = 0; t < ntl; ++t) {
                    // K steps of 32 bytes: 16 dims (16-bit) or 32 dims (8-bit)
#pragma unroll
                    for (int kk = 0; kk < L::rowBytes / 32; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t ad = sdesc_sw128(
                            sbase + L::q + t * L::qTile + (kk >> 2) * (kTileM * 128) + off, 16, 1024);
                        const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * L::kPanel + off, 16, 1024);
                        mma_ss(tmem + t * kTileCols, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(B_S_FULL + t));
                }
                // refill the stage that step st - 1 used with step st + 1
                if (st >= 1 && st + 1 < ns) {
                    ok = mbar_wait(bar(B_KV_FREE + (st - 1) % kStages), ((st - 1) / kStages) & 1,
                                   p.err_word, abort_flag);
                    if (!ok) break;
                    load_step(st + 1);
                    loaded = st + 1;
                }
                // O_t += P_t V over keys 64 h .. 64 h + 63: P from TMEM (KK keys
                // = 8 columns per MMA; high parts at 64 h, remainders at 64 h + PC).
                // The softmax writes keys 64..127 first, so their P.V runs while
                // it works on keys 0..63; a step with one block has no P.V for
                // the second half.
                const bool two = 2 * st + 1 < nb;
                auto pv_half = [&](int t, int h, bool first) {
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kq = 0; kq < KQ; ++kq) {
                            const uint32_t a = tmem + t * kTileCols + 64 * h + PC * part + 8 * kq;
                            const uint64_t bd = sdesc_sw128(
                                kbase + L::kvTile + (64 * h + KK * kq) * 128, L::kPanel, 1024);
                            const uint32_t acc = (first && part == 0 && kq == 0) ? 0u : 1u;
                            mma_ts(tmem + t * kTileCols + kOCol, a, bd, kIdescPV, acc);
                        }
                };
                if constexpr (WideSchedule<MODE>::split_p) {
                    for (int t = 0; t < ntl && ok; ++t) {
                        ok = mbar_wait(bar(B_P_HALF + t), st & 1, p.err_word, abort_flag);
                        if (!ok) break;
                        if (two) {
                            tc_fence_after();
                            pv_half(t, 1, st == 0);
                        }
                    }
                    for (int t = 0; t < ntl && ok; ++t) {
                        ok = mbar_wait(bar(B_P_FULL + t), st & 1, p.err_word, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        pv_half(t, 0, st == 0 && !two);
                        if (st == ns - 1) tc_commit(bar(B_O_DONE + t));
                    }
                } else {
                    // whole P at once; a one-block step's second half is
                    // P = 0 against V rows of zeros
                    for (int t = 0; t < ntl && ok; ++t) {
                        ok = mbar_wait(bar(B_P_FULL + t), st & 1, p.err_word, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int kk = 0; kk < kStep / KK; ++kk) {
                                const uint32_t a = tmem + t * kTileCols + 64 * (kk / KQ) + PC * part +
                                                   8 * (kk % KQ);
                                const uint64_t bd =
                                    sdesc_sw128(kbase + L::kvTile + kk * KK * 128, L::kPanel, 1024);
                                const uint32_t acc = (st > 0 || part > 0 || kk > 0) ? 1u : 0u;
                                mma_ts(tmem + t * kTileCols + kOCol, a, bd, kIdescPV, acc);
                            }
                        if (st == ns - 1) tc_commit(bar(B_O_DONE + t));
                    }
                }
                if (!ok) break;
                tc_commit(bar(B_KV_FREE + s));
            }
            if (!ok) {
                // a wait gave up (the abort flag is set): let every MMA and
                // copy this thread issued finish (bounded) before leaving
                tc_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0, nullptr, nullptr, 100000000ull);
                mbar_wait(bar(B_Q), 0, nullptr, nullptr, 100000000ull);
                for (int x = waited + 1; x <= loaded; ++x)
                    mbar_wait(bar(B_KV_FULL + x % kStages), (x / kStages) & 1, nullptr, nullptr,
                              100000000ull);
            }
        }
    } else {
        if constexpr (kSplitRegs) regs_acquire<kRegsSoftmax>();
        // ============================ softmax ============================
        const int t = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;                       // row of the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16) + t * kTileCols;
        float m_used = -INFINITY, l = 0.f;
        // a step's 128 scores (keys 0..63 then 64..127), or one 64-key half at a time
        uint32_t sv[kSplitRegs ? 128 : 64];
        // query row / qo head of this thread's tile row
        // (recomputed where used, so the plain mode keeps no registers for them)
        auto my_i = [&]() {
            return MODE == 3 ? item.row0 + t * p.TR + r % p.TR : item.row0 + t * p.TR + r / p.G;
        };
        auto my_h = [&]() { return MODE == 3 ? item.kvh * p.G + r / p.TR : item.kvh * p.G + r % p.G; };
        auto my_valid = [&]() { return my_i() < row_end && r / p.G < p.TR; };
        // multiplier of this row's raw scores (log2 units): the softmax scale,
        // times the row's dequantisation scales in the FP8 instantiations
        float rs = p.scale_log2;
        if constexpr (F8 != 0) {
            if (p.scale_q) rs *= p.scale_q[my_h()];
            if (p.scale_k) rs *= p.scale_k[item.kvh];
        }
        // allowed keys of block b for this row (bit j = key j of the block)
        auto allowed = [&](int b) -> uint64_t {
            if constexpr (MODE == 1) {
                return causal_bits64((int64_t)my_i() + (p.N - p.M) - block_key0(b));
            } else if constexpr (MODE == 3) {
                const WideWindow w = wins[blk0 + b];
                uint64_t m = ((uint64_t)w.hi << 32) | w.lo;
                if (p.causal) {
                    const int64_t lim = (int64_t)my_i() + (p.N - p.M);
                    uint64_t c = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) c |= (uint64_t)causal_bits16(lim - w.key[q]) << (16 * q);
                    m &= c;
                }
                return m;
            }
            return ~0ull;
        };
        // the two halves' masks of the next step are loaded during this one
        uint64_t am_next[2] = {~0ull, ~0ull};
        if constexpr (MODE != 0) {
            if (nb > 0) am_next[0] = allowed(0);
            if (nb > 1) am_next[1] = allowed(1);
        }
        // Masked keys: their scores set to -inf before the max.  Without a
        // soft cap or FP8 scales (the multiplier of the scores is then the
        // positive softmax scale) that is the whole mask: exp2(-inf - m) = 0.
        // The cap would map -inf to a finite value, and an FP8 scale may be
        // 0, so those instantiations also zero P key by key.
        constexpr bool kMaskOnce = MODE != 0 && !CAP && F8 == 0;
        auto apply_mask = [&](int h, uint64_t am) {
            if (am == ~0ull) return;                     // a fully allowed block
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (!((am >> j) & 1ull)) sv[(kSplitRegs ? 64 * h : 0) + j] = __float_as_uint(-INFINITY);
        };
        // P of one 64-key half from the scores in sv, written over that
        // half's S columns; returns the half's sum of P
        auto make_p = [&](int h, uint64_t am) -> float {
            uint32_t (&w)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sv[kSplitRegs ? 64 * h : 0]);
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (F8 != 0) {
                // keys 4k .. 4k + 3 -> high parts in w[2k], remainders in
                // w[2k + 1] (entries already read), four 8-bit P per word
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float pv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float u = __uint_as_float(w[4 * k + j]) * rs;
                        if constexpr (CAP) u = soft_cap_log2(u, p.capl2, p.inv_capl2);
                        float pp = fast_exp2(u - m_used + kPShift);
                        if constexpr (MODE != 0)
                            if (!((am >> (4 * k + j)) & 1ull)) pp = 0.f;
                        pv[j] = pp;
                    }
                    ls[k & 3] += (pv[0] + pv[1]) + (pv[2] + pv[3]);
                    const uint32_t h01 = f8_pack2<kE5>(pv[0], pv[1]);
                    const uint32_t h23 = f8_pack2<kE5>(pv[2], pv[3]);
                    const float2 b01 = f8_unpack2<kE5>(h01), b23 = f8_unpack2<kE5>(h23);
                    const uint32_t l01 = f8_pack2<kE5>(pv[0] - b01.x, pv[1] - b01.y);
                    const uint32_t l23 = f8_pack2<kE5>(pv[2] - b23.x, pv[3] - b23.y);
                    w[2 * k] = h01 | (h23 << 16);
                    w[2 * k + 1] = l01 | (l23 << 16);
                }
                tmem_st16_strided<0>(lane_base + 64 * h, w);
                tmem_st16_strided<1>(lane_base + 64 * h + 16, w);
            } else {
            // (a row that has seen no allowed key has m = -inf and only -inf
            // scores: subtracting 0 gives P = 0 instead of NaN)
            const float m_sub = (kMaskOnce && m_used == -INFINITY) ? 0.f : m_used;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                float u0 = __uint_as_float(w[2 * k]) * rs;
                float u1 = __uint_as_float(w[2 * k + 1]) * rs;
                if constexpr (CAP) {
                    u0 = soft_cap_log2(u0, p.capl2, p.inv_capl2);
                    u1 = soft_cap_log2(u1, p.capl2, p.inv_capl2);
                }
                float p0 = fast_exp2(u0 - m_sub);
                float p1 = fast_exp2(u1 - m_sub);
                if constexpr (MODE != 0 && !kMaskOnce) {
                    // masked keys give 0, also while the row has seen none (m = -inf)
                    if (!((am >> (2 * k)) & 1ull)) p0 = 0.f;
                    if (!((am >> (2 * k + 1)) & 1ull)) p1 = 0.f;
                }
                ls[k & 3] += p0 + p1;
                const uint32_t hw = E::pack2(p0, p1);
                const float2 hf = E::unpack2(hw);
                w[2 * k] = hw;
                w[2 * k + 1] = E::pack2(p0 - hf.x, p1 - hf.y);
            }
            tmem_st32_strided<0>(lane_base + 64 * h, w);
            tmem_st32_strided<1>(lane_base + 64 * h + 32, w);
            }
            return (ls[0] + ls[1]) + (ls[2] + ls[3]);
        };
        // a second tile without rows of this item has no work
        const int ns_t = t < ntl ? ns : 0;
        for (int st = 0; st < ns_t; ++st) {
            mbar_wait(bar(B_S_FULL + t), st & 1, p.err_word, abort_flag);
            tc_fence_after();
            const bool two = 2 * st + 1 < nb;
            const uint64_t am0 = am_next[0], am1 = am_next[1];
            if constexpr (MODE != 0) {
                if (2 * st + 2 < nb) am_next[0] = allowed(2 * st + 2);
                if (2 * st + 3 < nb) am_next[1] = allowed(2 * st + 3);
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if constexpr (kSplitRegs) {
                // the step's scores in one round trip (one block: its 64 only)
                if (two) {
                    tmem_ld128_sync(lane_base, *reinterpret_cast<uint32_t(*)[128]>(&sv[0]));
                } else {
                    tmem_ld64_sync(lane_base, *reinterpret_cast<uint32_t(*)[64]>(&sv[0]));
                }
                if constexpr (MODE != 0) apply_mask(0, am0);
#pragma unroll
                for (int j = 0; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sv[j]));
                if (two) {
                    if constexpr (MODE != 0) apply_mask(1, am1);
#pragma unroll
                    for (int j = 64; j < 64 * (kSplitRegs ? 2 : 1); ++j)
                        mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sv[j]));
                }
            } else {
                // keys 0..63, then 64..127 (kept in sv for their P)
                tmem_ld32(lane_base, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                tmem_ld32(lane_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                tmem_wait_ld();
                if constexpr (MODE != 0) apply_mask(0, am0);
#pragma unroll
                for (int j = 0; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sv[j]));
                if (two) {
                    tmem_ld32(lane_base + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(lane_base + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_wait_ld();
                    if constexpr (MODE != 0) apply_mask(1, am1);
#pragma unroll
                    for (int j = 0; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sv[j]));
                }
            }
            // the scale is positive and rounding monotonic: max of scaled = scaled max
            float bmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * rs;
            // the soft cap is increasing too: capped max = max of capped
            if constexpr (CAP)
                if (bmax != -INFINITY) bmax = soft_cap_log2(bmax, p.capl2, p.inv_capl2);
            const float m_new = fmaxf(m_used, bmax);
            const bool need = m_new > m_used + kThresh;
            // P.V of step st - 1 ran on the tensor core before this step's
            // Q.K^T, whose completion this thread waited for: O is settled
            if (st > 0 && __any_sync(0xffffffffu, need)) {
                const float f = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll (kSplitRegs ? 1 : D / 32)
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    if constexpr (kSplitRegs) {
                        tmem_ld32_sync(lane_base + kOCol + 32 * c, ov);
                    } else {
                        tmem_ld32(lane_base + kOCol + 32 * c, ov);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                    tmem_st32(lane_base + kOCol + 32 * c, ov);
                }
                l *= f;
            }
            if (need) m_used = m_new;
            if (two) {
                l += make_p(1, am1);               // keys 64..127
                if constexpr (WideSchedule<MODE>::split_p) {
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar(B_P_HALF + t));
                }
                // keys 0..63: still in sv, or read again (and masked again)
                if constexpr (!kSplitRegs) {
                    tmem_ld32(lane_base, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(lane_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_wait_ld();
                    if constexpr (kMaskOnce) apply_mask(0, am0);
                }
                l += make_p(0, am0);
            } else if constexpr (WideSchedule<MODE>::split_p) {
                // one block: no P.V for the second half (its barrier still
                // completes once per step)
                mbar_arrive(bar(B_P_HALF + t));
                l += make_p(0, am0);               // keys 0..63 are in sv
            } else {
                l += make_p(0, am0);               // keys 0..63 are in sv
                // the second block is zeros (V rows of zeros): P = 0 there
                uint32_t z[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) z[j] = 0u;
                tmem_st32(lane_base + 64, z);
                tmem_st32(lane_base + 96, z);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + t));
        }
        // ---- epilogue: O / l for the rows of this tile ----
        const int i = my_i(), h = my_h();
        const bool valid_row = my_valid();
        if (ns_t > 0) {
            mbar_wait(bar(B_O_DONE + t), 0, p.err_word, abort_flag);
            tc_fence_after();
        }
        const bool empty = !(l > 0.f);
        float vscale = 1.f;
        if constexpr (F8 != 0)
            if (p.scale_v) vscale = p.scale_v[item.kvh];
        const float inv = empty ? 0.f : vscale / l;
        using T = typename E::T;
        const int64_t orow_idx = MODE == 3 ? (int64_t)h * p.M + i : (int64_t)i * p.Hq + h;
        T* orow = static_cast<T*>(p.out) + orow_idx * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            if (ns_t > 0) {
                if constexpr (kSplitRegs) {
                    tmem_ld32_sync(lane_base + kOCol + 32 * c, ov);
                } else {
                    tmem_ld32(lane_base + kOCol + 32 * c, ov);
                    tmem_wait_ld();
                }
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
            p.lse[orow_idx] = empty ? -INFINITY : (m_used + __log2f(l) - kPShift) * kLn2;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <class E, int D, int MODE, bool CAP, int F8>
cudaError_t launch_wide_t(const BsrParams& bp, const WideParams& wp, int nitems, cudaStream_t stream) {
    using L = WideSmem<D, F8 ? 1 : 2>;
    const bool bf16 = std::is_same<E, BF16>::value;
    CUtensorMap mq, mk, mv;
    if (F8 != 0) {
        // 8-bit rows of 128 bytes: q NHD, k / v NHD or HND
        if (MODE == 3 || !make_map8(&mq, bp.q, D, bp.Hq, bp.M, wp.G, wp.TR))
            return cudaErrorInvalidValue;
        if (bp.kv_hnd ? (!make_map8_hnd(&mk, bp.k, D, bp.N, bp.Hkv, kBlk, 1) ||
                         !make_map8_hnd(&mv, bp.v, D, bp.N, bp.Hkv, kBlk, 1))
                      : (!make_map8(&mk, bp.k, D, bp.Hkv, bp.N, 1, kBlk) ||
                         !make_map8(&mv, bp.v, D, bp.Hkv, bp.N, 1, kBlk)))
            return cudaErrorInvalidValue;
    } else if (MODE == 3) {
        // key windows come as four quarters of kQuarter rows each
        if (!make_map_hnd(&mq, bp.q, bf16, D, bp.M, bp.Hq, wp.TR, wp.G) ||
            !make_map_hnd(&mk, bp.k, bf16, D, bp.N, bp.Hkv, kQuarter, 1) ||
            !make_map_hnd(&mv, bp.v, bf16, D, bp.N, bp.Hkv, kQuarter, 1))
            return cudaErrorInvalidValue;
    } else if (!make_map(&mq, bp.q, bf16, D, bp.Hq, bp.M, wp.G, wp.TR)) {
        return cudaErrorInvalidValue;
    } else if (bp.kv_hnd ? (!make_map_hnd(&mk, bp.k, bf16, D, bp.N, bp.Hkv, kBlk, 1) ||
                            !make_map_hnd(&mv, bp.v, bf16, D, bp.N, bp.Hkv, kBlk, 1))
                         : (!make_map(&mk, bp.k, bf16, D, bp.Hkv, bp.N, 1, kBlk) ||
                            !make_map(&mv, bp.v, bf16, D, bp.Hkv, bp.N, 1, kBlk))) {
        return cudaErrorInvalidValue;
    }
    auto kern = bsr_tc_wide_kernel<E, D, MODE, CAP, F8>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
    if (err != cudaSuccess) return err;
    if constexpr (WideSchedule<MODE>::split_regs) {
        // the register split assumes the block is launched with kRegsLaunch
        // registers a thread: with fewer, the softmax warps' request could
        // not be met (checked once per instantiation)
        static int regs_ok = -1;
        if (regs_ok < 0) {
            cudaFuncAttributes fa;
            err = cudaFuncGetAttributes(&fa, kern);
            if (err != cudaSuccess) return err;
            regs_ok = fa.numRegs == kRegsLaunch ? 1 : 0;
        }
        if (!regs_ok) return cudaErrorInvalidConfiguration;
    }
    kern<<<nitems, WideSchedule<MODE>::threads, L::alloc, stream>>>(mq, mk, mv, wp);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsr_tc_wide(const BsrParams& bp, const void* items, int nitems, int* err_word,
                               sfa_dtype dtype, cudaStream_t stream) {
    if (nitems == 0) return cudaSuccess;
    WideParams wp{};
    wp.out = bp.out;
    wp.lse = bp.lse;
    wp.indptr = bp.indptr;
    wp.indices = bp.indices;
    wp.items = static_cast<const WideItem*>(items);
    wp.err_word = err_word;
    wp.M = bp.M;
    wp.N = bp.N;
    wp.R = bp.R;
    wp.C = bp.mask_mode == 3 ? kBlk : bp.C;
    wp.causal = bp.causal;
    wp.kv_hnd = bp.mask_mode == 3 ? 1 : bp.kv_hnd;
    wp.scale_q = bp.scale_q;
    wp.scale_k = bp.scale_k;
    wp.scale_v = bp.scale_v;
    wp.Hq = bp.Hq;
    wp.G = bp.Hq / bp.Hkv;
    wp.TR = kTileM / wp.G;
    wp.scale_log2 = bp.scale_log2;
    const bool cap = bp.softcap_log2 > 0.f;
    wp.capl2 = cap ? bp.softcap_log2 : 0.f;
    wp.inv_capl2 = cap ? 1.f / bp.softcap_log2 : 0.f;
    const bool bf16 = dtype == SFA_DTYPE_BF16;
    if (bp.f8) {
        // FP8 q / k / v (head_dim 128, plain or causal blocks, no soft cap);
        // `dtype` is the output's
        if (bp.d != 128 || cap || (bp.mask_mode != 0 && bp.mask_mode != 1))
            return cudaErrorInvalidValue;
#define SFA_BSR_WIDE_F8(MODE_, F8_)                                                              \
    if (bp.mask_mode == MODE_ && bp.f8 == F8_)                                                   \
        return bf16 ? launch_wide_t<BF16, 128, MODE_, false, F8_>(bp, wp, nitems, stream)       \
                    : launch_wide_t<F16, 128, MODE_, false, F8_>(bp, wp, nitems, stream);
        SFA_BSR_WIDE_F8(0, 1)
        SFA_BSR_WIDE_F8(0, 2)
        SFA_BSR_WIDE_F8(1, 1)
        SFA_BSR_WIDE_F8(1, 2)
#undef SFA_BSR_WIDE_F8
        return cudaErrorInvalidValue;
    }
#define SFA_BSR_WIDE_MODE_CAP(MODE_, CAP_)                                                       \
    if (bp.mask_mode == MODE_ && cap == CAP_) {                                                  \
        if (bp.d == 128)                                                                         \
            return bf16 ? launch_wide_t<BF16, 128, MODE_, CAP_, 0>(bp, wp, nitems, stream)          \
                        : launch_wide_t<F16, 128, MODE_, CAP_, 0>(bp, wp, nitems, stream);          \
        if (bp.d == 64)                                                                          \
            return bf16 ? launch_wide_t<BF16, 64, MODE_, CAP_, 0>(bp, wp, nitems, stream)           \
                        : launch_wide_t<F16, 64, MODE_, CAP_, 0>(bp, wp, nitems, stream);           \
    }
#define SFA_BSR_WIDE_MODE(MODE_) SFA_BSR_WIDE_MODE_CAP(MODE_, false) SFA_BSR_WIDE_MODE_CAP(MODE_, true)
    SFA_BSR_WIDE_MODE(0)
    SFA_BSR_WIDE_MODE(1)
    SFA_BSR_WIDE_MODE(3)
#undef SFA_BSR_WIDE_MODE
#undef SFA_BSR_WIDE_MODE_CAP
    return cudaErrorInvalidValue;
}

}  // namespace sfa
