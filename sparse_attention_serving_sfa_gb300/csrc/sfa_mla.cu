// Top-K sparse attention for the MLA latent cache (128 query heads share one
// index list, Dk = 576 = 512 "nope" + 64 "rope" dims, Dv = 512, V = K[..., :512])
// on the 5th-generation tensor cores.
//
// "SparseFlashAttention 算子 API 描述", §1 (MLA: value is the first Dv dims of
// key), §2 具体子步骤 (gather, scaled dot product, causal mask, softmax over the
// selected slots, weighted sum), evaluated as an online softmax over 64-slot
// chunks.
//
// O for 128 heads x 512 dims (fp32) fills all 512 columns of one SM's tensor
// memory, so a unit (one index list and its 128 heads) is computed by a 2-CTA
// cluster that splits the head dimensions:
//   CTA r owns K/Q dims [256 r, 256 r + 256) (nope) and [512 + 32 r, 544 + 32 r)
//   (rope), and V / O dims [256 r, 256 r + 256) -- the first 256 of its K dims.
// Per 64-slot chunk, each CTA gathers only its 576 bytes of every selected K
// row (no duplicated gather) and computes a partial S_r = Q_r K_r^T; the two
// partials are exchanged with one bulk shared-memory copy into the peer CTA,
// so both CTAs hold the same S = S_0 + S_1, run the same online softmax and
// compute O_r += P V_r for their half of Dv (P as a 16-bit high part plus
// remainder, ~fp32 accurate).
//
// Tensor memory holds O, three S/P buffers (a chunk's scores, then its
// probabilities written over them as the A operand of P.V) and half of the
// unit's Q nope dims (the other half and the rope dims are read from shared
// memory; an MMA's A operand costs the same from either).  With three buffers
// QK runs up to two chunks ahead of P.V, so a chunk's scores are ready when
// the softmax wants to send them, and P(i + 1) can be written while P.V(i)
// runs.
//
// TMEM (512 columns): Q nope dims [0, 128) in [0, 64) | S/P buffers
// [64, 128), [128, 192), [192, 256) | O [256, 512).
//
// Roles per CTA (13 warps): 8 softmax warps (two warpgroups, thread = head =
// TMEM lane; warpgroup w takes slots [32 w, 32 w + 32) of a chunk and O dims
// [128 w, 128 w + 128) of the CTA's half), 1 MMA warp (Q TMA, tcgen05.mma
// issue from an event loop), 4 producer warps (cp.async gather, index
// prefetch, L2 prefetch of later chunks, visibility masks).  The softmax sends
// chunk i + 1's partial scores before computing chunk i's probabilities when
// they are ready, so the copy overlaps that work.  Work is stream-K over
// (unit, chunk) pairs per cluster; the parts of a unit split over clusters are
// written as fp32 partials and merged by a second kernel.
#include <cudaTypedefs.h>

#include <limits.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace sfa {
namespace {

constexpr int kChunk = 64;
constexpr int kHeads = 128;               // the MMA M dimension
constexpr int kDk = 576, kDv = 512;
constexpr int kHalfDv = 256;              // nope dims (and V / O dims) per CTA
constexpr int kStages = 3;
constexpr int kBufs = 3;                  // S/P buffers in tensor memory: QK runs up to 2 chunks ahead
constexpr int kSoftThreads = 256;
constexpr int kMmaWarp = 8;
constexpr int kProdWarp0 = 9;
constexpr int kProdThreads = 128;
constexpr int kThreads = kSoftThreads + 32 + kProdThreads;
constexpr int kTmemCols = 512;
constexpr int kQnCol = 0, kSCol = 64, kOCol = 256;   // Q nope dims [0, 128) | 3 S/P buffers | O
constexpr int kLookahead = 6;
constexpr int kPrefetch = 3;              // chunks ahead that the producers pull into L2
constexpr int kNoSlot = INT_MIN;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSeg = 8;                // clusters sharing one unit
constexpr uint32_t kXBytes = kHeads * kChunk * 4;

struct MlaSmem {
    static constexpr int nopePanel = kChunk * 128;          // 64 rows x 128 B (64 dims), 128B swizzle
    static constexpr int ropePanel = kChunk * 64;           // 64 rows x 64 B (32 dims), 64B swizzle
    static constexpr int kvStage = 4 * nopePanel + ropePanel;   // 36 KB
    static constexpr int kv = 0;
    static constexpr int stg = kv + kStages * kvStage;      // own partial S (send), 32 KB
    static constexpr int x = stg + kXBytes;                 // peer partial S (receive), 32 KB
    static constexpr int qn = x + kXBytes;                  // Q nope dims [128, 256): 2 panels x 128 rows x 128 B
    static constexpr int qr = qn + 2 * kHeads * 128;        // Q rope: 128 rows x 64 B, 64B swizzle
    static constexpr int red = qr + kHeads * 64;            // [2][128] row max per warpgroup
    static constexpr int red2 = red + 2 * kHeads * 4;       // [2][128] row sum per warpgroup
    static constexpr int bars = red2 + 2 * kHeads * 4;
    static constexpr int meta = bars + 24 * 8;              // [stage][4] uint16 visibility masks
    static constexpr int misc = meta + kStages * 8;         // tmem base, abort flag, early-send flag
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;
};
static_assert(MlaSmem::kvStage % 1024 == 0 && MlaSmem::qn % 1024 == 0 && MlaSmem::qr % 1024 == 0,
              "swizzle atoms must stay aligned");

enum {
    B_QR_FULL = 0, B_Q_FREE = 1, B_Q_READY = 2, B_KV_FULL = 3, B_KV_FREE = 6, B_S_FULL = 9,
    B_P_FULL = 12, B_O_DONE = 15, B_UNIT_DONE = 18, B_X_FULL = 19, B_X_EMPTY = 20, B_DRAIN = 21
};

struct MlaSched {
    int64_t total;      // chunks over all units
    int64_t units;
    int cpu;            // chunks per unit
    int clusters;
    int seg_max;
    int q_head_inner;   // q tensor map dims are {d, head, s1, b} (else {d, s1, head, b})
};

__host__ __device__ inline int64_t mla_range_begin(int64_t c, const MlaSched& s) {
    return c * s.total / s.clusters;
}
__host__ __device__ inline int64_t mla_cluster_of(int64_t x, const MlaSched& s) {
    return ((x + 1) * s.clusters - 1) / s.total;
}

struct UCoord {
    int b, n2, s1;
};
__device__ __forceinline__ UCoord ucoord(int64_t u, const SfaParams& p) {
    UCoord c;
    c.s1 = (int)(u % p.S1);
    c.n2 = (int)((u / p.S1) % p.N2);
    c.b = (int)(u / ((int64_t)p.S1 * p.N2));
    return c;
}

template <class E>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
sfa_mla_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mqr,
               const SfaParams p, const MlaSched sch) {
    using T = typename E::T;
    using L = MlaSmem;
    constexpr bool kBf16 = std::is_same<E, BF16>::value;
    constexpr uint32_t kIdescQK = idesc_f16(kHeads, kChunk, kBf16, false, false);
    constexpr uint32_t kIdescPV = idesc_f16(kHeads, kHalfDv, kBf16, false, true);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int64_t cl = blockIdx.x >> 1;
    const int c_begin = (int)mla_range_begin(cl, sch), c_end = (int)mla_range_begin(cl + 1, sch);
    const int n = c_end - c_begin;
    auto bar = [&](int i) { return sbase + L::bars + 8 * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar(B_QR_FULL), 1);
        mbar_init(bar(B_Q_FREE), 1);
        mbar_init(bar(B_Q_READY), kSoftThreads);
        mbar_init(bar(B_DRAIN), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), kProdThreads + kProdThreads / 32);
            mbar_init(bar(B_KV_FREE + s), 1);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_FULL + b), kSoftThreads);
            mbar_init(bar(B_O_DONE + b), 1);
        }
        mbar_init(bar(B_UNIT_DONE), 1);
        mbar_init(bar(B_X_FULL), 1);      // own arrive.expect_tx + the peer's bulk copy bytes
        mbar_init(bar(B_X_EMPTY), 1);     // the peer has read what this CTA sent it
        fence_barrier_init();
    }
    // launched with programmatic dependent launch: nothing above touches
    // global memory; wait here for the previous grid in the stream, and let
    // the next one (the merge, or the next call) start launching
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == kMmaWarp) tmem_alloc(sbase + L::misc, kTmemCols);
    tc_fence_before();
    cluster_sync();      // both CTAs' barriers exist before any remote access
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::misc);

    const int cpu = sch.cpu;
    auto unit_of = [&](int c) { return c / cpu; };       // chunk counts fit in int (host check)

    if (warp >= kProdWarp0) {
        // ============================ producers ============================
        // Warp pw gathers slots 16 pw .. 16 pw + 15 of every chunk: per slot
        // one 512-byte nope run (lane = 16-byte piece), then the 64-byte rope
        // runs of its 16 rows, 8 rows per instruction.  Lane l holds the index
        // of slot 16 pw + l % 16.  Unit coordinates advance incrementally.
        const int pw = warp - kProdWarp0;
        const int sl = lane & 15;
        struct Cursor {
            int cc;
            UCoord uc;
            const int32_t* ig;
            const T* kg;
        };
        auto point = [&](Cursor& k) {
            k.ig = p.idx + k.uc.b * p.i_sb + k.uc.n2 * p.i_sh + k.uc.s1 * p.i_ss;
            k.kg = static_cast<const T*>(p.k) + k.uc.b * p.k_sb + k.uc.n2 * p.k_sh;
        };
        auto cursor_at = [&](int c) {
            Cursor k;
            const int u = c / cpu;
            k.cc = c - u * cpu;
            k.uc = ucoord(u, p);
            point(k);
            return k;
        };
        auto advance = [&](Cursor& k) {
            if (++k.cc < cpu) return;
            k.cc = 0;
            if (++k.uc.s1 == p.S1) {
                k.uc.s1 = 0;
                if (++k.uc.n2 == p.N2) {
                    k.uc.n2 = 0;
                    ++k.uc.b;
                }
            }
            point(k);
        };
        Cursor fk = cursor_at(c_begin);                      // index fetch: kLookahead ahead
        Cursor pk = cursor_at(c_begin);                      // L2 prefetch: kPrefetch ahead
        Cursor k = cursor_at(c_begin);                       // the chunk being gathered
        for (int t = 0; t < kPrefetch; ++t) advance(pk);
        int fc = c_begin;
        auto fetch = [&]() {
            int id = kNoSlot;
            if (fc < c_end) {
                const int j = fk.cc * kChunk + 16 * pw + sl;
                if (j < p.topK) id = fk.ig[j];
                advance(fk);
                ++fc;
            }
            return id;
        };
        int ring[kLookahead];
#pragma unroll
        for (int r = 0; r < kLookahead; ++r) ring[r] = fetch();
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(bar(B_KV_FREE + s), ((i / kStages) & 1) ^ 1, p.err_word, abort_flag)) break;
            const int myid = ring[0];
#pragma unroll
            for (int r = 0; r + 1 < kLookahead; ++r) ring[r] = ring[r + 1];
            ring[kLookahead - 1] = fetch();
            const int diag = k.uc.s1 + (p.S2 - p.S1);
            const bool in_range = myid >= 0 && myid < p.S2;
            if (!in_range && myid != kNoSlot && p.validate && lane < 16) atomicOr(p.err_word, kErrIndexRange);
            const bool vis = in_range && !(p.causal && myid > diag);
            const int myrow = in_range ? myid : -1;
            unsigned char* st = smem + L::kv + s * L::kvStage;
            // nope dims [256 rank, +256): panel = lane / 8, 16-byte chunk lane % 8
            const T* nope = k.kg + (int)rank * kHalfDv + 8 * lane;
            const int pn = lane >> 3, c = lane & 7;
#pragma unroll 8
            for (int r = 0; r < 16; ++r) {
                const int id = __shfl_sync(0xffffffffu, myrow, r);
                const int row = 16 * pw + r;
                cp_async_16_zfill(st + pn * L::nopePanel + row * 128 + ((c ^ (row & 7)) << 4),
                                  nope + (id >= 0 ? (int64_t)id * p.k_ss : 0), id >= 0 ? 16 : 0);
            }
            // rope dims [512 + 32 rank, +32): 64-byte rows, chunk c at c ^ ((row / 2) % 4)
            const T* rope = k.kg + 512 + 32 * (int)rank + 8 * (lane & 3);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int r = 8 * t + (lane >> 2);
                const int id = __shfl_sync(0xffffffffu, myrow, r);
                const int row = 16 * pw + r;
                cp_async_16_zfill(st + 4 * L::nopePanel + row * 64 + (((lane & 3) ^ ((row >> 1) & 3)) << 4),
                                  rope + (id >= 0 ? (int64_t)id * p.k_ss : 0), id >= 0 ? 16 : 0);
            }
            cp_async_mbar_arrive(bar(B_KV_FULL + s));
            // rows of chunk i + kPrefetch into L2 ahead of their stage being
            // free: lane l takes slot l % 16, lines l / 16, 2 + l / 16 of its
            // nope run and (lanes < 16) its rope line
            if (i + kPrefetch < n) {
                const int pid = ring[kPrefetch - 1];
                if (pid >= 0 && pid < p.S2) {
                    const char* rowp = reinterpret_cast<const char*>(pk.kg + (int64_t)pid * p.k_ss);
                    prefetch_l2(rowp + 512 * (int)rank + 128 * (lane >> 4));
                    prefetch_l2(rowp + 512 * (int)rank + 256 + 128 * (lane >> 4));
                    if (lane < 16) prefetch_l2(rowp + 1024 + 64 * (int)rank);
                }
                advance(pk);
            }
            const uint32_t mask = __ballot_sync(0xffffffffu, vis) & 0xffffu;
            if (lane == 0) {
                reinterpret_cast<uint16_t*>(smem + L::meta)[4 * s + pw] = (uint16_t)mask;
                mbar_arrive(bar(B_KV_FULL + s));
            }
            advance(k);
        }
        // no copy may still be in flight when the warp leaves
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        // ============================ MMA issue ============================
        // QK(j) may be issued once PV(j - 3) is (its S/P buffer j % 3 is then
        // free in pipe order): QK(i + 1) is required before P(i) can exist,
        // QK(i + 2) goes in when its rows have landed; PV(i) as soon as P(i)
        // is there.  An event loop, so that a later chunk's gather never
        // holds up a ready PV.
        if (lane == 0 && n > 0) {
            tma_prefetch_map(&mq);
            tma_prefetch_map(&mqr);
            uint32_t qfree_phase = 0, q_phase = 0;
            bool ok = true;
            // the unit's Q rope panel (TMA) and its Q nope half (written to
            // tensor memory by the softmax threads)
            auto unit_q = [&](int u) {
                const UCoord uc = ucoord(u, p);
                mbar_arrive_expect_tx(bar(B_QR_FULL), kHeads * 64 + 2 * kHeads * 128);
                const int c1 = sch.q_head_inner ? uc.n2 * kHeads : uc.s1;
                const int c2 = sch.q_head_inner ? uc.s1 : uc.n2 * kHeads;
                tma_load_4d(sbase + L::qr, &mqr, 512 + 32 * (int)rank, c1, c2, uc.b, bar(B_QR_FULL));
                for (int pn = 0; pn < 2; ++pn)
                    tma_load_4d(sbase + L::qn + pn * (kHeads * 128), &mq, (int)rank * kHalfDv + 128 + 64 * pn,
                                c1, c2, uc.b, bar(B_QR_FULL));
                ok = ok && mbar_wait(bar(B_QR_FULL), q_phase, p.err_word, abort_flag);
                ok = ok && mbar_wait(bar(B_Q_READY), q_phase, p.err_word, abort_flag);
                q_phase ^= 1;
                tc_fence_after();
            };
            auto qk = [&](int j) {
                const int s = j % kStages;
                ok = ok && mbar_wait(bar(B_KV_FULL + s), (j / kStages) & 1, p.err_word, abort_flag);
                fence_proxy_async_smem();     // cp.async (generic proxy) data -> tensor core
                tc_fence_after();
                const uint32_t kb = sbase + L::kv + s * L::kvStage;
                const uint32_t d = tmem + kSCol + 64 * (j % kBufs);
                // nope dims [0, 128): A from tensor memory; [128, 256): A from shared memory
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * L::nopePanel + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16_ts(d, tmem + kQnCol + 8 * kk, bd, kIdescQK, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 8; kk < 16; ++kk) {
                    const uint64_t ad = sdesc_sw128(sbase + L::qn + ((kk - 8) >> 2) * (kHeads * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * L::nopePanel + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16(d, ad, bd, kIdescQK, 1u);
                }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t ad = sdesc_sw64(sbase + L::qr + kk * 32, 512);
                    const uint64_t bd = sdesc_sw64(kb + 4 * L::nopePanel + kk * 32, 512);
                    tc_mma_f16(d, ad, bd, kIdescQK, 1u);
                }
                tc_commit(bar(B_S_FULL + j % kBufs));
            };
            int unit_cur = unit_of(c_begin);
            int unit_end = min(c_end, (unit_cur + 1) * cpu) - c_begin;   // first chunk past this unit
            unit_q(unit_cur);
            int next_qk = 0;
            uint64_t idle_since = 0;
            for (int i = 0; i < n && ok;) {
                if (next_qk < unit_end && next_qk <= i + 1) {
                    qk(next_qk++);
                    continue;
                }
                if (next_qk < unit_end && next_qk == i + 2 &&
                    mbar_try_wait(bar(B_KV_FULL + next_qk % kStages), (next_qk / kStages) & 1)) {
                    qk(next_qk++);
                    continue;
                }
                if (!mbar_try_wait(bar(B_P_FULL + i % kBufs), (i / kBufs) & 1)) {
                    // nothing to issue yet: poll, with the same bound as the waits
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint64_t now = global_timer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > 2000000000ull) {
                        atomicOr(p.err_word, kErrWaitTimeout);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    continue;
                }
                idle_since = 0;
                const int s = i % kStages;
                tc_fence_after();
                const uint32_t kb = sbase + L::kv + s * L::kvStage;
                const uint32_t pa = tmem + kSCol + 64 * (i % kBufs);
                const bool first = (i == 0) || (c_begin + i) % cpu == 0;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk) {
                        const uint64_t bd = sdesc_sw128(kb + kk * 16 * 128, L::nopePanel, 1024);
                        const uint32_t acc = (first && part == 0 && kk == 0) ? 0u : 1u;
                        tc_mma_f16_ts(tmem + kOCol, pa + 32 * part + 8 * kk, bd, kIdescPV, acc);
                    }
                tc_commit(bar(B_O_DONE + i % kBufs));
                tc_commit(bar(B_KV_FREE + s));
                ++i;
                if (i == unit_end) {
                    tc_commit(bar(B_UNIT_DONE));   // the unit's O is final
                    if (i < n) {
                        // the rope panel and Q columns are rewritten once
                        // every MMA of the unit is done
                        tc_commit(bar(B_Q_FREE));
                        ok = ok && mbar_wait(bar(B_Q_FREE), qfree_phase, p.err_word, abort_flag);
                        qfree_phase ^= 1;
                        ++unit_cur;
                        unit_end = min(c_end, (unit_cur + 1) * cpu) - c_begin;
                        unit_q(unit_cur);
                    }
                }
            }
            if (!ok) {
                // a wait gave up: let every MMA this thread issued finish
                // (bounded) before the tensor memory is released
                tc_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0, nullptr, nullptr, 100000000ull);
            }
        }
    } else {
        // ============================ softmax ============================
        const int w = tid >> 7;                              // warpgroup: slot / dim half
        const int r = tid & (kHeads - 1);                    // head row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t x_peer = map_peer(sbase + L::x, peer);
        const uint32_t xfull_peer = map_peer(bar(B_X_FULL), peer);
        const uint32_t xempty_peer = map_peer(bar(B_X_EMPTY), peer);
        float* red = reinterpret_cast<float*>(smem + L::red);
        float* red2 = reinterpret_cast<float*>(smem + L::red2);
        volatile int* early_flag = reinterpret_cast<volatile int*>(smem + L::misc + 8);
        // Q nope dims [256 rank + 64 w, +64) of head r into TMEM columns
        // [32 w, 32 w + 32): two 16-bit dims per column (dims [128, 256) of
        // the CTA's half come by TMA into shared memory)
        auto load_qn = [&](int u) {
            const UCoord uc = ucoord(u, p);
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const T*>(p.q) + uc.b * p.q_sb + uc.s1 * p.q_ss +
                (int64_t)(uc.n2 * kHeads + r) * p.q_sh + (int)rank * kHalfDv + 64 * w);
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 x = __ldg(src + j);
                v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
            }
            tmem_st32(lane_base + kQnCol + 32 * w, v);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_Q_READY));
        };
        // send(j): this CTA's partial scores of chunk j to the peer (one bulk
        // copy from the staging buffer into the peer's receive buffer); sv
        // keeps them for the sum
        uint32_t sv[32];
        auto send = [&](int j) {
            mbar_wait(bar(B_S_FULL + j % kBufs), (j / kBufs) & 1, p.err_word, abort_flag);
            tc_fence_after();
            tmem_ld32(lane_base + kSCol + 64 * (j % kBufs) + 32 * w, sv);
            tmem_wait_ld();
            // the staging buffer is free once the peer has read the last copy
            if (tid == 0 && j > 0)
                mbar_wait_cluster(bar(B_X_EMPTY), (j - 1) & 1, p.err_word, abort_flag);
            named_sync(1, kSoftThreads);
            unsigned char* stg = smem + L::stg + r * 256;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4*>(stg + (((8 * w + q) ^ (r & 15)) << 4)) =
                    make_uint4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
            fence_proxy_async_smem();         // generic writes -> bulk copy engine
            named_sync(1, kSoftThreads);
            if (tid == 0) {
                mbar_arrive_expect_tx(bar(B_X_FULL), kXBytes);
                bulk_s2cluster(x_peer, sbase + L::stg, kXBytes, xfull_peer);
            }
        };
        if (n > 0) {
            load_qn(unit_of(c_begin));
            send(0);
        }
        float m_used = -INFINITY, l = 0.f;
        bool first_of_unit = true;
        uint32_t unit_phase = 0;
        for (int i = 0; i < n; ++i) {
            const int c = c_begin + i;
            const int u = unit_of(c);
            const bool last_of_unit = (i + 1 == n) || unit_of(c + 1) != u;
            // ---- receive the peer's partial scores of chunk i ----
            mbar_wait(bar(B_KV_FULL + i % kStages), (i / kStages) & 1, p.err_word, abort_flag);
            mbar_wait(bar(B_X_FULL), i & 1, p.err_word, abort_flag);
            const uint2 vis = reinterpret_cast<const uint2*>(smem + L::meta)[i % kStages];
            const uint32_t vw = w ? vis.y : vis.x;
            const unsigned char* xr = smem + L::x + r * 256;
            float s[32];
            float bmax = -INFINITY;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 o = *reinterpret_cast<const uint4*>(xr + (((8 * w + q) ^ (r & 15)) << 4));
                const float ov[4] = {__uint_as_float(o.x), __uint_as_float(o.y), __uint_as_float(o.z),
                                     __uint_as_float(o.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int jj = 4 * q + e;
                    // both CTAs add the two partials in the same (commutative) way
                    const float v = __uint_as_float(sv[jj]) + ov[e];
                    s[jj] = ((vw >> jj) & 1u) ? v * p.scale_log2 : -INFINITY;
                    bmax = fmaxf(bmax, s[jj]);
                }
            }
            red[w * kHeads + r] = bmax;
            // send chunk i + 1 before this chunk's softmax when its scores are
            // already computed (the copy then overlaps the work below), else
            // after P(i) is out; a new unit's first chunk waits for that unit's
            // Q, written in the epilogue
            if (tid == 0)
                *early_flag = !last_of_unit && mbar_try_wait(bar(B_S_FULL + (i + 1) % kBufs), ((i + 1) / kBufs) & 1);
            named_sync(1, kSoftThreads);      // X read by every thread, row maxima posted
            if (tid == 0) mbar_arrive_remote(xempty_peer);
            bmax = fmaxf(red[r], red[kHeads + r]);
            const bool early = *early_flag != 0;
            if (early) send(i + 1);
            // ---- online softmax over the chunk (mask shared by all heads) ----
            const float m_new = fmaxf(m_used, bmax);
            const bool need = m_new > m_used + kRescaleThreshold;
            const float f = need ? fast_exp2(m_used - m_new) : 1.f;   // 0 while m_used is -inf
            if (need) m_used = m_new;
            uint32_t hw[16], lw[16];
            float lsum = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float a = s[2 * e], b = s[2 * e + 1];
                const float p0 = (a == -INFINITY) ? 0.f : fast_exp2(a - m_used);
                const float p1 = (b == -INFINITY) ? 0.f : fast_exp2(b - m_used);
                lsum += p0 + p1;
                hw[e] = E::pack2(p0, p1);
                const float2 h = E::unpack2(hw[e]);
                lw[e] = E::pack2(p0 - h.x, p1 - h.y);
            }
            l = l * f + lsum;                 // this warpgroup's share of the row sum
            if (!first_of_unit && __any_sync(0xffffffffu, need)) {
                // O is rescaled once P.V of the previous chunk is done: its
                // buffer's barrier, whose previous use (chunk i - 4) is done
                // and whose next (chunk i + 2) cannot be, so the phase is
                // unambiguous.
                const int pb = (i - 1) % kBufs;
                mbar_wait(bar(B_O_DONE + pb), ((i - 1) / kBufs) & 1, p.err_word, abort_flag);
                tc_fence_after();
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t ov[32];
                    tmem_ld32(lane_base + kOCol + 128 * w + 32 * cb, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                    tmem_st32(lane_base + kOCol + 128 * w + 32 * cb, ov);
                }
            }
            // P over the S columns of its chunk: high parts in [sp, sp + 32),
            // remainders in [sp + 32, sp + 64); slot j -> column j / 2
            const uint32_t sp = kSCol + 64 * (i % kBufs);
            tmem_st16(lane_base + sp + 16 * w, hw);
            tmem_st16(lane_base + sp + 32 + 16 * w, lw);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + i % kBufs));
            first_of_unit = false;
            if (!last_of_unit) {
                if (!early) send(i + 1);
                continue;
            }

            // ---- epilogue of unit u: dims [256 rank + 128 w, +128) ----
            mbar_wait(bar(B_UNIT_DONE), unit_phase, p.err_word, abort_flag);
            unit_phase ^= 1;
            tc_fence_after();
            red2[w * kHeads + r] = l;
            named_sync(1, kSoftThreads);
            const float lt = red2[r] + red2[kHeads + r];
            const int64_t first = (int64_t)u * cpu, lastc = first + cpu - 1;
            const int64_t c_lo = mla_cluster_of(first, sch), c_hi = mla_cluster_of(lastc, sch);
            const bool split = c_hi > c_lo;
            const UCoord uc = ucoord(u, p);
            const int n1 = uc.n2 * kHeads + r;
            const int64_t row = (int64_t)u * kHeads + r;
            const int64_t slot = row * sch.seg_max + (cl - c_lo);
            const bool empty = !(lt > 0.f);
            const float inv = empty ? 0.f : 1.f / lt;
            const int d0 = (int)rank * kHalfDv + 128 * w;
            T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss + d0;
            float* wo = split ? p.ws_o + slot * kDv + d0 : nullptr;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t ov[32];
                tmem_ld32(lane_base + kOCol + 128 * w + 32 * cb, ov);
                tmem_wait_ld();
                if (!split) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 q;
                        q.x = empty ? 0u : E::pack2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
                        q.y = empty ? 0u : E::pack2(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
                        q.z = empty ? 0u : E::pack2(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv);
                        q.w = empty ? 0u : E::pack2(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + 32 * cb + j) = q;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(wo + 32 * cb + j) =
                            make_float4(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]),
                                        __uint_as_float(ov[j + 2]), __uint_as_float(ov[j + 3]));
                }
            }
            if (!split) {
                if (rank == 0 && w == 0 && p.lse)
                    p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] =
                        empty ? -INFINITY : (m_used + __log2f(lt)) * kLn2;
            } else if (w == 0) {
                // (m, l) of this part; both CTAs of the cluster write the same values
                p.ws_ml[slot * 2] = m_used;
                p.ws_ml[slot * 2 + 1] = lt;
            }
            m_used = -INFINITY;
            l = 0.f;
            first_of_unit = true;
            // tensor memory's Q columns are free (every MMA of the unit is
            // done): the next unit's Q, then its first chunk's exchange
            if (i + 1 < n) {
                load_qn(u + 1);
                send(i + 1);
            }
        }
        // the last copy sent to the peer has landed before this CTA can leave
        if (tid == 0 && n > 0)
            mbar_wait_cluster(bar(B_X_EMPTY), (n - 1) & 1, p.err_word, nullptr, 100000000ull);
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();      // the peer no longer writes into this CTA's shared memory
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge of the parts of split units: one warp per output row (unit, head);
// lane l combines dims [16 l, 16 l + 16) of every part.  Rows of units that a
// single cluster finished were written by the main kernel.
template <class E>
__global__ void __launch_bounds__(512) sfa_mla_combine(const SfaParams p, const MlaSched sch) {
    using T = typename E::T;
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= sch.units * kHeads) return;
    const int64_t u = row / kHeads;
    const int h = (int)(row % kHeads);
    const int64_t first = u * sch.cpu;
    const int64_t c_lo = mla_cluster_of(first, sch), c_hi = mla_cluster_of(first + sch.cpu - 1, sch);
    const int nseg = (int)(c_hi - c_lo + 1);
    if (nseg == 1) return;
    const float* ml = p.ws_ml + row * sch.seg_max * 2;
    float M = -INFINITY;
    for (int k = 0; k < nseg; ++k) M = fmaxf(M, ml[2 * k]);
    float wk[kMaxSeg];
    float Ls = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxSeg; ++k) {
        wk[k] = 0.f;
        if (k < nseg) {
            wk[k] = rescale_factor(ml[2 * k], M);
            Ls += wk[k] * ml[2 * k + 1];
        }
    }
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    const float* base = p.ws_o + row * sch.seg_max * kDv + 16 * lane;
#pragma unroll
    for (int k = 0; k < kMaxSeg; ++k) {
        if (k < nseg) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = *reinterpret_cast<const float4*>(base + (int64_t)k * kDv + 4 * q);
                acc[4 * q] += wk[k] * x.x;
                acc[4 * q + 1] += wk[k] * x.y;
                acc[4 * q + 2] += wk[k] * x.z;
                acc[4 * q + 3] += wk[k] * x.w;
            }
        }
    }
    const bool empty = !(Ls > 0.f);
    const float inv = empty ? 0.f : 1.f / Ls;
    const UCoord uc = ucoord(u, p);
    const int n1 = uc.n2 * kHeads + h;
    T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss + 16 * lane;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint4 o;
        o.x = empty ? 0u : E::pack2(acc[8 * q] * inv, acc[8 * q + 1] * inv);
        o.y = empty ? 0u : E::pack2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv);
        o.z = empty ? 0u : E::pack2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv);
        o.w = empty ? 0u : E::pack2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv);
        *reinterpret_cast<uint4*>(orow + 8 * q) = o;
    }
    if (lane == 0 && p.lse)
        p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] = empty ? -INFINITY : (M + __log2f(Ls)) * kLn2;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D maps of q ordered by stride: {d, head, s1, b} when heads are adjacent
// (BSND), else {d, s1, head, b}.  Box = `box_d` dims x 128 heads: 64 dims with
// 128-byte swizzle (Q nope panels) or 32 dims with 64-byte swizzle (a CTA's
// rope dims).
bool make_q_map(CUtensorMap* map, const SfaParams& p, bool bf16, bool head_inner, int box_d) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t n_a = head_inner ? p.N1 : p.S1, n_b = head_inner ? p.S1 : p.N1;
    const int64_t s_a = head_inner ? p.q_sh : p.q_ss, s_b = head_inner ? p.q_ss : p.q_sh;
    const cuuint64_t gdim[4] = {(cuuint64_t)p.Dk, n_a, n_b, (cuuint64_t)p.B};
    const cuuint64_t gstride[3] = {(cuuint64_t)s_a * 2, (cuuint64_t)s_b * 2, (cuuint64_t)p.q_sb * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, head_inner ? (cuuint32_t)kHeads : 1u,
                               head_inner ? 1u : (cuuint32_t)kHeads, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
              const_cast<void*>(p.q), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
              box_d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device setup of the MLA kernel (cached): the shared-memory opt-in and
// the number of clusters that fit on the device at once -- pairs of SMs
// inside one GPC, so possibly fewer than SMs / 2.  Returns 0 on failure.
template <class E>
int prepare_device(int num_sms) {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] > 0) return cache[dev];
    if (cudaFuncSetAttribute(sfa_mla_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MlaSmem::alloc) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = MlaSmem::alloc;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sfa_mla_kernel<E>, &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = num_sms / 2;
    }
    if (n > num_sms / 2) n = num_sms / 2;
    if (n < 1) n = 1;
    cache[dev] = n;
    return n;
}

template <class E>
cudaError_t launch_t(SfaParams p, int num_sms, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const int resident = prepare_device<E>(num_sms);
    if (resident < 1) return cudaErrorInvalidConfiguration;
    MlaSched s;
    s.q_head_inner = p.q_sh <= p.q_ss ? 1 : 0;
    CUtensorMap mq, mqr;
    const bool bf16 = std::is_same<E, BF16>::value;
    if (!make_q_map(&mq, p, bf16, s.q_head_inner != 0, 64) ||
        !make_q_map(&mqr, p, bf16, s.q_head_inner != 0, 32))
        return cudaErrorInvalidValue;
    s.cpu = (p.topK + kChunk - 1) / kChunk;
    s.units = (int64_t)p.B * p.N2 * p.S1;
    s.total = s.units * s.cpu;
    int64_t clusters = resident;
    if (p.num_ctas > 0) clusters = (p.num_ctas + 1) / 2;    // tuning / tests
    // fewer units than resident clusters: split every unit into the same
    // number of segments, so that each cluster's range lies inside one unit
    // (MLA decode, 32 units of 32 chunks: 64 clusters 70.5 us against 77.2 us
    // for the 76 resident ones)
    if (p.num_ctas == 0) {
        const int64_t seg = clusters / s.units;
        if (seg >= 2) clusters = s.units * (seg < s.cpu ? seg : s.cpu);
    }
    if (clusters > s.total) clusters = s.total;
    if (clusters < 1) clusters = 1;
    // keep the number of clusters sharing one unit within kMaxSeg: a unit of
    // cpu chunks meets at most ceil(cpu / shortest range) + 1 ranges
    for (;;) {
        const int64_t lmin = s.total / clusters;
        int64_t seg = (s.cpu + lmin - 1) / lmin + 1;
        if (seg > s.cpu) seg = s.cpu;
        if (seg <= kMaxSeg || clusters == 1) {
            s.seg_max = (int)seg;
            break;
        }
        clusters = clusters * 3 / 4;
    }
    s.clusters = (int)clusters;
    if (s.seg_max > 1) {
        const int64_t rows = s.units * kHeads;
        const size_t need = (size_t)rows * s.seg_max * ((size_t)kDv + 2) * sizeof(float);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
        p.ws_o = static_cast<float*>(ws);
        p.ws_ml = p.ws_o + rows * s.seg_max * kDv;
    }
    cudaError_t err = launch_pdl(sfa_mla_kernel<E>, dim3((unsigned)(2 * s.clusters)), dim3(kThreads),
                                 (size_t)MlaSmem::alloc, stream, mq, mqr, p, s);
    count_launches(1);
    if (err != cudaSuccess || s.seg_max == 1) return err;
    // merge of split units; launched early (programmatic dependent launch),
    // it waits for the main kernel's results before reading them
    const int64_t rows = s.units * kHeads;
    err = launch_pdl(sfa_mla_combine<E>, dim3((unsigned)((rows + 15) / 16)), dim3(512), 0, stream, p, s);
    count_launches(1);
    return err;
}

}  // namespace

bool mla_supported(const SfaParams& p) {
    const bool prefix = (p.v == p.k) && (p.v_ss == p.k_ss);
    const int64_t chunks = (int64_t)p.B * p.N2 * p.S1 * ((p.topK + kChunk - 1) / kChunk);
    return p.G == kHeads && p.Dk == kDk && p.Dv == kDv && prefix && chunks < (int64_t(1) << 31);
}

size_t mla_ws_bytes(const SfaParams& p) {
    const int64_t cpu = (p.topK + kChunk - 1) / kChunk;
    const int64_t seg = cpu < kMaxSeg ? cpu : kMaxSeg;
    const int64_t rows = (int64_t)p.B * p.N2 * p.S1 * kHeads;
    return seg > 1 ? (size_t)rows * seg * ((size_t)kDv + 2) * sizeof(float) : 0;
}

cudaError_t launch_sfa_mla(const SfaParams& p, sfa_dtype dtype, int num_sms, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
    if (!mla_supported(p)) return cudaErrorInvalidValue;
    return dtype == SFA_DTYPE_BF16 ? launch_t<BF16>(p, num_sms, ws, ws_bytes, stream)
                                   : launch_t<F16>(p, num_sms, ws, ws_bytes, stream);
}

}  // namespace sfa
