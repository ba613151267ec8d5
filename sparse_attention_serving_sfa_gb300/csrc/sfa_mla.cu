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
// memory, so a unit (one index list and its 128 heads) is computed by a pair
// of CTAs that split the output dims: CTA r owns O dims [256 r, 256 r + 256).
// Each CTA of the pair gathers the whole selected K rows (1152 bytes; the
// second read of a row comes from L2), computes the full S = Q K^T over all
// 576 dims itself and runs its own online softmax -- the two CTAs never
// exchange data, so neither waits for the other -- then O_r += P V_r for its
// half of Dv (P as a 16-bit high part plus remainder, ~fp32 accurate).  The
// pair is launched as a cluster only so that both halves of a unit run at the
// same time and share the row reads in L2.
//
// Tensor memory (512 columns): Q dims [0, 256) as the A operand of Q.K^T in
// [0, 128) | two S/P buffers [128, 192), [192, 256) (a chunk's scores, then
// its probabilities written over them as the A operand of P.V) | O [256, 512).
// Shared memory: two stages of a chunk's K rows (9 panels of 64 dims, 128-byte
// swizzle, 72 KB each) and Q dims [256, 576) (5 panels, 80 KB).
//
// Roles per CTA (9 warps): 4 softmax warps (one warpgroup, thread = head =
// TMEM lane, all 64 slots of a chunk), 1 MMA warp (Q TMA, tcgen05.mma issue
// from an event loop: Q.K^T of chunk i + 1 as soon as its rows have landed,
// P.V of chunk i as soon as its P is written), 4 producer warps (cp.async
// gather of whole rows, index prefetch, L2 prefetch two chunks ahead,
// visibility masks).  Work is stream-K over (unit, chunk) pairs per pair of
// CTAs.  When every unit is cut into exactly two ranges, the two pairs of a
// unit run as one 4-CTA cluster and the first merges the second's O and
// (m, l) through distributed shared memory; otherwise the parts of a unit
// split over pairs are written as fp32 partials and merged by a second
// kernel.  (An earlier design split the K dims over the
// pair and exchanged partial scores through distributed shared memory every
// chunk: per-chunk timelines showed the pair running in lockstep through that
// exchange, ~5,100 cycles per chunk for ~1,900 cycles of tensor work.)
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
constexpr int kHalfDv = 256;              // V / O dims per CTA
constexpr int kStages = 2;
constexpr int kBufs = 2;                  // S/P buffers in tensor memory
constexpr int kSoftThreads = 128;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kProdThreads = 128;
constexpr int kThreads = kSoftThreads + 32 + kProdThreads;
constexpr int kTmemCols = 512;
constexpr int kQtDims = 256;              // Q dims held in tensor memory
constexpr int kQtCol = 0, kSCol = 128, kOCol = 256;
constexpr int kPanels = kDk / 64;         // 9 panels of 64 dims per K row
constexpr int kQsPanels = (kDk - kQtDims) / 64;   // 5 Q panels in shared memory
constexpr int kPieces = kDk / 8;          // 16-byte pieces per K row
constexpr int kLookahead = 6;
constexpr int kPrefetch = 2;              // chunks ahead that the producers pull into L2
constexpr int kNoSlot = INT_MIN;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSeg = 8;                // pairs sharing one unit

struct MlaSmem {
    static constexpr int panel = kChunk * 128;              // 64 rows x 128 B (64 dims)
    static constexpr int kvStage = kPanels * panel;         // 72 KB: a chunk's K rows
    static constexpr int qpanel = kHeads * 128;             // 128 heads x 128 B
    static constexpr int kv = 0;
    static constexpr int qs = kv + kStages * kvStage;       // Q dims [256, 576)
    static constexpr int bars = qs + kQsPanels * qpanel;
    static constexpr int meta = bars + 16 * 8;              // [stage][4] uint16 visibility masks
    static constexpr int misc = meta + kStages * 8;         // tmem base, abort flag
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;
};
static_assert(MlaSmem::alloc <= 232448, "dynamic shared memory per block");
static_assert(MlaSmem::kvStage % 1024 == 0 && MlaSmem::qs % 1024 == 0 && MlaSmem::qpanel % 1024 == 0,
              "swizzle atoms must stay aligned");

enum {
    B_Q_FULL = 0, B_Q_FREE = 1, B_Q_READY = 2, B_KV_FULL = 3, B_KV_FREE = 5, B_S_FULL = 7,
    B_P_FULL = 9, B_O_DONE = 11, B_UNIT_DONE = 13, B_DRAIN = 14
};

struct MlaSched {
    int64_t total;      // chunks over all units
    int64_t units;
    int cpu;            // chunks per unit
    int clusters;       // CTA pairs
    int seg_max;
    int q_head_inner;   // q tensor map dims are {d, head, s1, b} (else {d, s1, head, b})
    int quad;           // every unit is two ranges run by the two pairs of one 4-CTA
                        // cluster, merged in distributed shared memory
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

// Launched in clusters of 2 CTAs (a pair), or of 4 (two pairs holding the two
// ranges of one unit) when sch.quad is set.
template <class E>
__global__ void __launch_bounds__(kThreads, 1)
sfa_mla_kernel(const __grid_constant__ CUtensorMap mq, const SfaParams p, const MlaSched sch) {
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
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1;                  // this CTA's half of the output dims
    const int64_t cl = blockIdx.x >> 1;
    const int c_begin = (int)mla_range_begin(cl, sch), c_end = (int)mla_range_begin(cl + 1, sch);
    const int n = c_end - c_begin;
    auto bar = [&](int i) { return sbase + L::bars + 8 * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_FREE), 1);
        mbar_init(bar(B_Q_READY), kSoftThreads);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_UNIT_DONE), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), kProdThreads + kProdThreads / 32);
            mbar_init(bar(B_KV_FREE + s), 1);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_FULL + b), kSoftThreads);
            mbar_init(bar(B_O_DONE + b), 1);
        }
        fence_barrier_init();
    }
    // launched with programmatic dependent launch: nothing above touches
    // global memory; wait here for the previous grid in the stream, and let
    // the next one (the merge, or the next call) start launching.  When the
    // caller states that the inputs were ready before that grid, the softmax
    // threads wait instead before their first write (a unit's epilogue);
    // until then the kernel only reads q, k and the indices.  (A CTA of this
    // kernel fills an SM's shared memory, so it starts only on an SM the
    // previous grid has left, with its tensor memory released.)
    if (!p.inputs_ready) grid_dependency_wait();
    grid_launch_dependents();
    if (warp == kMmaWarp) tmem_alloc(sbase + L::misc, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::misc);

    const int cpu = sch.cpu;
    auto unit_of = [&](int c) { return c / cpu; };       // chunk counts fit in int (host check)

    if (warp >= kProdWarp0) {
        // ============================ producers ============================
        // Warp pw gathers slots 16 pw .. 16 pw + 15 of every chunk, one whole
        // row (72 16-byte pieces: lane = piece, three instructions) at a time,
        // piece c of panel q at row * 128 + ((c ^ row % 8) << 4) of the
        // panel.  Lane l holds the index of slot 16 pw + l % 16.
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
#pragma unroll 4
            for (int r = 0; r < 16; ++r) {
                const int id = __shfl_sync(0xffffffffu, myrow, r);
                const int row = 16 * pw + r;
                const T* src = k.kg + (id >= 0 ? (int64_t)id * p.k_ss : 0);
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    const int pc = lane + 32 * t;
                    if (pc < kPieces) {
                        const int q = pc >> 3, c = pc & 7;
                        cp_async_16_zfill(st + q * L::panel + row * 128 + ((c ^ (row & 7)) << 4),
                                          src + 8 * pc, id >= 0 ? 16 : 0);
                    }
                }
            }
            cp_async_mbar_arrive(bar(B_KV_FULL + s));
            // rows of chunk i + kPrefetch into L2 ahead of their stage being
            // free: lane l takes slot l % 16 and 5 (l < 16) or 4 of its nine
            // 128-byte lines
            if (i + kPrefetch < n) {
                const int pid = ring[kPrefetch - 1];
                if (pid >= 0 && pid < p.S2) {
                    const char* rowp = reinterpret_cast<const char*>(pk.kg + (int64_t)pid * p.k_ss);
                    const int l0 = (lane >> 4) * 5, l1 = (lane >> 4) ? 9 : 5;
                    for (int line = l0; line < l1; ++line) prefetch_l2(rowp + 128 * line);
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
        // Q.K^T(j) needs its rows and S buffer j % 2, free once P.V(j - 2) is
        // issued (tensor-core order); P.V(i) needs P(i).  An event loop, so
        // that a ready P.V never waits behind a later chunk's gather.
        if (lane == 0 && n > 0) {
            tma_prefetch_map(&mq);
            uint32_t qfree_phase = 0, q_phase = 0;
            bool ok = true;
            // the unit's Q dims [256, 576) by TMA, and its dims [0, 256)
            // written to tensor memory by the softmax threads
            auto unit_q = [&](int u) {
                const UCoord uc = ucoord(u, p);
                mbar_arrive_expect_tx(bar(B_Q_FULL), kQsPanels * L::qpanel);
                const int c1 = sch.q_head_inner ? uc.n2 * kHeads : uc.s1;
                const int c2 = sch.q_head_inner ? uc.s1 : uc.n2 * kHeads;
                for (int pn = 0; pn < kQsPanels; ++pn)
                    tma_load_4d(sbase + L::qs + pn * L::qpanel, &mq, kQtDims + 64 * pn, c1, c2, uc.b,
                                bar(B_Q_FULL));
                ok = ok && mbar_wait(bar(B_Q_FULL), q_phase, p.err_word, abort_flag);
                ok = ok && mbar_wait(bar(B_Q_READY), q_phase, p.err_word, abort_flag);
                q_phase ^= 1;
                tc_fence_after();
            };
            auto qk = [&](int j) {
                const int s = j % kStages;
                fence_proxy_async_smem();     // cp.async (generic proxy) data -> tensor core
                tc_fence_after();
                const uint32_t kb = sbase + L::kv + s * L::kvStage;
                const uint32_t d = tmem + kSCol + 64 * (j % kBufs);
                // dims [0, 256): A from tensor memory; [256, 576): A from shared memory
#pragma unroll
                for (int kk = 0; kk < kQtDims / 16; ++kk) {
                    const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * L::panel + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16_ts(d, tmem + kQtCol + 8 * kk, bd, kIdescQK, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = kQtDims / 16; kk < kDk / 16; ++kk) {
                    const int qk_ = kk - kQtDims / 16;
                    const uint64_t ad =
                        sdesc_sw128(sbase + L::qs + (qk_ >> 2) * L::qpanel + (qk_ & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * L::panel + (kk & 3) * 32, 16, 1024);
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
                // Q.K^T of the next chunk: required before anything else when
                // it is chunk i itself; one chunk ahead when its rows are in
                if (next_qk < unit_end && next_qk <= i) {
                    ok = mbar_wait(bar(B_KV_FULL + next_qk % kStages), (next_qk / kStages) & 1, p.err_word,
                                   abort_flag);
                    if (!ok) break;
                    qk(next_qk++);
                    continue;
                }
                // P.V of chunk i as soon as its P is written (it frees the
                // stage); until then Q.K^T of the next chunk if its rows are in
                if (!mbar_test_wait(bar(B_P_FULL + i % kBufs), (i / kBufs) & 1)) {
                    if (next_qk < unit_end && next_qk == i + 1 &&
                        mbar_test_wait(bar(B_KV_FULL + next_qk % kStages), (next_qk / kStages) & 1)) {
                        qk(next_qk++);
                        continue;
                    }
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
                // O_r += P V_r: V_r = dims [256 r, 256 r + 256) of the chunk's
                // rows (panels 4 r .. 4 r + 3), an MN-major operand
                const uint32_t vb = sbase + L::kv + s * L::kvStage + 4 * (int)rank * L::panel;
                const uint32_t pa = tmem + kSCol + 64 * (i % kBufs);
                const bool first = (i == 0) || (c_begin + i) % cpu == 0;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk) {
                        const uint64_t bd = sdesc_sw128(vb + kk * 16 * 128, L::panel, 1024);
                        const uint32_t acc = (first && part == 0 && kk == 0) ? 0u : 1u;
                        tc_mma_f16_ts(tmem + kOCol, pa + 32 * part + 8 * kk, bd, kIdescPV, acc);
                    }
                tc_commit(bar(B_O_DONE + i % kBufs));
                tc_commit(bar(B_KV_FREE + s));
                ++i;
                if (i == unit_end) {
                    tc_commit(bar(B_UNIT_DONE));   // the unit's O is final
                    if (i < n) {
                        // the Q panels and Q columns are rewritten once every
                        // MMA of the unit is done
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
        const int r = tid;                                   // head row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        // Q dims [0, 256) of head r into TMEM columns [0, 128): two 16-bit
        // dims per column (dims [256, 576) come by TMA into shared memory)
        auto load_q = [&](int u) {
            const UCoord uc = ucoord(u, p);
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const T*>(p.q) + uc.b * p.q_sb + uc.s1 * p.q_ss +
                (int64_t)(uc.n2 * kHeads + r) * p.q_sh);
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 x = __ldg(src + 8 * cb + j);
                    v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
                }
                tmem_st32(lane_base + kQtCol + 32 * cb, v);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_Q_READY));
        };
        if (n > 0) load_q(unit_of(c_begin));
        float m_used = -INFINITY, l = 0.f;
        bool first_of_unit = true;
        uint32_t unit_phase = 0;
        for (int i = 0; i < n; ++i) {
            const int c = c_begin + i;
            const int u = unit_of(c);
            const bool last_of_unit = (i + 1 == n) || unit_of(c + 1) != u;
            // the chunk's visibility masks, then its scores
            mbar_wait(bar(B_KV_FULL + i % kStages), (i / kStages) & 1, p.err_word, abort_flag);
            const uint2 vm = reinterpret_cast<const uint2*>(smem + L::meta)[i % kStages];
            const uint64_t vis = ((uint64_t)vm.y << 32) | vm.x;   // bit j = slot j visible
            mbar_wait(bar(B_S_FULL + i % kBufs), (i / kBufs) & 1, p.err_word, abort_flag);
            tc_fence_after();
            uint32_t sv[64];
            const uint32_t sp = kSCol + 64 * (i % kBufs);
            tmem_ld32(lane_base + sp, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(lane_base + sp + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_wait_ld();
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float v = ((vis >> j) & 1ull) ? __uint_as_float(sv[j]) * p.scale_log2 : -INFINITY;
                sv[j] = __float_as_uint(v);
                mx4[j & 3] = fmaxf(mx4[j & 3], v);
            }
            const float bmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            // ---- online softmax over the chunk (mask shared by all heads) ----
            const float m_new = fmaxf(m_used, bmax);
            const bool need = m_new > m_used + kRescaleThreshold;
            const float f = need ? fast_exp2(m_used - m_new) : 1.f;   // 0 while m_used is -inf
            if (need) m_used = m_new;
            uint32_t hw[32], lw[32];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float a = __uint_as_float(sv[2 * e]), b = __uint_as_float(sv[2 * e + 1]);
                const float p0 = (a == -INFINITY) ? 0.f : fast_exp2(a - m_used);
                const float p1 = (b == -INFINITY) ? 0.f : fast_exp2(b - m_used);
                ls[e & 3] += p0 + p1;
                hw[e] = E::pack2(p0, p1);
                const float2 h = E::unpack2(hw[e]);
                lw[e] = E::pack2(p0 - h.x, p1 - h.y);
            }
            l = l * f + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
            if (!first_of_unit && __any_sync(0xffffffffu, need)) {
                // O is rescaled once P.V of the previous chunk is done: its
                // buffer's barrier, whose previous use (chunk i - 3) is done
                // (this chunk's Q.K^T followed it in tensor-core order) and
                // whose next (chunk i + 1) cannot be, so the phase is
                // unambiguous.
                const int pb = (i - 1) % kBufs;
                mbar_wait(bar(B_O_DONE + pb), ((i - 1) / kBufs) & 1, p.err_word, abort_flag);
                tc_fence_after();
#pragma unroll 1
                for (int cb = 0; cb < kHalfDv / 32; ++cb) {
                    uint32_t ov[32];
                    tmem_ld32(lane_base + kOCol + 32 * cb, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                    tmem_st32(lane_base + kOCol + 32 * cb, ov);
                }
            }
            // P over the S columns of its chunk: high parts in [sp, sp + 32),
            // remainders in [sp + 32, sp + 64); slot j -> column j / 2
            tmem_st32(lane_base + sp, hw);
            tmem_st32(lane_base + sp + 32, lw);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + i % kBufs));
            first_of_unit = false;
            if (!last_of_unit) continue;

            // ---- epilogue of unit u: this CTA's dims [256 rank, +256) ----
            if (p.inputs_ready) grid_dependency_wait();   // (returns at once after the first time)
            mbar_wait(bar(B_UNIT_DONE), unit_phase, p.err_word, abort_flag);
            unit_phase ^= 1;
            tc_fence_after();
            const int64_t first = (int64_t)u * cpu, lastc = first + cpu - 1;
            const int64_t c_lo = mla_cluster_of(first, sch), c_hi = mla_cluster_of(lastc, sch);
            const bool split = c_hi > c_lo;
            if (sch.quad) {
                // this range's O (float4 j of head r at [j][r]: consecutive
                // heads, consecutive 16 bytes) and (m, l) stay in shared
                // memory (the stages and Q panels are idle: the unit's MMAs
                // are done and every copy has landed) for the cluster merge
                // at the end of the kernel
                float4* so = reinterpret_cast<float4*>(smem + L::kv);
#pragma unroll 1
                for (int cb = 0; cb < kHalfDv / 32; ++cb) {
                    uint32_t ov[32];
                    tmem_ld32(lane_base + kOCol + 32 * cb, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        so[(8 * cb + t) * kHeads + r] =
                            make_float4(__uint_as_float(ov[4 * t]), __uint_as_float(ov[4 * t + 1]),
                                        __uint_as_float(ov[4 * t + 2]), __uint_as_float(ov[4 * t + 3]));
                }
                reinterpret_cast<float2*>(smem + L::qs)[r] = make_float2(m_used, l);
                m_used = -INFINITY;
                l = 0.f;
                first_of_unit = true;
                continue;                                // a quad range holds one unit
            }
            const UCoord uc = ucoord(u, p);
            const int n1 = uc.n2 * kHeads + r;
            const int64_t row = (int64_t)u * kHeads + r;
            const int64_t slot = row * sch.seg_max + (cl - c_lo);
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            const int d0 = (int)rank * kHalfDv;
            T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss + d0;
            float* wo = split ? p.ws_o + slot * kDv + d0 : nullptr;
#pragma unroll 1
            for (int cb = 0; cb < kHalfDv / 32; ++cb) {
                uint32_t ov[32];
                tmem_ld32(lane_base + kOCol + 32 * cb, ov);
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
                if (rank == 0 && p.lse)
                    p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] =
                        empty ? -INFINITY : (m_used + __log2f(l)) * kLn2;
            } else {
                // (m, l) of this part; both CTAs of the pair compute the same values
                p.ws_ml[slot * 2] = m_used;
                p.ws_ml[slot * 2 + 1] = l;
            }
            m_used = -INFINITY;
            l = 0.f;
            first_of_unit = true;
            // tensor memory's Q columns are free (every MMA of the unit is
            // done): the next unit's Q
            if (i + 1 < n) load_q(u + 1);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (sch.quad) {
        // the cluster's first pair merges the second pair's state of the unit
        // (same output half: CTA crank + 2), reading its shared memory
        cluster_sync();
        if (crank < 2 && tid < kSoftThreads && n > 0) {
            const int h = tid;
            const float2 a = reinterpret_cast<const float2*>(smem + L::qs)[h];
            const float2 b = ld_cluster_f2(map_peer(smem_u32(smem + L::qs) + 8 * h, crank + 2));
            const float M = fmaxf(a.x, b.x);
            const float fa = rescale_factor(a.x, M), fb = rescale_factor(b.x, M);
            const float Ls = fa * a.y + fb * b.y;
            const bool empty = !(Ls > 0.f);
            const float inv = empty ? 0.f : 1.f / Ls;
            const UCoord uc = ucoord(unit_of(c_begin), p);
            const int n1 = uc.n2 * kHeads + h;
            T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss + (int)rank * kHalfDv;
            const float4* so = reinterpret_cast<const float4*>(smem + L::kv);
            const uint32_t peer_o = map_peer(smem_u32(smem + L::kv), crank + 2);
#pragma unroll 4
            for (int j = 0; j < kHalfDv / 4; j += 2) {
                const float4 x0 = so[j * kHeads + h], x1 = so[(j + 1) * kHeads + h];
                const float4 y0 = ld_cluster_f4(peer_o + 16u * (uint32_t)(j * kHeads + h));
                const float4 y1 = ld_cluster_f4(peer_o + 16u * (uint32_t)((j + 1) * kHeads + h));
                uint4 o;
                o.x = empty ? 0u : E::pack2((fa * x0.x + fb * y0.x) * inv, (fa * x0.y + fb * y0.y) * inv);
                o.y = empty ? 0u : E::pack2((fa * x0.z + fb * y0.z) * inv, (fa * x0.w + fb * y0.w) * inv);
                o.z = empty ? 0u : E::pack2((fa * x1.x + fb * y1.x) * inv, (fa * x1.y + fb * y1.y) * inv);
                o.w = empty ? 0u : E::pack2((fa * x1.z + fb * y1.z) * inv, (fa * x1.w + fb * y1.w) * inv);
                *reinterpret_cast<uint4*>(orow + 4 * j) = o;
            }
            if (rank == 0 && p.lse)
                p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] = empty ? -INFINITY : (M + __log2f(Ls)) * kLn2;
        }
        // the second pair stays resident until the first has read it
        cluster_sync();
    }
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

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
    int n = max_active_clusters(sfa_mla_kernel<E>, kThreads, MlaSmem::alloc, 2);
    if (n < 1) n = num_sms / 2;
    if (n > num_sms / 2) n = num_sms / 2;
    if (n < 1) n = 1;
    cache[dev] = n;
    return n;
}

// Clusters of two pairs (4 CTAs) of the MLA kernel resident at once (cached).
template <class E>
int quad_clusters() {
    static int cache[64] = {0};      // count + 1; 0: not asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) cache[dev] = max_active_clusters(sfa_mla_kernel<E>, kThreads, MlaSmem::alloc, 4) + 1;
    return cache[dev] - 1;
}

template <class E>
cudaError_t launch_t(SfaParams p, int num_sms, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const int resident = prepare_device<E>(num_sms);
    if (resident < 1) return cudaErrorInvalidConfiguration;
    MlaSched s;
    s.q_head_inner = p.q_sh <= p.q_ss ? 1 : 0;
    CUtensorMap mq;
    const bool bf16 = std::is_same<E, BF16>::value;
    if (!make_q_map(&mq, p, bf16, s.q_head_inner != 0, 64)) return cudaErrorInvalidValue;
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
    // every unit cut in two ranges (an even chunk count: range c is chunks
    // [c cpu / 2, (c + 1) cpu / 2)), and room for all the 4-CTA clusters at
    // once: the two pairs of a unit run as one cluster and merge in
    // distributed shared memory, without partials or a merge kernel
    s.quad = (p.num_ctas == 0 && clusters == 2 * s.units && s.cpu % 2 == 0 &&
              quad_clusters<E>() >= s.units) ? 1 : 0;
    if (s.seg_max > 1 && !s.quad) {
        const int64_t rows = s.units * kHeads;
        const size_t need = (size_t)rows * s.seg_max * ((size_t)kDv + 2) * sizeof(float);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
        p.ws_o = static_cast<float*>(ws);
        p.ws_ml = p.ws_o + rows * s.seg_max * kDv;
    }
    cudaError_t err = launch_pdl_clustered(sfa_mla_kernel<E>, dim3((unsigned)(2 * s.clusters)), dim3(kThreads),
                                           (size_t)MlaSmem::alloc, stream, s.quad ? 4 : 2, mq, p, s);
    count_launches(1);
    if (err != cudaSuccess || s.seg_max == 1 || s.quad) return err;
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
