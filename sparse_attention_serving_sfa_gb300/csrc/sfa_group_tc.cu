// Top-K sparse attention for GQA groups of 9 to 16 query heads on the
// 5th-generation tensor cores, with the gathered slots on the MMA's M side:
// the path for calls with many index lists (prefill).  (Groups of up to 8
// heads run faster on the warp-MMA kernel of sfa_decode.cu: measured on
// GB300 at G = 8, Dk 192, 8,192 lists of 2,048 slots, 1.03 ms there against
// 1.45 ms here; at G = 12 and 16 this kernel takes 0.43 and 1.62 ms where the
// CUDA-core kernel takes 2.95 and 11.4 ms.)
//
// "SparseFlashAttention 算子 API 描述", §2 具体子步骤 (sparse gather, scaled dot
// product, bottom-right causal mask, softmax over the selected slots, weighted
// sum), with the softmax evaluated online over 128-slot chunks.  The G query
// heads of one index list are too few for the M side of a tensor-core MMA
// (64 or 128 rows), so both contractions are transposed:
//   S^T [128 slots x 16] = K_sel [128 x Dk] . Q^T [Dk x 16]         (M = 128, N = 16)
//   O^T [Dv x 32]       += V_sel^T [Dv x 128] . [P_hi^T | P_lo^T]    (M = Dv = 128, N = 32)
// with the heads padded to 16 columns (zero rows of Q), and P as a 16-bit high
// part plus the 16-bit rounding of the remainder side by side in one N = 32
// operand (so the V tile is read once per chunk; the output adds the two
// column halves).
//
// Roles (9 warps, one CTA per SM, persistent over contiguous ranges of whole
// index lists -- nothing to merge):
//   - 4 producer warps: warp w gathers slots 32 w .. 32 w + 31 of every
//     chunk with 16-byte cp.async copies, 8 lanes per row, into the K (and V)
//     panels of a ring of shared-memory stages (rows of 64 dims = 128 bytes,
//     128-byte swizzle), plus the list's q rows into the stage's Q panels when
//     the stage held another list before; completion on the stage's mbarrier
//     (cp.async.mbarrier.arrive), a visibility mask per slot;
//   - 1 MMA warp (one thread): Q.K^T of chunk j + 1 as soon as its rows have
//     landed, P.V of chunk j as soon as its P is written (two S buffers in
//     tensor memory), commits that free the stages and P buffers;
//   - 4 softmax warps, thread t = slot t of a chunk = TMEM lane t: the chunk's
//     per-head maxima (a reduce-scatter across the warp, then across the four
//     warps through shared memory), the conditional O rescale (only when a
//     head's running max grows by more than 2^8), P = exp2(s - m) split into
//     the two 16-bit parts and written to shared memory as the B operand of
//     P.V, per-thread running sums; at the end of a list thread t = output
//     dim t reads O^T's row t, divides by the sums and writes out and lse.
// Tensor memory: two S^T buffers, each the sum of one 16-column partial per
// 64-dim panel of Dk (independent MMA chains), and O^T as two 32-column
// accumulators (even and odd 16-slot steps), 128 or 256 columns in all.
#include <cudaTypedefs.h>

#include <limits.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace sfa {
namespace {

constexpr int kChunk = 128;               // slots per chunk (the MMA M side)
constexpr int kN = 16;                    // padded query heads (the MMA N side)
constexpr int kDv = 128;
constexpr int kSoftThreads = 128;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kProdThreads = 128;
constexpr int kThreads = kSoftThreads + 32 + kProdThreads;
constexpr int kLookahead = 6;             // chunks of indices prefetched
constexpr int kNoSlot = INT_MIN;
constexpr float kRescaleThreshold = 8.0f; // log2 units
constexpr int kMaxStages = 4;

enum { B_KV_FULL = 0, B_KV_FREE = B_KV_FULL + kMaxStages, B_S_FULL = B_KV_FREE + kMaxStages,
       B_P_FULL = B_S_FULL + 2, B_P_FREE = B_P_FULL + 2, B_O_DONE = B_P_FREE + 2,
       B_UNIT_DONE = B_O_DONE + 2, B_DRAIN = B_UNIT_DONE + 1, kBars = B_DRAIN + 1 };

// Tensor memory: per S buffer one 16-column partial S^T per 64-dim panel of
// Dk (separate accumulator chains, summed by the softmax), then two O^T
// accumulators of 32 columns (even / odd 16-slot steps of P.V).
template <int DK>
struct GtTmem {
    static constexpr int sBuf = (DK / 64) * kN;
    static constexpr int o0 = 2 * sBuf, o1 = o0 + 2 * kN;
    static constexpr int used = o1 + 2 * kN;
    static constexpr int cols = used <= 128 ? 128 : 256;
};

template <int DK, bool VK>
struct GtSmem {
    static constexpr int panel = kChunk * 128;            // 128 rows x 128 B (64 dims)
    static constexpr int kPanels = DK / 64;
    static constexpr int vPanels = VK ? 0 : kDv / 64;
    static constexpr int qPanel = kN * 128;               // 16 rows x 128 B
    static constexpr int vOff = kPanels * panel;
    static constexpr int qOff = vOff + vPanels * panel;
    static constexpr int stage = qOff + kPanels * qPanel;
    static constexpr int pPanel = 2 * kN * 128;           // 32 rows (hi heads, lo heads) x 128 B
    static constexpr int pBuf = 2 * pPanel;               // 128 slots = 2 panels of 64
    static constexpr int fixedBytes = 2 * pBuf + 2 * 4 * kN * 4 + 4 * kN * 4 + kMaxStages * 16 + kBars * 8 + 16;
    static constexpr int stages_fit = (232448 - 1024 - fixedBytes) / stage;
    static constexpr int NS = stages_fit > kMaxStages ? kMaxStages : stages_fit;
    static constexpr int p = NS * stage;                  // two P buffers
    static constexpr int red = p + 2 * pBuf;              // [2][4 warps][16] chunk maxima
    static constexpr int redl = red + 2 * 4 * kN * 4;     // [4 warps][16] sums
    static constexpr int meta = redl + 4 * kN * 4;        // [stage][4 warps] visibility masks
    static constexpr int bars = meta + kMaxStages * 16;
    static constexpr int misc = bars + kBars * 8;         // tmem base, abort flag
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;
    static_assert(NS >= 2, "two stages fit");
    static_assert(alloc <= 232448, "dynamic shared memory per block");
    static_assert(stage % 1024 == 0 && p % 1024 == 0, "swizzle atoms stay aligned");
};


struct GtSched {
    int64_t units;   // index lists
    int cpu;         // chunks per list
    int ctas;
};

struct UnitCoord {
    int b, n2, s1;
};
__device__ __forceinline__ UnitCoord unit_coord(int64_t u, const SfaParams& p) {
    UnitCoord c;
    c.s1 = (int)(u % p.S1);
    c.n2 = (int)((u / p.S1) % p.N2);
    c.b = (int)(u / ((int64_t)p.S1 * p.N2));
    return c;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Reduce-scatter of GP per-lane values over the warp: afterwards lane l
// holds the reduction over all 32 lanes of value head_of(l) (max or sum).
template <int GP, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[GP], int lane) {
    int n = GP;
    int off = 16;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        if (n > 1) {
            const int half = n / 2;
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int j = 0; j < GP / 2; ++j) {
                if (j < half) {
                    const float send = up ? v[j] : v[j + half];
                    const float keep = up ? v[j + half] : v[j];
                    const float got = __shfl_xor_sync(0xffffffffu, send, off);
                    v[j] = MAX ? fmaxf(keep, got) : keep + got;
                }
            }
            n = half;
        } else {
            const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
            v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
        }
        off >>= 1;
    }
    return v[0];
}
// The value index lane l holds after warp_reduce_scatter<GP>.
template <int GP>
__device__ __forceinline__ int head_of(int lane) {
    int h = 0, n = GP, off = 16;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        if (n > 1) {
            n /= 2;
            if (lane & off) h += n;
        }
        off >>= 1;
    }
    return h;
}

template <class E, int DK, bool VK, int GP>
__global__ void __launch_bounds__(kThreads, 1) sfa_group_tc_kernel(const SfaParams p, const GtSched sch) {
    using T = typename E::T;
    using L = GtSmem<DK, VK>;
    using TM = GtTmem<DK>;
    constexpr int NS = L::NS;
    constexpr int KP = DK / 64;
    constexpr bool kBf16 = std::is_same<E, BF16>::value;
    constexpr uint32_t kIdescQK = idesc_f16(kChunk, kN, kBf16, false, false);
    constexpr uint32_t kIdescPV = idesc_f16(kDv, 2 * kN, kBf16, true, false);
    static_assert(GP == 16, "padded group");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cpu = sch.cpu;
    const int64_t u_begin = (int64_t)blockIdx.x * sch.units / sch.ctas;
    const int64_t u_end = ((int64_t)blockIdx.x + 1) * sch.units / sch.ctas;
    const int n = (int)((u_end - u_begin) * cpu);            // chunks of this CTA (host-checked)
    const int64_t c0 = u_begin * cpu;                          // first global chunk
    auto bar = [&](int i) { return sbase + L::bars + 8 * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc + 4);
    const int G = p.G;

    // zero the Q panels of every stage (rows >= G are never copied) and the
    // P buffers (rows of heads >= G are never written)
    for (int s = 0; s < NS; ++s) {
        uint4* qz = reinterpret_cast<uint4*>(smem + s * L::stage + L::qOff);
        for (int e = tid; e < L::kPanels * L::qPanel / 16; e += kThreads) qz[e] = make_uint4(0, 0, 0, 0);
    }
    for (int e = tid; e < 2 * L::pBuf / 16; e += kThreads)
        reinterpret_cast<uint4*>(smem + L::p)[e] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B_KV_FULL + s), kProdThreads + kProdThreads / 32);
            mbar_init(bar(B_KV_FREE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_FULL + b), kSoftThreads);
            mbar_init(bar(B_P_FREE + b), 1);
            mbar_init(bar(B_O_DONE + b), 1);
        }
        mbar_init(bar(B_UNIT_DONE), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();     // the zero fill above precedes tensor-core reads
    // launched with programmatic dependent launch: nothing above touches
    // global memory
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == kMmaWarp) tmem_alloc(sbase + L::misc, TM::cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::misc);

    if (warp >= kProdWarp0) {
        // ============================ producers ============================
        // Warp pw gathers slots 32 pw .. 32 pw + 31 of every chunk, four rows
        // per step: lane l copies 16-byte piece (l % 8) + 8 j of row l / 8,
        // which lands in chunk (l % 8) ^ (row % 8) of the row's line of panel j.
        const int pw = warp - kProdWarp0;
        const int rg = lane >> 3, pl = lane & 7;
        struct Cursor {
            int cc;
            UnitCoord uc;
        };
        auto cursor_at = [&](int64_t u) {
            Cursor k;
            k.cc = 0;
            k.uc = unit_coord(u, p);
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
        };
        Cursor fk = cursor_at(u_begin), k = cursor_at(u_begin);
        int fc = 0;
        auto fetch = [&]() {
            int id = kNoSlot;
            if (fc < n) {
                const int32_t* ig = p.idx + fk.uc.b * p.i_sb + fk.uc.n2 * p.i_sh + fk.uc.s1 * p.i_ss;
                const int j = fk.cc * kChunk + 32 * pw + lane;
                if (j < p.topK) id = ig[j];
                advance(fk);
                ++fc;
            }
            return id;
        };
        int ring[kLookahead];
#pragma unroll
        for (int r = 0; r < kLookahead; ++r) ring[r] = fetch();
        // stage s's visibility mask and arrivals: every producer thread
        // arrives, lane 0 after writing its warp's mask
        auto release = [&](int s, uint32_t m) {
            if (lane == 0) reinterpret_cast<uint32_t*>(smem + L::meta)[4 * s + pw] = m;
            __syncwarp();
            mbar_arrive(bar(B_KV_FULL + s));
            if (lane == 0) mbar_arrive(bar(B_KV_FULL + s));
        };
        uint32_t prev_mask = 0;
        int released = -1;                  // last chunk whose copies were issued
        for (int i = 0; i < n; ++i) {
            const int s = i % NS;
            if (!mbar_wait(bar(B_KV_FREE + s), ((i / NS) & 1) ^ 1, p.err_word, abort_flag)) break;
            const int myid = ring[0];
#pragma unroll
            for (int r = 0; r + 1 < kLookahead; ++r) ring[r] = ring[r + 1];
            ring[kLookahead - 1] = fetch();
            const UnitCoord uc = k.uc;
            const int diag = uc.s1 + (p.S2 - p.S1);
            const bool in_range = myid >= 0 && myid < p.S2;
            if (!in_range && myid != kNoSlot && p.validate) atomicOr(p.err_word, kErrIndexRange);
            const bool vis = in_range && !(p.causal && myid > diag);
            const int myrow = in_range ? myid : -1;
            const T* kg = static_cast<const T*>(p.k) + uc.b * p.k_sb + uc.n2 * p.k_sh;
            const T* vg = static_cast<const T*>(p.v) + uc.b * p.v_sb + uc.n2 * p.v_sh;
            unsigned char* st = smem + s * L::stage;
#pragma unroll 2
            for (int it = 0; it < 8; ++it) {
                const int rr = 4 * it + rg;
                const int id = __shfl_sync(0xffffffffu, myrow, rr);
                const int row = 32 * pw + rr;
                const int sw = (pl ^ (row & 7)) << 4;
                const T* krow = kg + (id >= 0 ? (int64_t)id * p.k_ss : 0);
#pragma unroll
                for (int j = 0; j < DK / 64; ++j)
                    cp_async_16_zfill(st + j * L::panel + row * 128 + sw, krow + 8 * (pl + 8 * j),
                                      id >= 0 ? 16 : 0);
                if constexpr (!VK) {
                    const T* vrow = vg + (id >= 0 ? (int64_t)id * p.v_ss : 0);
#pragma unroll
                    for (int j = 0; j < kDv / 64; ++j)
                        cp_async_16_zfill(st + L::vOff + j * L::panel + row * 128 + sw,
                                          vrow + 8 * (pl + 8 * j), id >= 0 ? 16 : 0);
                }
            }
            // the list's q rows, unless this stage already holds them (the
            // stage's previous chunk, NS chunks back, was of the same list)
            const int64_t cg = c0 + i;
            if (i < NS || cg / cpu != (cg - NS) / cpu) {
                const T* qg = static_cast<const T*>(p.q) + uc.b * p.q_sb + uc.s1 * p.q_ss;
                for (int e = pw * 32 + lane; e < G * (DK / 8); e += kProdThreads) {
                    const int h = e / (DK / 8), pc = e % (DK / 8);
                    cp_async_16(st + L::qOff + (pc >> 3) * L::qPanel + (h >> 3) * 1024 + (h & 7) * 128 +
                                    (((pc & 7) ^ (h & 7)) << 4),
                                qg + (int64_t)(uc.n2 * G + h) * p.q_sh + 8 * pc);
                }
            }
            cp_async_commit();
            // The tensor core reads the rows (async proxy): a stage is
            // released once its copies have landed and the thread that made
            // them has fenced them -- one chunk late, so that two chunks'
            // copies stay in flight.
            const uint32_t mask = __ballot_sync(0xffffffffu, vis);
            if (i > 0) {
                cp_async_wait<1>();
                fence_proxy_async_smem();
                release((i - 1) % NS, prev_mask);
            }
            prev_mask = mask;
            advance(k);
            released = i;
        }
        if (released >= 0) {
            // the last chunk issued
            cp_async_wait<0>();
            fence_proxy_async_smem();
            release(released % NS, prev_mask);
        }
        // no copy may still be in flight when the warp leaves
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        // ============================ MMA issue ============================
        if (lane == 0 && n > 0) {
            bool ok = true;
            auto qk = [&](int j) {
                const int s = j % NS;
                tc_fence_after();
                const uint32_t st = sbase + s * L::stage;
                const uint32_t d = tmem + TM::sBuf * (j & 1);
                // one accumulator chain per 64-dim panel, issued interleaved
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        const uint64_t ad = sdesc_sw128(st + q * L::panel + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(st + L::qOff + q * L::qPanel + kk * 32, 16, 1024);
                        tc_mma_f16(d + kN * q, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                tc_commit(bar(B_S_FULL + (j & 1)));
            };
            int next_qk = 0;
            uint64_t idle_since = 0;
            for (int i = 0; i < n && ok;) {
                if (next_qk < n && next_qk <= i) {
                    ok = mbar_wait(bar(B_KV_FULL + next_qk % NS), (next_qk / NS) & 1, p.err_word, abort_flag);
                    if (!ok) break;
                    qk(next_qk++);
                    continue;
                }
                // P.V of chunk i as soon as its P is written (it frees the
                // stage); until then Q.K^T of the next chunk if its rows are in
                if (!mbar_test_wait(bar(B_P_FULL + (i & 1)), (i >> 1) & 1)) {
                    if (next_qk < n && next_qk == i + 1 &&
                        mbar_test_wait(bar(B_KV_FULL + next_qk % NS), (next_qk / NS) & 1)) {
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
                const int s = i % NS;
                tc_fence_after();
                // O^T += V^T [P_hi^T | P_lo^T]: V^T an MN-major operand (the
                // V panels of the chunk's rows: K's first two when V is its
                // prefix), P K-major from its buffer
                const uint32_t vb = sbase + s * L::stage + (VK ? 0 : L::vOff);
                const uint32_t pb = sbase + L::p + (i & 1) * L::pBuf;
                const bool first = (c0 + i) % cpu == 0;
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk) {
                    const uint64_t ad = sdesc_sw128(vb + kk * 16 * 128, L::panel, 1024);
                    const uint64_t bd = sdesc_sw128(pb + (kk >> 2) * L::pPanel + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16(tmem + ((kk & 1) ? TM::o1 : TM::o0), ad, bd, kIdescPV,
                               (first && kk < 2) ? 0u : 1u);
                }
                tc_commit(bar(B_KV_FREE + s));
                tc_commit(bar(B_P_FREE + (i & 1)));
                tc_commit(bar(B_O_DONE + (i & 1)));
                ++i;
                if ((c0 + i) % cpu == 0) tc_commit(bar(B_UNIT_DONE));   // the list's O is final
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
        const int t = tid;                                   // slot t / output dim t = TMEM lane t
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        float* red = reinterpret_cast<float*>(smem + L::red);     // [2][4][16]
        float* redl = reinterpret_cast<float*>(smem + L::redl);   // [4][16]
        const int my_head = head_of<GP>(lane);
        float m_used[GP], l[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m_used[h] = -INFINITY;
            l[h] = 0.f;
        }
        // P element (row r of the operand, slot t) in a P buffer
        const uint32_t p_slot = (uint32_t)((t >> 6) * L::pPanel) + (uint32_t)((t & 7) * 2);
        const int p_chunk = (t & 63) >> 3;
        uint32_t unit_phase = 0;
        for (int i = 0; i < n; ++i) {
            const int s = i % NS, b = i & 1;
            const int64_t cg = c0 + i;
            const bool first_of_unit = cg % cpu == 0;
            const bool last_of_unit = (cg + 1) % cpu == 0;
            mbar_wait(bar(B_KV_FULL + s), (i / NS) & 1, p.err_word, abort_flag);
            const uint32_t vm = reinterpret_cast<const uint32_t*>(smem + L::meta)[4 * s + warp];
            const bool vis = (vm >> lane) & 1u;
            mbar_wait(bar(B_S_FULL + b), (i >> 1) & 1, p.err_word, abort_flag);
            tc_fence_after();
            uint32_t sv[KP * kN];
            {
                const uint32_t sa = lane_base + TM::sBuf * b;
                if constexpr (KP == 2) tmem_ld32_sync(sa, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                if constexpr (KP == 3) tmem_ld48_sync(sa, *reinterpret_cast<uint32_t(*)[48]>(&sv[0]));
                if constexpr (KP == 4) tmem_ld64_sync(sa, *reinterpret_cast<uint32_t(*)[64]>(&sv[0]));
            }
            float x[GP], cm[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                float acc = __uint_as_float(sv[h]);
#pragma unroll
                for (int q = 1; q < KP; ++q) acc += __uint_as_float(sv[kN * q + h]);
                x[h] = (vis && h < G) ? acc * p.scale_log2 : -INFINITY;
                cm[h] = x[h];
            }
            // the chunk's maximum of every head over the 128 slots
            const float wm = warp_reduce_scatter<GP, true>(cm, lane);
            float* rb = red + (i & 1) * 4 * kN;
            if ((lane & (32 / GP - 1)) == 0) rb[warp * kN + my_head] = wm;
            named_sync(1, kSoftThreads);
            bool any = false;
            float f[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float c = fmaxf(fmaxf(rb[h], rb[kN + h]), fmaxf(rb[2 * kN + h], rb[3 * kN + h]));
                const float m_new = fmaxf(m_used[h], c);
                const bool need = m_new > m_used[h] + kRescaleThreshold;
                f[h] = need ? fast_exp2(m_used[h] - m_new) : 1.f;   // 0 while m_used is -inf
                if (need) m_used[h] = m_new;
                any |= need;
            }
            float pv[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                pv[h] = (x[h] == -INFINITY) ? 0.f : fast_exp2(x[h] - m_used[h]);
                l[h] = l[h] * f[h] + pv[h];
            }
            if (any && !first_of_unit) {
                // O is rescaled once P.V of the previous chunk is done
                const int pbf = (i - 1) & 1;
                mbar_wait(bar(B_O_DONE + pbf), ((i - 1) >> 1) & 1, p.err_word, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    uint32_t ov[32];
                    const uint32_t oa = lane_base + (a ? TM::o1 : TM::o0);
                    tmem_ld32_sync(oa, ov);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        ov[c] = __float_as_uint(__uint_as_float(ov[c]) * ((c & 15) < GP ? f[(c & 15) % GP] : 1.f));
                    tmem_st32(oa, ov);
                }
                tmem_wait_st();
            }
            // P of this chunk into buffer b, once P.V of chunk i - 2 has read it
            if (i >= 2) mbar_wait(bar(B_P_FREE + b), ((i - 2) >> 1) & 1, p.err_word, abort_flag);
            const uint32_t pbase = sbase + L::p + b * L::pBuf + p_slot;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h < G) {
                    const uint32_t hw = E::pack2(pv[h], 0.f);
                    const float hi = E::unpack2(hw).x;
                    const uint32_t lw = E::pack2(pv[h] - hi, 0.f);
                    const int rh = h, rl = kN + h;
                    st_shared_u16(pbase + (rh >> 3) * 1024 + (rh & 7) * 128 + ((p_chunk ^ (rh & 7)) << 4),
                                  (uint16_t)(hw & 0xffffu));
                    st_shared_u16(pbase + (rl >> 3) * 1024 + (rl & 7) * 128 + ((p_chunk ^ (rl & 7)) << 4),
                                  (uint16_t)(lw & 0xffffu));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + b));
            if (!last_of_unit) continue;

            // ---- epilogue of the list: thread t = output dim t ----
            mbar_wait(bar(B_UNIT_DONE), unit_phase, p.err_word, abort_flag);
            unit_phase ^= 1;
            tc_fence_after();
            float ls[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) ls[h] = l[h];
            const float wl = warp_reduce_scatter<GP, false>(ls, lane);
            if ((lane & (32 / GP - 1)) == 0) redl[warp * kN + my_head] = wl;
            uint32_t ov[32], ow[32];
            tmem_ld32_sync(lane_base + TM::o0, ov);
            tmem_ld32_sync(lane_base + TM::o1, ow);
            tc_fence_before();
            named_sync(1, kSoftThreads);
            const int64_t u = cg / cpu;
            const UnitCoord uc = unit_coord(u, p);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h < G) {
                    const float Ls = (redl[h] + redl[kN + h]) + (redl[2 * kN + h] + redl[3 * kN + h]);
                    const bool empty = !(Ls > 0.f);
                    const float o = (__uint_as_float(ov[h]) + __uint_as_float(ov[kN + h])) +
                                    (__uint_as_float(ow[h]) + __uint_as_float(ow[kN + h]));
                    const int n1 = uc.n2 * G + h;
                    T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss;
                    const uint32_t w = E::pack2(empty ? 0.f : o / Ls, 0.f);
                    reinterpret_cast<uint16_t*>(orow)[t] = (uint16_t)(w & 0xffffu);
                    if (t == h && p.lse)
                        p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] =
                            empty ? -INFINITY : (m_used[h] + __log2f(Ls)) * kLn2;
                }
            }
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                m_used[h] = -INFINITY;
                l[h] = 0.f;
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TM::cols);
    }
}

template <class E, int DK, bool VK, int GP>
cudaError_t run_t(const SfaParams& p, int num_sms, cudaStream_t stream) {
    using L = GtSmem<DK, VK>;
    auto kern = sfa_group_tc_kernel<E, DK, VK, GP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
    if (err != cudaSuccess) return err;
    GtSched s;
    s.cpu = (p.topK + kChunk - 1) / kChunk;
    s.units = (int64_t)p.B * p.N2 * p.S1;
    int64_t ctas = p.num_ctas > 0 ? p.num_ctas : num_sms;
    if (ctas > s.units) ctas = s.units;
    s.ctas = (int)ctas;
    if ((s.units + ctas - 1) / ctas * s.cpu >= (int64_t(1) << 30)) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(s.ctas), dim3(kThreads), (size_t)L::alloc, stream, p, s);
}

template <class E, int DK, bool VK>
cudaError_t run_g(const SfaParams& p, int num_sms, cudaStream_t stream) {
    return run_t<E, DK, VK, kN>(p, num_sms, stream);
}

template <class E>
cudaError_t run_e(const SfaParams& p, bool vk, int num_sms, cudaStream_t stream) {
    switch (p.Dk) {
        case 128: return vk ? run_g<E, 128, true>(p, num_sms, stream) : run_g<E, 128, false>(p, num_sms, stream);
        case 192: return vk ? run_g<E, 192, true>(p, num_sms, stream) : run_g<E, 192, false>(p, num_sms, stream);
        case 256: return vk ? run_g<E, 256, true>(p, num_sms, stream) : run_g<E, 256, false>(p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool group_tc_supported(const SfaParams& p, int num_sms) {
    const int64_t units = (int64_t)p.B * p.N2 * p.S1;
    const int64_t cpu = (p.topK + kChunk - 1) / kChunk;
    // at least four whole index lists per CTA of a one-per-SM grid (fewer
    // lists go to the stream-K decode kernel, which can split them)
    const int64_t ctas = p.num_ctas > 0 ? p.num_ctas : num_sms;
    const bool many = units >= 4 * ctas;
    return p.G > 8 && p.G <= kN && p.Dv == kDv && (p.Dk == 128 || p.Dk == 192 || p.Dk == 256) &&
           many && (units + ctas - 1) / ctas * cpu < (int64_t(1) << 30);
}

cudaError_t launch_sfa_group_tc(const SfaParams& p, sfa_dtype dtype, int num_sms, cudaStream_t stream) {
    if (!group_tc_supported(p, num_sms)) return cudaErrorInvalidValue;
    // value rows are the key rows' prefix when v aliases k
    const bool vk = (p.v == p.k) && (p.v_ss == p.k_ss);
    cudaError_t err = dtype == SFA_DTYPE_BF16 ? run_e<BF16>(p, vk, num_sms, stream)
                                              : run_e<F16>(p, vk, num_sms, stream);
    count_launches(1);
    return err;
}

}  // namespace sfa
