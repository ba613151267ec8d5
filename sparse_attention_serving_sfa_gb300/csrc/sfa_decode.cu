// Top-K sparse attention for small GQA groups (G <= 8 query heads share one
// index list): the decode / prefill gather path.
//
// "SparseFlashAttention 算子 API 描述", §2 具体子步骤 (sparse gather, scaled dot
// product, bottom-right causal mask, softmax over the selected slots,
// weighted sum), with the softmax evaluated online over 64-slot chunks.
//
// Each selected slot costs (Dk [+ Dv]) * 2 gathered bytes and only
// 2 * G * (Dk + Dv) FLOPs, so the kernel is built around the gather:
//   - persistent grid (SM count x CTAs per SM) over the flat sequence of
//     (index list, 64-slot chunk) pairs, split into equal contiguous ranges
//     (stream-K): every SM streams the same number of bytes, no tail waves;
//   - two producer warps gather each chunk's K rows (and V rows, unless V is
//     the key prefix view), plus the group's q rows at the first chunk of an
//     index list, with 16-byte cp.async, eight lanes per row and four rows
//     per step (coalesced), into padded rows of a ring of shared-memory
//     stages (as many as fit two CTAs per SM); completion is tracked by
//     mbarriers (cp.async.mbarrier.arrive), indices are prefetched eight
//     chunks ahead, slots past topK or with an out-of-range index are
//     zero-filled and masked.  (Per-row bulk TMA copies were measured at ~85 cycles per
//     256-byte row per SM -- about 0.9 TB/s over the GPU -- too slow for
//     row gathers.)
//   - four consumer warps each own 16 slots of every chunk and keep their own
//     online-softmax state: the two small contractions, S^T = K Q^T
//     ([16 slots x Dk] x [Dk x 8 heads], heads past G zero) and
//     O^T += V^T P^T ([Dv x 16 slots] x [16 x 8]), run as warp-level mma.sync
//     (bf16/fp16 in, fp32 accumulate), operands fetched with ldmatrix, P kept
//     in registers between the two
//     (as a 16-bit high part plus a 16-bit remainder, two MMAs);
//     this keeps the instruction count per gathered byte low enough for the
//     gather to set the pace;
//   - at the end of an index list the four warps' states are merged through
//     the K / V tiles of the stage holding its last chunk (released after
//     the merge); a range that holds the whole list writes the output,
//     otherwise its partial (O, running max, sum) goes to the workspace and
//     the last CTA to finish the list (a per-list arrival counter in the
//     workspace head, reset by that CTA) merges the L2-resident partials and
//     writes the output -- one launch, no separate combine kernel;
//   - with fewer index lists than resident CTAs, every list is split into
//     the same number (2..8) of segments and a list's segments run as one
//     thread-block cluster: each CTA leaves its partial in its own shared
//     memory and the cluster's first CTA merges them over distributed shared
//     memory (two cluster barriers instead of a fence, an atomic and a round
//     trip through L2).
#include <limits.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sfa {
namespace {

constexpr int kChunk = 64;                    // slots per stage
constexpr int kConsWarps = 4;                 // each owns 16 slots of a chunk
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kProdWarps = 2;                 // each gathers 32 slots of a chunk
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kThreads = kConsThreads + kProdThreads;
constexpr int kNoSlot = INT_MIN;              // marks a slot past topK
constexpr int kRowPad = 16;                   // bytes of padding per smem row
constexpr int kHeads = 8;                     // G <= 8: the N = 8 side of the MMAs
constexpr int kLookahead = 8;                 // chunks of indices prefetched
constexpr int kMaxCluster = 8;                // portable cluster size

// Chunk ranges of the persistent CTAs.  Stream-K: equal contiguous ranges of
// the flat chunk sequence (an index list may be split across CTAs, which then
// merge through the workspace).  Aligned: each CTA takes whole index lists
// (used when there are many more lists than CTAs; nothing to merge).
struct DecodeSched {
    int64_t total;   // chunks over all index lists
    int64_t units;   // index lists
    int cpu;         // chunks per index list
    int ctas;        // grid size
    int seg_max;     // most CTAs sharing one index list
    int aligned;     // 1: ranges hold whole index lists
    int cluster;     // >= 2: list u is split into `cluster` segments, run by the
                     // thread-block cluster u (CTAs cluster * u + rank)
};

__host__ __device__ inline int64_t range_begin(int64_t c, const DecodeSched& s) {
    if (s.cluster > 1) {
        const int64_t u = c / s.cluster, j = c - u * s.cluster;
        return u * s.cpu + (j * s.cpu) / s.cluster;
    }
    return s.aligned ? (c * s.units / s.ctas) * s.cpu : c * s.total / s.ctas;
}
// CTA whose range holds chunk x.
__host__ __device__ inline int64_t cta_of(int64_t x, const DecodeSched& s) {
    if (s.cluster > 1) {
        const int64_t u = x / s.cpu, j = x - u * s.cpu;
        return u * s.cluster + ((j + 1) * s.cluster - 1) / s.cpu;
    }
    return s.aligned ? ((x / s.cpu + 1) * s.ctas - 1) / s.units : ((x + 1) * s.ctas - 1) / s.total;
}

template <int DK, int DV, bool VK, int NS>
struct Smem {
    static constexpr int ks = DK * 2 + kRowPad;          // K row stride (bytes)
    static constexpr int vs = VK ? ks : DV * 2 + kRowPad;
    static constexpr int kTile = kChunk * ks;
    static constexpr int vTile = VK ? 0 : kChunk * vs;
    static constexpr int qTile = kHeads * ks;            // 8 rows, rows >= G stay zero
    static constexpr int stage = kTile + vTile + qTile;
    static constexpr int meta = NS * stage;              // NS x int4 {-, mask lo, mask hi, -}
    static constexpr int bars = meta + NS * 16;          // full[NS], empty[NS]
    static constexpr int ml = bars + 2 * NS * 8;         // [4 warps][8 rows] float2 (m, l)
    static constexpr int abort = ml + kConsWarps * kHeads * 8;
    static constexpr int total = abort + 16;
    // the 4 warps' O states of a list ([4][8][DV] float) go to the K / V
    // tiles of a stage the consumers hold (its q rows are left alone)
    static constexpr int obufBytes = kConsWarps * kHeads * DV * 4;
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

// Position in the flat chunk sequence, advanced without divisions:
// index list u = (b * N2 + n2) * S1 + s1, chunk cc of that list.
struct Cursor {
    int64_t u;
    int cc;
    UnitCoord uc;
};
__device__ __forceinline__ Cursor cursor_at(int64_t c, int cpu, const SfaParams& p) {
    Cursor k;
    k.u = c / cpu;
    k.cc = (int)(c - k.u * cpu);
    k.uc = unit_coord(k.u, p);
    return k;
}
__device__ __forceinline__ void advance(Cursor& k, int cpu, const SfaParams& p) {
    if (++k.cc == cpu) {
        k.cc = 0;
        ++k.u;
        if (++k.uc.s1 == p.S1) {
            k.uc.s1 = 0;
            if (++k.uc.n2 == p.N2) {
                k.uc.n2 = 0;
                ++k.uc.b;
            }
        }
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// D(16x8, fp32) += A(16x16, row-major) * B(16x8, column-major), 16-bit
// inputs (bf16 or fp16 as E), fp32 accumulate.
template <class E>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (std::is_same<E, BF16>::value) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Low 16 bits of x when `hi` is false, else the high 16 bits, in the low half.
__device__ __forceinline__ uint32_t half_of(uint32_t x, bool hi) { return hi ? (x >> 16) : (x & 0xffffu); }

template <class E, int DK, int DV, bool VK, int NS>
__global__ void __launch_bounds__(kThreads) sfa_decode_kernel(const SfaParams p, const DecodeSched sch) {
    using T = typename E::T;
    using L = Smem<DK, DV, VK, NS>;
    constexpr int KT = DK / 16;      // k-steps of Q.K^T
    constexpr int NT = DV / 8;       // n-tiles of P.V
    static_assert(KT % 2 == 0 && NT % 2 == 0, "head dims must be multiples of 32 and 16");
    static_assert(kHeads * DV * 4 + kHeads * 8 <= L::kTile + L::vTile, "a cluster merge partial fits a stage");
    static_assert(L::obufBytes <= L::kTile + L::vTile, "the merge buffer fits a stage's K / V tiles");
    static_assert(NS >= 2, "the cluster merge uses two stages");

    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t smem_base = smem_u32(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c_begin = range_begin(blockIdx.x, sch);
    const int64_t c_end = range_begin((int64_t)blockIdx.x + 1, sch);
    const uint32_t full0 = smem_base + L::bars, empty0 = full0 + NS * 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::abort);
    volatile int* last_flag = abort_flag + 1;     // this CTA merges the list
    const int G = p.G;

    // zero the q tiles (rows >= G are never copied) and set up the barriers
    for (int s = 0; s < NS; ++s) {
        uint4* qt = reinterpret_cast<uint4*>(smem + s * L::stage + L::kTile + L::vTile);
        for (int e = tid; e < L::qTile / 16; e += kThreads) qt[e] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            // full: one cp.async arrival per producer thread + one plain
            // arrival per producer warp after it wrote its half of the mask
            mbar_init(full0 + 8 * s, kProdThreads + kProdWarps);
            mbar_init(empty0 + 8 * s, kConsWarps);
        }
        fence_barrier_init();
    }
    fence_proxy_async_smem();    // zero fill above precedes later bulk copies
    // launched with programmatic dependent launch: nothing above touches
    // global memory; wait here for the previous grid in the stream (its
    // writes are then visible), and let the next one start launching.  When
    // the caller states that the inputs were ready before that grid, the wait
    // moves to the merge, before this kernel's first global write (out, lse,
    // workspace); until then it only reads q, k, v and the indices (and may
    // set bits of the error word, an atomic OR).
    if (!p.inputs_ready) grid_dependency_wait();
    grid_launch_dependents();
    __syncthreads();

    if (warp >= kConsWarps) {
        // ======================= producer warps =======================
        // warp pw gathers slots 32 pw .. 32 pw + 31 of every chunk, four rows
        // per step: lane l copies 16-byte pieces l % 8, l % 8 + 8, ... of
        // row l / 8 of the step (every lane busy whatever the row length).
        const int pw = warp - kConsWarps;
        const int cpu = sch.cpu;
        const int quarter = lane >> 3, ql = lane & 7;
        Cursor fk = cursor_at(c_begin, cpu, p);     // index prefetch cursor
        int64_t fc = c_begin;
        auto fetch = [&]() {
            int id = kNoSlot;
            if (fc < c_end) {
                const int32_t* ig =
                    p.idx + fk.uc.b * p.i_sb + fk.uc.n2 * p.i_sh + fk.uc.s1 * p.i_ss;
                const int j = fk.cc * kChunk + 32 * pw + lane;
                if (j < p.topK) id = ig[j];
                advance(fk, cpu, p);
                ++fc;
            }
            return id;
        };
        // indices run kLookahead chunks ahead of the gathers: under a full
        // gather load their latency is several microseconds
        int qring[kLookahead];
#pragma unroll
        for (int r = 0; r < kLookahead; ++r) qring[r] = fetch();
        Cursor k = cursor_at(c_begin, cpu, p);
        int64_t i = 0;
        for (int64_t c = c_begin; c < c_end; ++c, ++i) {
            const int s = (int)(i % NS);
            const uint32_t round = (uint32_t)(i / NS);
            if (!mbar_wait(empty0 + 8 * s, (round & 1u) ^ 1u, p.err_word, abort_flag)) break;
            const int myid = qring[0];
#pragma unroll
            for (int r = 0; r + 1 < kLookahead; ++r) qring[r] = qring[r + 1];
            qring[kLookahead - 1] = fetch();

            const UnitCoord uc = k.uc;
            const int diag = uc.s1 + (p.S2 - p.S1);
            const bool in_range = myid >= 0 && myid < p.S2;
            if (!in_range && myid != kNoSlot && p.validate) atomicOr(p.err_word, kErrIndexRange);
            const bool vis = in_range && !(p.causal && myid > diag);
            const T* kg = static_cast<const T*>(p.k) + uc.b * p.k_sb + uc.n2 * p.k_sh;
            const T* vg = static_cast<const T*>(p.v) + uc.b * p.v_sb + uc.n2 * p.v_sh;
            unsigned char* st = smem + s * L::stage;
#pragma unroll 4
            for (int r = 0; r < 32; r += 4) {
                const int src_lane = r + quarter;
                const int id = __shfl_sync(0xffffffffu, myid, src_lane);
                const bool ok = id >= 0 && id < p.S2;
                const int j = 32 * pw + src_lane;
                const T* krow = kg + (ok ? (int64_t)id * p.k_ss : 0);
#pragma unroll
                for (int pc = ql; pc < DK / 8; pc += 8)
                    cp_async_16_zfill(st + j * L::ks + pc * 16, krow + pc * 8, ok ? 16 : 0);
                if constexpr (!VK) {
                    const T* vrow = vg + (ok ? (int64_t)id * p.v_ss : 0);
#pragma unroll
                    for (int pc = ql; pc < DV / 8; pc += 8)
                        cp_async_16_zfill(st + L::kTile + j * L::vs + pc * 16, vrow + pc * 8, ok ? 16 : 0);
                }
            }
            // the group's q rows (piece e of G * Dk / 8), only into the stage
            // of an index list's first chunk in this range: the consumers
            // read q from that stage alone
            if (k.cc == 0 || c == c_begin) {
                const T* qg = static_cast<const T*>(p.q) + uc.b * p.q_sb + uc.s1 * p.q_ss;
                for (int e = pw * 32 + lane; e < G * (DK / 8); e += kProdThreads) {
                    const int h = e / (DK / 8), pc = e % (DK / 8);
                    cp_async_16(st + L::kTile + L::vTile + h * L::ks + pc * 16,
                                qg + (int64_t)(uc.n2 * G + h) * p.q_sh + pc * 8);
                }
            }
            cp_async_mbar_arrive(full0 + 8 * s);
            const uint32_t mask = __ballot_sync(0xffffffffu, vis);
            if (lane == 0) {
                reinterpret_cast<uint32_t*>(smem + L::meta)[4 * s + 1 + pw] = mask;
                mbar_arrive(full0 + 8 * s);
            }
            advance(k, cpu, p);
        }
        // no copy may still be in flight when the warp leaves
        cp_async_wait<0>();
        if (sch.cluster > 1) {
            // the consumers' two cluster barriers of the merge count every
            // thread of the cluster that has not exited: take part in both
            __syncwarp();
            cluster_sync();
            cluster_sync();
        }
        return;
    }

    // ======================= consumer warps =======================
    // Warp w owns slots 16 w .. 16 w + 15 of every chunk.  Both contractions
    // put the 16 slots (or 16 output dims) on the MMA's M side and the <= 8
    // query heads on its N = 8 side:
    //   S^T [16 slots x 8 heads]  = K_w [16 x Dk] . Q^T [Dk x 8]
    //   O^T [Dv x 8 heads]       += V_w^T [Dv x 16 slots] . P^T [16 x 8]
    // Lane l holds heads hc = 2 (l % 4) + {0, 1} of rows l / 4 and l / 4 + 8.
    const int quad = lane & 3, rq = lane >> 2;
    const int hc = 2 * quad;
    float2* ml_buf = reinterpret_cast<float2*>(smem + L::ml);
    constexpr int MT = DV / 16;          // m-tiles of O^T

    float o[MT][4];                      // O^T[16 mt + rq (+8)][hc (+1)]
    float m_run[2], l_part[2];
    uint32_t qb[KT][2];                  // Q^T B-fragments of the current index list
    int64_t cur = -1;

    // Merge of the 4 warps' states of index list `u`, then either the final
    // output (this CTA holds all of the list's chunks) or a partial.  Called
    // after the P.V of the list's last chunk in this range, whose stage `s`
    // the consumers still hold: the warps' O states go to its K / V tiles
    // (at the end of a clustered range, when every stage is idle, to stage 1:
    // stage 0 takes the partial the cluster reads).
    auto flush = [&](int64_t u, int s) {
        float* obuf = reinterpret_cast<float*>(smem + (sch.cluster > 1 ? 1 : s) * L::stage);
        if (p.inputs_ready) grid_dependency_wait();   // (returns at once after the first time)
        named_sync(1, kConsThreads);        // every warp is done with the stage's rows
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float l = l_part[e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            if (rq == 0) ml_buf[warp * kHeads + hc + e] = make_float2(m_run[e], l);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                obuf[(warp * kHeads + hc + (e & 1)) * DV + 16 * mt + rq + 8 * (e >> 1)] = o[mt][e];
        named_sync(1, kConsThreads);
        const UnitCoord uc = unit_coord(u, p);
        auto write_out = [&](int g, int d2, float M, float Ls, float ax, float ay) {
            const int n1 = uc.n2 * G + g;
            T* orow = static_cast<T*>(p.out) + uc.b * p.o_sb + n1 * p.o_sh + uc.s1 * p.o_ss;
            const bool empty = !(Ls > 0.f);
            const float inv = empty ? 0.f : 1.f / Ls;
            reinterpret_cast<uint32_t*>(orow)[d2] = empty ? 0u : E::pack2(ax * inv, ay * inv);
            if (p.lse && d2 == 0)
                p.lse[uc.b * p.l_sb + n1 * p.l_sh + uc.s1 * p.l_ss] =
                    empty ? -INFINITY : (M + __log2f(Ls)) * kLn2;
        };
        if (sch.cluster > 1) {
            // This CTA's state of the list (over its 4 warps) goes to its own
            // stage area, idle now: every chunk of the range is consumed and
            // no copy is in flight.  [G][DV] O, then [G] (max, sum).
            float* part_o = reinterpret_cast<float*>(smem);
            float2* part_ml = reinterpret_cast<float2*>(smem + kHeads * DV * 4);
            for (int e = tid; e < G * (DV / 2); e += kConsThreads) {
                const int g = e / (DV / 2), d2 = e % (DV / 2);
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) M = fmaxf(M, ml_buf[w * kHeads + g].x);
                float Ls = 0.f, ax = 0.f, ay = 0.f;
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) {
                    const float2 ml = ml_buf[w * kHeads + g];
                    const float f = rescale_factor(ml.x, M);
                    const float2 ov = *reinterpret_cast<const float2*>(obuf + (w * kHeads + g) * DV + 2 * d2);
                    Ls += f * ml.y;
                    ax += f * ov.x;
                    ay += f * ov.y;
                }
                reinterpret_cast<float2*>(part_o + g * DV)[d2] = make_float2(ax, ay);
                if (d2 == 0) part_ml[g] = make_float2(M, Ls);
            }
            // every CTA's partial is visible to the whole cluster ...
            cluster_sync();
            if (cluster_ctarank() == 0) {
                // ... and the first CTA merges them, reading the others'
                // shared memory (all loads issued before any use)
                const int ncl = sch.cluster;
                for (int e = tid; e < G * (DV / 2); e += kConsThreads) {
                    const int g = e / (DV / 2), d2 = e % (DV / 2);
                    const uint32_t a_ml = smem_u32(part_ml + g);
                    const uint32_t a_o = smem_u32(part_o + g * DV + 2 * d2);
                    float2 mv[kMaxCluster], ov[kMaxCluster];
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) {
                        mv[r] = make_float2(-INFINITY, 0.f);
                        ov[r] = make_float2(0.f, 0.f);
                        if (r < ncl) {
                            mv[r] = ld_cluster_f2(map_peer(a_ml, (uint32_t)r));
                            ov[r] = ld_cluster_f2(map_peer(a_o, (uint32_t)r));
                        }
                    }
                    float M = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) M = fmaxf(M, mv[r].x);
                    float Ls = 0.f, ax = 0.f, ay = 0.f;
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) {
                        const float f = rescale_factor(mv[r].x, M);
                        Ls += f * mv[r].y;
                        ax += f * ov[r].x;
                        ay += f * ov[r].y;
                    }
                    write_out(g, d2, M, Ls, ax, ay);
                }
            }
            // no CTA leaves while the first one may still read its memory
            cluster_sync();
            return;
        }
        const int64_t first = u * sch.cpu, last = first + sch.cpu - 1;
        const int64_t c_lo = cta_of(first, sch), c_hi = cta_of(last, sch);
        const int nseg = (int)(c_hi - c_lo + 1);
        for (int e = tid; e < G * (DV / 2); e += kConsThreads) {
            const int g = e / (DV / 2), d2 = e % (DV / 2);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) M = fmaxf(M, ml_buf[w * kHeads + g].x);
            float Ls = 0.f, ax = 0.f, ay = 0.f;
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) {
                const float2 ml = ml_buf[w * kHeads + g];
                const float f = rescale_factor(ml.x, M);
                const float2 ov = *reinterpret_cast<const float2*>(obuf + (w * kHeads + g) * DV + 2 * d2);
                Ls += f * ml.y;
                ax += f * ov.x;
                ay += f * ov.y;
            }
            if (nseg == 1) {
                write_out(g, d2, M, Ls, ax, ay);
            } else {
                const int64_t slot = (u * G + g) * sch.seg_max + (blockIdx.x - c_lo);
                reinterpret_cast<float2*>(p.ws_o + slot * p.Dv)[d2] = make_float2(ax, ay);
                if (d2 == 0) {
                    p.ws_ml[slot * 2] = M;
                    p.ws_ml[slot * 2 + 1] = Ls;
                }
            }
        }
        if (nseg > 1) {
            // publish the partial, count arrivals; the last CTA merges
            __threadfence();
            named_sync(1, kConsThreads);
            if (tid == 0) {
                const unsigned prev = atomicAdd(p.counters + u, 1u);
                *last_flag = (prev == (unsigned)(nseg - 1)) ? 1 : 0;
            }
            named_sync(1, kConsThreads);
            if (*last_flag) {
                __threadfence();
                // all loads of a pair's segments are issued before any use
                constexpr int KB = 8;
                for (int e = tid; e < G * (DV / 2); e += kConsThreads) {
                    const int g = e / (DV / 2), d2 = e % (DV / 2);
                    const int64_t row = u * G + g;
                    const float* ml = p.ws_ml + row * sch.seg_max * 2;
                    const float2* wo = reinterpret_cast<const float2*>(p.ws_o + row * sch.seg_max * p.Dv) + d2;
                    float M = -INFINITY, Ls = 0.f, ax = 0.f, ay = 0.f;
                    for (int k0 = 0; k0 < nseg; k0 += KB) {
                        float2 mv[KB], ov[KB];
#pragma unroll
                        for (int k2 = 0; k2 < KB; ++k2) {
                            const bool ok = k0 + k2 < nseg;
                            mv[k2] = ok ? __ldcg(reinterpret_cast<const float2*>(ml) + k0 + k2)
                                        : make_float2(-INFINITY, 0.f);
                            ov[k2] = ok ? __ldcg(wo + (int64_t)(k0 + k2) * (p.Dv / 2))
                                        : make_float2(0.f, 0.f);
                        }
                        float Mb = M;
#pragma unroll
                        for (int k2 = 0; k2 < KB; ++k2) Mb = fmaxf(Mb, mv[k2].x);
                        const float r = rescale_factor(M, Mb);
                        Ls *= r;
                        ax *= r;
                        ay *= r;
#pragma unroll
                        for (int k2 = 0; k2 < KB; ++k2) {
                            const float f = rescale_factor(mv[k2].x, Mb);
                            Ls += f * mv[k2].y;
                            ax += f * ov[k2].x;
                            ay += f * ov[k2].y;
                        }
                        M = Mb;
                    }
                    write_out(g, d2, M, Ls, ax, ay);
                }
                if (tid == 0) atomicExch(p.counters + u, 0u);   // ready for the next call
            }
        }
        named_sync(1, kConsThreads);
    };

    // per-lane ldmatrix row addresses (bytes, relative to a stage)
    const int mi = lane >> 3, mr = lane & 7;
    // K A-fragments: slot 16 w + mr + 8 (mi & 1), dim block (mi >> 1)
    const uint32_t k_lane = (uint32_t)((16 * warp + mr + 8 * (mi & 1)) * L::ks + (mi >> 1) * 16);
    // Q^T B-fragments: head row mr, dim block mi (two k-steps per x4)
    const uint32_t q_lane = (uint32_t)(L::kTile + L::vTile + mr * L::ks + mi * 16);
    // V^T A-fragments (transposed): slot 16 w + mr + 8 (mi >> 1), dim block (mi & 1)
    const uint32_t v_lane = (uint32_t)((VK ? 0 : L::kTile) + (16 * warp + mr + 8 * (mi >> 1)) * L::vs +
                                       (mi & 1) * 16);
    // sources of the P^T B-fragment: slots 2 quad (+1) hold head rq in lane
    // 4 slot + rq / 2, element rq % 2
    const int srcA = 4 * (2 * quad) + (rq >> 1), srcB = srcA + 4;
    const bool odd_head = rq & 1;

    int64_t i = 0;
    Cursor k = cursor_at(c_begin, sch.cpu, p);
    for (int64_t c = c_begin; c < c_end; ++c, ++i, advance(k, sch.cpu, p)) {
        const int s = (int)(i % NS);
        // after a timeout the data is garbage, but every consumer warp still
        // runs the same barrier sequence to the end (no early exit)
        mbar_wait(full0 + 8 * s, (uint32_t)((i / NS) & 1), p.err_word, abort_flag);
        const uint32_t st = smem_base + s * L::stage;
        const int4 meta = reinterpret_cast<const int4*>(smem + L::meta)[s];
        const int64_t u = k.u;
        const uint32_t vis16 =
            ((warp < 2 ? (uint32_t)meta.y : (uint32_t)meta.z) >> (16 * (warp & 1))) & 0xffffu;

        if (u != cur) {
            cur = u;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m_run[e] = -INFINITY;
                l_part[e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KT; kk += 2) {
                uint32_t r4[4];
                ldsm_x4(st + q_lane + kk * 32, r4);
                qb[kk][0] = r4[0];
                qb[kk][1] = r4[1];
                qb[kk + 1][0] = r4[2];
                qb[kk + 1][1] = r4[3];
            }
        }

        // ---- S^T = K Q^T (two accumulator chains: even / odd k-steps) ----
        uint32_t ka[KT][4];
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) ldsm_x4(st + k_lane + kk * 32, ka[kk]);
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KT; kk += 2) {
            mma16816<E>(sa, ka[kk], qb[kk][0], qb[kk][1]);
            mma16816<E>(sb, ka[kk + 1], qb[kk + 1][0], qb[kk + 1][1]);
        }
        // sc[e]: slot rq (e < 2) or rq + 8 (e >= 2), head hc + (e & 1)
        float sc[4];
        const bool vlo = (vis16 >> rq) & 1u, vhi = (vis16 >> (rq + 8)) & 1u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool v = (e < 2) ? vlo : vhi;
            sc[e] = v ? (sa[e] + sb[e]) * p.scale_log2 : -INFINITY;
        }
        // ---- online softmax of heads hc, hc + 1 over the warp's 16 slots ----
        float alpha[2], pr[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(sc[e], sc[e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[e], mx);
            alpha[e] = rescale_factor(m_run[e], m_new);
            m_run[e] = m_new;
            pr[e] = (sc[e] == -INFINITY) ? 0.f : fast_exp2(sc[e] - m_new);
            pr[e + 2] = (sc[e + 2] == -INFINITY) ? 0.f : fast_exp2(sc[e + 2] - m_new);
            l_part[e] = l_part[e] * alpha[e] + pr[e] + pr[e + 2];
        }
        // ---- P^T as the B operand: high 16-bit part and remainder ----
        // packed (head hc, head hc + 1) of slot rq and of slot rq + 8
        const uint32_t h01 = E::pack2(pr[0], pr[1]), h23 = E::pack2(pr[2], pr[3]);
        const float2 f01 = E::unpack2(h01), f23 = E::unpack2(h23);
        const uint32_t l01 = E::pack2(pr[0] - f01.x, pr[1] - f01.y);
        const uint32_t l23 = E::pack2(pr[2] - f23.x, pr[3] - f23.y);
        // lane (head rq, slots 2 quad, 2 quad + 1 [+8]) gathers from the owners
        const uint32_t hA0 = __shfl_sync(0xffffffffu, h01, srcA), hB0 = __shfl_sync(0xffffffffu, h01, srcB);
        const uint32_t hA8 = __shfl_sync(0xffffffffu, h23, srcA), hB8 = __shfl_sync(0xffffffffu, h23, srcB);
        const uint32_t lA0 = __shfl_sync(0xffffffffu, l01, srcA), lB0 = __shfl_sync(0xffffffffu, l01, srcB);
        const uint32_t lA8 = __shfl_sync(0xffffffffu, l23, srcA), lB8 = __shfl_sync(0xffffffffu, l23, srcB);
        const uint32_t bh0 = half_of(hA0, odd_head) | (half_of(hB0, odd_head) << 16);
        const uint32_t bh1 = half_of(hA8, odd_head) | (half_of(hB8, odd_head) << 16);
        const uint32_t bl0 = half_of(lA0, odd_head) | (half_of(lB0, odd_head) << 16);
        const uint32_t bl1 = half_of(lA8, odd_head) | (half_of(lB8, odd_head) << 16);

        // ---- O^T = alpha O^T + V^T P^T ----
        uint32_t va[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) ldsm_x4_t(st + v_lane + mt * 32, va[mt]);
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= alpha[0];
                o[mt][1] *= alpha[1];
                o[mt][2] *= alpha[0];
                o[mt][3] *= alpha[1];
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816<E>(o[mt], va[mt], bh0, bh1);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816<E>(o[mt], va[mt], bl0, bl1);
        // the list's last chunk in this range: merge and write (or publish)
        // before the stage is released
        if (c + 1 == c_end || k.cc + 1 == sch.cpu) flush(cur, s);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if (cur < 0 && sch.cluster > 1) {
        cluster_sync();     // (an empty range: every segment holds a chunk)
        cluster_sync();
    }
}

// Resident clusters of `cluster` CTAs of `kern` on the current device, asked
// once per (kernel, device, cluster size).
template <class K>
int resident_clusters(K kern, int smem, int cluster) {
    static std::atomic<int> known[kMaxDevices][kMaxCluster + 1];   // count + 1; 0: not asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = known[dev][cluster].load(std::memory_order_relaxed);
    if (n == 0) {
        n = max_active_clusters(kern, kThreads, smem, cluster) + 1;
        known[dev][cluster].store(n, std::memory_order_relaxed);
    }
    return n - 1;
}

// Deepest ring that fits in shared memory next to the merge buffers, for
// one or two CTAs per SM (228 KB of shared memory per SM, 1 KB of it
// reserved per resident CTA).
template <int DK, int DV, bool VK, int CPS>
constexpr int stages_for() {
    constexpr int budget = (CPS == 1 ? 220 : 113) * 1024;
    constexpr int fixed = Smem<DK, DV, VK, 1>::total - Smem<DK, DV, VK, 1>::stage;
    constexpr int ns = (budget - fixed) / Smem<DK, DV, VK, 1>::stage;
    return ns > 6 ? 6 : (ns < 2 ? 2 : ns);
}

template <class E, int DK, int DV, bool VK, int CPS>
cudaError_t run_t(SfaParams p, int num_sms, void* ws, size_t ws_bytes, cudaStream_t stream) {
    constexpr int NS = stages_for<DK, DV, VK, CPS>();
    using L = Smem<DK, DV, VK, NS>;
    auto kern = sfa_decode_kernel<E, DK, DV, VK, NS>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
    if (err != cudaSuccess) return err;
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, L::total);
    if (err != cudaSuccess) return err;
    if (occ < 1) occ = 1;
    DecodeSched s;
    s.cpu = (p.topK + kChunk - 1) / kChunk;
    s.units = (int64_t)p.B * p.N2 * p.S1;
    s.total = s.units * s.cpu;
    int64_t ctas = p.num_ctas > 0 ? p.num_ctas : (int64_t)num_sms * occ;
    // many index lists per CTA: whole lists per range balance well enough
    s.aligned = (s.units >= 8 * ctas || s.units > kMaxCounters) ? 1 : 0;
    // fewer lists than resident CTAs: split every list into the same number
    // of segments (ctas = lists x segments), so that each range lies inside
    // one list -- a range that crosses into the next list pays a merge in
    // mid-range (measured on GQA decode, 128 lists of 16 chunks: 256 CTAs
    // 18.6 us against 20.4 us for the 304 resident ones).  With 2..8
    // segments, and room for all the clusters at once, a list's segments run
    // as one cluster and merge in distributed shared memory.
    s.cluster = 0;
    if (!s.aligned && p.num_ctas == 0) {
        const int64_t seg = ctas / s.units;
        if (seg >= 2) {
            const int64_t nseg = seg < s.cpu ? seg : s.cpu;
            ctas = s.units * nseg;
            if (nseg <= kMaxCluster && resident_clusters(kern, L::total, (int)nseg) >= s.units)
                s.cluster = (int)nseg;
        }
    }
    if (ctas > (s.aligned ? s.units : s.total)) ctas = s.aligned ? s.units : s.total;
    s.ctas = (int)ctas;
    if (s.aligned || s.cluster > 1) {
        s.seg_max = 1;
    } else {
        const int64_t lmin = s.total / s.ctas;             // shortest range
        int64_t seg = (s.cpu + lmin - 1) / lmin + 1;
        if (seg > s.cpu) seg = s.cpu;
        s.seg_max = (int)seg;
    }
    if (s.seg_max > 1) {
        const int64_t rows = (int64_t)p.B * p.N2 * p.S1 * p.G;
        const size_t need = (size_t)rows * s.seg_max * ((size_t)p.Dv + 2) * sizeof(float);
        if (!ws || ws_bytes < need || !p.counters) return cudaErrorInvalidValue;
        p.ws_o = static_cast<float*>(ws);
        p.ws_ml = p.ws_o + rows * s.seg_max * p.Dv;
    }
    err = launch_pdl_clustered(kern, dim3(s.ctas), dim3(kThreads), L::total, stream, s.cluster, p, s);
    count_launches(1);
    return err;
}

template <class E, int DK, int DV, bool VK>
cudaError_t run_c(const SfaParams& p, int num_sms, void* ws, size_t ws_bytes, cudaStream_t stream) {
    return p.ctas_per_sm == 1 ? run_t<E, DK, DV, VK, 1>(p, num_sms, ws, ws_bytes, stream)
                              : run_t<E, DK, DV, VK, 2>(p, num_sms, ws, ws_bytes, stream);
}

template <class E>
cudaError_t run_e(const SfaParams& p, bool vk, int num_sms, void* ws, size_t ws_bytes,
                  cudaStream_t stream) {
#define SFA_DECODE_CASE(DK_, DV_)                                                        \
    if (p.Dk == DK_ && p.Dv == DV_)                                                      \
        return vk ? run_c<E, DK_, DV_, true>(p, num_sms, ws, ws_bytes, stream)           \
                  : run_c<E, DK_, DV_, false>(p, num_sms, ws, ws_bytes, stream);
    SFA_DECODE_CASE(64, 64)
    SFA_DECODE_CASE(128, 64)
    SFA_DECODE_CASE(128, 128)
    SFA_DECODE_CASE(192, 128)
    SFA_DECODE_CASE(192, 192)
    SFA_DECODE_CASE(256, 128)
    SFA_DECODE_CASE(256, 256)
#undef SFA_DECODE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool decode_supported(const SfaParams& p) {
    const bool dims = (p.Dk == 64 && p.Dv == 64) || (p.Dk == 128 && (p.Dv == 64 || p.Dv == 128)) ||
                      (p.Dk == 192 && (p.Dv == 128 || p.Dv == 192)) ||
                      (p.Dk == 256 && (p.Dv == 128 || p.Dv == 256));
    return dims && p.G >= 1 && p.G <= kHeads;
}

size_t decode_ws_bytes(const SfaParams& p) {
    // seg_max <= chunks per index list (whatever the grid size)
    const int64_t rows = (int64_t)p.B * p.N2 * p.S1 * p.G;
    const int64_t cpu = (p.topK + kChunk - 1) / kChunk;
    return cpu > 1 ? (size_t)rows * cpu * ((size_t)p.Dv + 2) * sizeof(float) : 0;
}

cudaError_t launch_sfa_decode(const SfaParams& p, sfa_dtype dtype, int num_sms, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
    if (!decode_supported(p)) return cudaErrorInvalidValue;
    // value rows are the key rows' prefix when v aliases k
    const bool vk = (p.v == p.k) && (p.v_ss == p.k_ss);
    return dtype == SFA_DTYPE_BF16 ? run_e<BF16>(p, vk, num_sms, ws, ws_bytes, stream)
                                   : run_e<F16>(p, vk, num_sms, ws, ws_bytes, stream);
}

}  // namespace sfa
