// Measurement probe: the sparse gather of a top-K call on its own.
//
// Reads every K row (and V row, unless V is the key prefix view) that a call
// of sfa_run with the same arguments gathers -- "SparseFlashAttention 算子
// API 描述", §2 具体子步骤, the sparse gather step -- and nothing else: no
// scores, no softmax, no output.  The time it takes bounds from below what
// any kernel that must fetch those bytes can take, so it is the ceiling the
// attention kernels' gather rate is judged against (random rows of HBM for
// decode, rows mostly resident in L2 for prefill).
//
// Work: blocks of 32 consecutive slots (of the flat sequence of all index
// lists) per warp, dealt out grid-stride to a persistent grid of two
// 256-thread CTAs per SM.  Lane l loads the index of slot l and its row
// addresses; then the warp reads the 32 rows several at a time, the lanes
// covering each row's 16-byte pieces (coalesced, as the attention kernels'
// producers do): 16 rows per lane in flight for rows of up to 512 bytes, 8
// up to 1024, 5 up to 1536.  Each thread folds what it read into one word so
// that no load can be dropped.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace sfa {
namespace {

constexpr int kProbeThreads = 256;

struct ProbeArgs {
    const uint4* k;
    const uint4* v;
    const int32_t* idx;
    int64_t lists;          // B * S1 * N2 index lists of topK positions
    int topK, S1, S2, N2;
    int kp, vp;             // 16-byte pieces per K row / per V row (0: V is K's prefix)
    int64_t k_row, v_row;   // row distance in 16-byte pieces (K row length, V row length)
    int bsnd;
    uint32_t* sink;
};

__device__ __forceinline__ const uint4* shfl_ptr(const uint4* p, int src) {
    const uint64_t u = reinterpret_cast<uint64_t>(p);
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)u, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(u >> 32), src);
    return reinterpret_cast<const uint4*>(((uint64_t)hi << 32) | lo);
}

// T: 16-byte pieces per lane and row (rows of up to 512 T bytes); R rows per round.
template <int T, int R>
__global__ void __launch_bounds__(kProbeThreads) sfa_gather_probe_kernel(const ProbeArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kProbeThreads + threadIdx.x) >> 5;
    const int64_t warps = (int64_t)gridDim.x * (kProbeThreads / 32);
    const int64_t slots = a.lists * a.topK;
    const int per = a.kp + a.vp;
    uint32_t acc = 0;
    for (int64_t s0 = warp * 32; s0 < slots; s0 += warps * 32) {
        // this lane's slot: its index, and the addresses of its K and V rows
        const int64_t slot = s0 + lane;
        const uint4* krow = nullptr;
        const uint4* vrow = nullptr;
        if (slot < slots) {
            const int id = a.idx[slot];          // index lists are contiguous runs of topK
            if (id >= 0 && id < a.S2) {
                // (b, n2) of the list: BSND lists are ((b * S1 + s1) * N2 + n2),
                // BNSD lists ((b * N2 + n2) * S1 + s1)
                const int64_t list = slot / a.topK;
                const int64_t b = list / ((int64_t)a.S1 * a.N2);
                const int64_t n2 = a.bsnd ? list % a.N2 : (list / a.S1) % a.N2;
                const int64_t row = a.bsnd ? (b * a.S2 + id) * a.N2 + n2
                                           : (b * a.N2 + n2) * a.S2 + id;
                krow = a.k + row * a.k_row;
                vrow = a.v + row * a.v_row;
            }
        }
        const int nrows = slots - s0 < 32 ? (int)(slots - s0) : 32;
        for (int j0 = 0; j0 < nrows; j0 += R) {
            uint4 got[R][T];
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const int j = j0 + u;
                const uint4* kr = shfl_ptr(krow, j < nrows ? j : 0);
                const uint4* vr = shfl_ptr(vrow, j < nrows ? j : 0);
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const int pc = lane + 32 * t;
                    got[u][t] = make_uint4(0, 0, 0, 0);
                    if (j < nrows && kr && pc < per)
                        got[u][t] = pc < a.kp ? __ldcg(kr + pc) : __ldcg(vr + (pc - a.kp));
                }
            }
#pragma unroll
            for (int u = 0; u < R; ++u)
#pragma unroll
                for (int t = 0; t < T; ++t)
                    acc ^= got[u][t].x ^ got[u][t].y ^ got[u][t].z ^ got[u][t].w;
        }
    }
    // one word per CTA, written only when it could matter, so the loads stay
    if (acc == 0x9e3779b9u) a.sink[blockIdx.x] = acc;
}

// ---- the same gather by TMA row gathers -----------------------------------
// One CTA per SM, grid-stride over 64-slot chunks of the flat slot sequence.
// Warp 0 turns a chunk's indices into row coordinates (lane l: slots l and
// 32 + l) and lanes 0..15 each copy four rows with tile::gather4 copies (one
// per column box of the row) into a ring of shared-memory stages, counted in
// bytes on the stage's mbarrier; warp 1 waits for each stage and releases it.
// Nothing reads the rows: the time is that of the copies alone.
constexpr int kTmaRows = 64;
constexpr int kTmaMaxStages = 8;

struct ProbeTmaArgs {
    const int32_t* idx;
    int64_t lists;
    int topK, S1, S2, N2, bsnd;
    int kboxes, vboxes;          // column boxes of a K / V row (no V boxes: V is K's prefix)
    int kbox, vbox;              // box widths (elements)
    int stages;
    uint32_t stage_bytes;
    int* err;
};

__global__ void __launch_bounds__(64, 1)
    sfa_gather_probe_tma_kernel(const __grid_constant__ CUtensorMap kmap,
                                const __grid_constant__ CUtensorMap vmap, const ProbeTmaArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = smem_u32(smem);
    const uint32_t full0 = base + (uint32_t)a.stages * a.stage_bytes;
    const uint32_t empty0 = full0 + 8 * kTmaMaxStages;
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(smem + (size_t)a.stages * a.stage_bytes + 16 * kTmaMaxStages);
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int64_t slots = a.lists * a.topK;
    const int64_t chunks = (slots + kTmaRows - 1) / kTmaRows;
    const uint32_t k_bytes = (uint32_t)a.kbox * 2u, v_bytes = (uint32_t)a.vbox * 2u;
    int64_t i = 0;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_map(&kmap);
            if (a.vboxes) tma_prefetch_map(&vmap);
        }
        for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++i) {
            const int s = (int)(i % a.stages);
            const uint32_t par = (uint32_t)((i / a.stages) & 1);
            if (!mbar_wait(empty0 + 8 * s, par ^ 1u, a.err, abort_flag)) break;
            int row[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t slot = c * kTmaRows + 32 * h + lane;
                int r = 0;                       // slots past the end / invalid: row 0
                if (slot < slots) {
                    const int id = a.idx[slot];
                    if (id >= 0 && id < a.S2) {
                        const int64_t list = slot / a.topK;
                        const int64_t b = list / ((int64_t)a.S1 * a.N2);
                        const int64_t n2 = a.bsnd ? list % a.N2 : (list / a.S1) % a.N2;
                        r = (int)(a.bsnd ? (b * a.S2 + id) * a.N2 + n2 : (b * a.N2 + n2) * a.S2 + id);
                    }
                }
                row[h] = r;
            }
            if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * s, a.stage_bytes);
            __syncwarp();
            // lane g < 16 copies rows 4 g .. 4 g + 3 of the chunk
            int rr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int src = 4 * (lane & 15) + j;
                const int r0 = __shfl_sync(0xffffffffu, row[0], src & 31);
                const int r1 = __shfl_sync(0xffffffffu, row[1], src & 31);
                rr[j] = src < 32 ? r0 : r1;
            }
            if (lane < 16) {
                const uint32_t st = base + (uint32_t)s * a.stage_bytes;
                for (int bx = 0; bx < a.kboxes; ++bx)
                    tma_gather4(st + (uint32_t)(bx * kTmaRows + 4 * lane) * k_bytes, &kmap, bx * a.kbox,
                                rr[0], rr[1], rr[2], rr[3], full0 + 8 * s);
                const uint32_t vst = st + (uint32_t)(a.kboxes * kTmaRows) * k_bytes;
                for (int bx = 0; bx < a.vboxes; ++bx)
                    tma_gather4(vst + (uint32_t)(bx * kTmaRows + 4 * lane) * v_bytes, &vmap, bx * a.vbox,
                                rr[0], rr[1], rr[2], rr[3], full0 + 8 * s);
            }
        }
    } else {
        for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++i) {
            const int s = (int)(i % a.stages);
            const uint32_t par = (uint32_t)((i / a.stages) & 1);
            if (!mbar_wait(full0 + 8 * s, par, a.err, abort_flag)) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
    }
}

// Widest box of at most 256 elements (a multiple of 8) that divides d.
int gather_box(int d) {
    for (int n = 1; n <= d; ++n)
        if (d % n == 0 && d / n <= 256 && (d / n) % 8 == 0) return d / n;
    return 0;
}

}  // namespace
}  // namespace sfa

using namespace sfa;

extern "C" sfa_status sfa_gather_probe_tma(const void* k, const void* v, const int32_t* sparse_idx,
                                           int B, int S1, int S2, int N2, int Dk, int Dv, int topK,
                                           sfa_layout layout, sfa_stream_t stream) {
    if (!k || !v || !sparse_idx) return SFA_ERR_INVALID_ARG;
    if (B < 1 || S1 < 1 || S2 < 1 || N2 < 1 || topK < 1 || topK > S2) return SFA_ERR_INVALID_ARG;
    if (Dk % 64 != 0 || Dv % 64 != 0 || Dv > Dk || Dk < 64) return SFA_ERR_INVALID_ARG;
    if (layout != SFA_LAYOUT_BSND && layout != SFA_LAYOUT_BNSD) return SFA_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(k) || !a16(v) || !a16(sparse_idx)) return SFA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)B * S2 * N2;
    if (rows >= ((int64_t)1 << 31)) return SFA_ERR_UNSUPPORTED;
    const bool prefix = v == k;
    ProbeTmaArgs a{};
    a.idx = sparse_idx;
    a.lists = (int64_t)B * S1 * N2;
    a.topK = topK; a.S1 = S1; a.S2 = S2; a.N2 = N2;
    a.bsnd = layout == SFA_LAYOUT_BSND ? 1 : 0;
    a.kbox = gather_box(Dk);
    a.kboxes = Dk / a.kbox;
    a.vbox = prefix ? 8 : gather_box(Dv);
    a.vboxes = prefix ? 0 : Dv / a.vbox;
    a.stage_bytes = (uint32_t)kTmaRows * 2u * (uint32_t)(Dk + (prefix ? 0 : Dv));
    a.stages = (int)((224u * 1024u) / a.stage_bytes);
    if (a.stages > kTmaMaxStages) a.stages = kTmaMaxStages;
    if (a.stages < 2) return SFA_ERR_UNSUPPORTED;
    a.err = device_error_word();
    CUtensorMap kmap, vmap;
    // rows of a contiguous k / v: (b, s, n2) or (b, n2, s) order, one row per
    // Dk (Dv) elements; the prefix view reads K's rows
    if (!make_rows_map(&kmap, k, true, Dk, rows, Dk, a.kbox)) return SFA_ERR_CUDA;
    if (!prefix && !make_rows_map(&vmap, v, true, Dv, rows, Dv, a.vbox)) return SFA_ERR_CUDA;
    if (prefix) vmap = kmap;
    const size_t smem = (size_t)a.stages * a.stage_bytes + 16 * kTmaMaxStages + 16;
    cudaError_t err = cudaFuncSetAttribute(sfa_gather_probe_tma_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return SFA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    sfa_gather_probe_tma_kernel<<<num_sms(), 64, smem, st>>>(kmap, vmap, a);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

extern "C" sfa_status sfa_gather_probe(const void* k, const void* v, const int32_t* sparse_idx,
                                       int B, int S1, int S2, int N2, int Dk, int Dv, int topK,
                                       sfa_layout layout, void* sink, size_t sink_bytes,
                                       sfa_stream_t stream) {
    if (!k || !v || !sparse_idx || !sink) return SFA_ERR_INVALID_ARG;
    if (B < 1 || S1 < 1 || S2 < 1 || N2 < 1 || topK < 1 || topK > S2) return SFA_ERR_INVALID_ARG;
    if (Dk % 64 != 0 || Dv % 64 != 0 || Dv > Dk || Dk < 64) return SFA_ERR_INVALID_ARG;
    if (layout != SFA_LAYOUT_BSND && layout != SFA_LAYOUT_BNSD) return SFA_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(k) || !a16(v) || !a16(sparse_idx) || !a16(sink)) return SFA_ERR_INVALID_ARG;
    const int sms = num_sms();
    const int grid = 2 * sms;
    if (sink_bytes < (size_t)grid * sizeof(uint32_t)) return SFA_ERR_WORKSPACE;
    ProbeArgs a{};
    const bool prefix = v == k;
    // up to three 16-byte pieces per lane and row: at most 1536 bytes per slot
    if (Dk / 8 + (prefix ? 0 : Dv / 8) > 96) return SFA_ERR_UNSUPPORTED;
    a.k = static_cast<const uint4*>(k);
    a.v = static_cast<const uint4*>(v);
    a.idx = sparse_idx;
    a.lists = (int64_t)B * S1 * N2;
    a.topK = topK; a.S1 = S1; a.S2 = S2; a.N2 = N2;
    a.kp = Dk / 8;                        // 8 16-bit elements per piece
    a.vp = prefix ? 0 : Dv / 8;
    a.k_row = Dk / 8;
    a.v_row = Dv / 8;
    a.bsnd = layout == SFA_LAYOUT_BSND ? 1 : 0;
    a.sink = static_cast<uint32_t*>(sink);
    const int pieces = a.kp + a.vp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (pieces <= 32)
        sfa_gather_probe_kernel<1, 16><<<grid, kProbeThreads, 0, st>>>(a);
    else if (pieces <= 64)
        sfa_gather_probe_kernel<2, 8><<<grid, kProbeThreads, 0, st>>>(a);
    else
        sfa_gather_probe_kernel<3, 5><<<grid, kProbeThreads, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}
