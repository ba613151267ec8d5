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

}  // namespace
}  // namespace sfa

using namespace sfa;

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
