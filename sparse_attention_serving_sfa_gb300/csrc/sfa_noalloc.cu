// sfa_run_noalloc: the generic top-K path with its split partials kept in a
// fixed device array instead of an allocated workspace, for callers that
// cannot allocate device memory (see include/sfa.h).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "dispatch.h"
#include "internal.h"

namespace sfa {
namespace {

// The scratch array.  In host code this name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SFA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr int kChunk = 32;      // slot granule of the generic kernel's splits

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up on first use,
// with that device current).  nullptr on failure.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace sfa

using namespace sfa;

extern "C" sfa_status sfa_run_noalloc(const void* q, const void* k, const void* v,
                                      const int32_t* sparse_idx, int B, int S1, int S2, int N1,
                                      int N2, int Dk, int Dv, int topK, float scale,
                                      sfa_layout layout, int causal, sfa_dtype dtype, void* out,
                                      float* lse, sfa_stream_t stream) {
    sfa_status st = check_args(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale,
                               (int)layout, causal, (int)dtype, out, lse, nullptr);
    if (st != SFA_OK) return st;
    size_t bound = 0;
    st = sfa_workspace_size(B, S1, N1, N2, Dk, Dv, topK, 0, &bound);
    if (st != SFA_OK) return st;
    if (bound > SFA_NOALLOC_SCRATCH_BYTES) return SFA_ERR_WORKSPACE;
    void* scratch = scratch_for_current_device();
    if (!scratch) return SFA_ERR_CUDA;

    SfaParams p{};
    p.q = q; p.k = k; p.v = v; p.idx = sparse_idx; p.out = out; p.lse = lse;
    p.B = B; p.S1 = S1; p.S2 = S2; p.N1 = N1; p.N2 = N2; p.G = N1 / N2;
    p.Dk = Dk; p.Dv = Dv; p.topK = topK;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    resolve_strides(p, (int)layout, v == k);

    // Split count of the generic kernel: about two CTAs per SM, at most
    // max_splits_for(topK) (the count sfa_workspace_size bounds).
    const int hb = p.G > 4 ? 8 : 4;
    const int64_t ctas = (int64_t)B * N2 * S1 * ((p.G + hb - 1) / hb);
    int want = (int)((2LL * num_sms() + ctas - 1) / ctas);
    if (want > max_splits_for(topK)) want = max_splits_for(topK);
    if (want < 1) want = 1;
    int per = (topK + want - 1) / want;
    per = ((per + kChunk - 1) / kChunk) * kChunk;
    p.slots_per_split = per;
    p.splits = (topK + per - 1) / per;
    if (p.splits > 1) {
        if (sfa_split_ws_bytes((int64_t)B * S1 * N1, p.splits, Dv) > SFA_NOALLOC_SCRATCH_BYTES)
            return SFA_ERR_WORKSPACE;
        p.ws_o = static_cast<float*>(scratch);
        p.ws_ml = p.ws_o + (int64_t)B * S1 * N1 * p.splits * Dv;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = launch_sfa_generic(p, dtype, s);
    if (err == cudaSuccess && p.splits > 1) err = launch_sfa_combine(p, dtype, s);
    return err == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}
