// sfa_run_noalloc: the generic top-K path with its split partials kept in a
// fixed device array instead of an allocated workspace, for callers that
// cannot allocate device memory (see include/sfa.h).
#include <math.h>

#include "common.cuh"
#include "dispatch.h"
#include "internal.h"

namespace sfa {
namespace {

// The scratch array.  In host code this name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress (SymbolCache), with the
// device current, once per device and context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SFA_NOALLOC_SCRATCH_BYTES];

SymbolCache g_scratch_cache;

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
    // the largest split count this entry point can choose must fit the array
    // (the same bound on every device, whatever its SM count)
    if (sfa_split_ws_bytes((int64_t)B * S1 * N1, max_splits_for(topK), Dv) >
        SFA_NOALLOC_SCRATCH_BYTES)
        return SFA_ERR_WORKSPACE;
    void* scratch = g_scratch_cache.address(reinterpret_cast<const void*>(&g_noalloc_scratch));
    if (!scratch) return SFA_ERR_CUDA;

    SfaParams p{};
    p.q = q; p.k = k; p.v = v; p.idx = sparse_idx; p.out = out; p.lse = lse;
    p.B = B; p.S1 = S1; p.S2 = S2; p.N1 = N1; p.N2 = N2; p.G = N1 / N2;
    p.Dk = Dk; p.Dv = Dv; p.topK = topK;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    resolve_strides(p, (int)layout, v == k);

    // the generic kernel's own split plan (the one sfa_run_ex uses for it)
    const Plan plan = generic_split_plan(p, num_sms(), 0);
    p.splits = plan.splits;
    p.slots_per_split = plan.slots_per_split;
    if (p.splits > 1) {
        p.ws_o = static_cast<float*>(scratch);
        p.ws_ml = p.ws_o + (int64_t)B * S1 * N1 * p.splits * Dv;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = launch_sfa_generic(p, dtype, s);
    if (err == cudaSuccess && p.splits > 1) err = launch_sfa_combine(p, dtype, s);
    return err == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}
