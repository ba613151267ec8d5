// Path selection for a top-K sparse attention call.
#pragma once

#include "internal.h"

namespace sfa {

enum PathKind {
    PATH_GENERIC = 0,  // warp-FMA kernel, any supported shape
    PATH_DECODE = 1,   // small-group persistent gather kernel (sfa_decode.cu)
    PATH_MLA = 2,      // 128-head MLA tensor-core kernel (sfa_mla.cu)
    PATH_GROUP_TC = 3, // many index lists, 8 < G <= 16, Dv = 128: tensor cores (sfa_group_tc.cu)
};

struct Plan {
    int kind = PATH_GENERIC;
    int splits = 1;            // topK splits (partials merged by the combine kernel)
    int slots_per_split = 0;   // multiple of the path's chunk size
    size_t extra_ws_bytes = 0; // workspace beyond the split partials
};

// Picks the kernel path and split count for `p` (sizes and strides filled).
Plan choose_plan(const SfaParams& p, sfa_dtype dtype, int num_sms, int forced_splits);

// Launches the plan's kernels on `stream`; `extra_ws` holds
// plan.extra_ws_bytes bytes.
cudaError_t run_plan(const Plan& plan, SfaParams& p, sfa_dtype dtype, void* extra_ws,
                     int num_sms, cudaStream_t stream);

// Upper bound of Plan::extra_ws_bytes over every plan these sizes can get.
size_t plan_extra_ws_bytes(int B, int S1, int N1, int N2, int Dk, int Dv, int topK);

// Largest split count any plan uses for this topK.
int max_splits_for(int topK);

// Split plan of the generic warp-FMA kernel for `p` (sizes filled): about two
// CTAs per SM, at most max_splits_for(topK) splits of whole 32-slot chunks,
// unless `forced_splits` > 0.  kind = PATH_GENERIC.
Plan generic_split_plan(const SfaParams& p, int num_sms, int forced_splits);

}  // namespace sfa
