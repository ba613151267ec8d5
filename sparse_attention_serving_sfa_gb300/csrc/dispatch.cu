// Path selection for a top-K sparse attention call.
#include "dispatch.h"

namespace sfa {

namespace {
constexpr int kMaxSplits = 32;
constexpr int kGenericChunk = 32;

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Splits of whole chunks so that no split is empty.
void set_splits(Plan& pl, int topK, int want, int chunk) {
    if (want < 1) want = 1;
    int per = ceil_div(topK, want);
    per = ceil_div(per, chunk) * chunk;
    pl.slots_per_split = per;
    pl.splits = ceil_div(topK, per);
}
}  // namespace

int max_splits_for(int topK) {
    int s = ceil_div(topK, 64);
    return s < kMaxSplits ? s : kMaxSplits;
}

size_t plan_extra_ws_bytes(int B, int S1, int N1, int N2, int Dk, int Dv, int topK) {
    SfaParams p{};
    p.B = B; p.S1 = S1; p.N1 = N1; p.N2 = N2; p.G = N1 / N2;
    p.Dk = Dk; p.Dv = Dv; p.topK = topK;
    p.v = p.k = &p;   // value is the key prefix (aliasing decides the MLA path)
    if (mla_supported(p)) return mla_ws_bytes(p);
    return decode_supported(p) ? decode_ws_bytes(p) : 0;
}

Plan choose_plan(const SfaParams& p, sfa_dtype, int num_sms, int forced_splits) {
    Plan pl;
    if (mla_supported(p) && forced_splits <= 0) {
        pl.kind = PATH_MLA;
        pl.splits = 1;
        pl.slots_per_split = p.topK;
        pl.extra_ws_bytes = mla_ws_bytes(p);
        return pl;
    }
    if (forced_splits <= 0 && group_tc_supported(p, num_sms)) {
        // whole index lists per CTA: no splits, no workspace
        pl.kind = PATH_GROUP_TC;
        pl.splits = 1;
        pl.slots_per_split = p.topK;
        return pl;
    }
    if (decode_supported(p)) {
        // persistent stream-K kernel: its own schedule, partials in extra_ws
        pl.kind = PATH_DECODE;
        pl.splits = 1;
        pl.slots_per_split = p.topK;
        pl.extra_ws_bytes = decode_ws_bytes(p);
        return pl;
    }
    return generic_split_plan(p, num_sms, forced_splits);
}

Plan generic_split_plan(const SfaParams& p, int num_sms, int forced_splits) {
    Plan pl;
    pl.kind = PATH_GENERIC;
    const int hb = p.G > 4 ? 8 : 4;
    const int64_t ctas = (int64_t)p.B * p.N2 * p.S1 * ceil_div(p.G, hb);
    int want = forced_splits > 0 ? forced_splits
                                 : (int)((2LL * num_sms + ctas - 1) / ctas);
    if (forced_splits <= 0 && want > max_splits_for(p.topK)) want = max_splits_for(p.topK);
    set_splits(pl, p.topK, want, kGenericChunk);
    return pl;
}

cudaError_t run_plan(const Plan& plan, SfaParams& p, sfa_dtype dtype, void* extra_ws,
                     int num_sms, cudaStream_t stream) {
    p.splits = plan.splits;
    p.slots_per_split = plan.slots_per_split;
    if (plan.kind == PATH_MLA)
        return launch_sfa_mla(p, dtype, num_sms, extra_ws, plan.extra_ws_bytes, stream);
    if (plan.kind == PATH_DECODE)
        return launch_sfa_decode(p, dtype, num_sms, extra_ws, plan.extra_ws_bytes, stream);
    if (plan.kind == PATH_GROUP_TC) return launch_sfa_group_tc(p, dtype, num_sms, stream);
    cudaError_t err = launch_sfa_generic(p, dtype, stream);
    if (err != cudaSuccess) return err;
    if (p.splits > 1) err = launch_sfa_combine(p, dtype, stream);
    return err;
}

}  // namespace sfa
