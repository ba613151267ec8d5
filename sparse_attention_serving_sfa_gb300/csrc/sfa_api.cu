// C ABI of the top-K sparse attention path: argument checks, layout ->
// stride resolution, split selection, workspace and kernel dispatch.
#include <math.h>

#include <atomic>
#include <map>
#include <mutex>
#include <thread>
#include <tuple>

#include "common.cuh"
#include "dispatch.h"
#include "internal.h"
#include "ptx.cuh"

namespace sfa {

// Library-wide device error word: bit 0 = a call with index validation on
// saw an index outside [0, S2).
__device__ int g_error_word = 0;

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

// Driver entry points through the runtime (the library does not link the
// driver library directly, so it also loads on machines without one).
template <class F>
F driver_fn(const char* name, int version) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(ptr);
}

}  // namespace

unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static std::once_flag once;
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    std::call_once(once, [] {
        get_current = driver_fn<GetCurrent>("cuCtxGetCurrent", 4000);
        get_id = driver_fn<GetId>("cuCtxGetId", 12000);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

void* SymbolCache::address(const void* symbol) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (!ptr[dev] || id == 0 || ctx[dev] != id) {
        // first use on this device, or a context made after a device reset:
        // the lookup also creates the device's primary context if needed
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
        ptr[dev] = p;
        ctx[dev] = current_context_id();
    }
    return ptr[dev];
}

namespace {

SymbolCache g_error_word_cache;

}  // namespace

int* device_error_word() {
    return static_cast<int*>(g_error_word_cache.address(reinterpret_cast<const void*>(&g_error_word)));
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Library-owned workspaces, one per (device, stream): calls on one stream run
// in stream order, calls on different streams never share one.  The
// per-thread default stream handle names a different stream in each host
// thread, so it is also keyed by the calling thread.
struct OwnedBuffer {
    void* ptr = nullptr;
    size_t bytes = 0;
    unsigned long long ctx = 0;   // context the buffer was allocated in
};
std::mutex g_ws_mu;
std::map<std::tuple<int, cudaStream_t, std::thread::id>, OwnedBuffer> g_ws;

cudaError_t owned_workspace(size_t need, cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const std::thread::id who =
        stream == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
    std::lock_guard<std::mutex> lock(g_ws_mu);
    OwnedBuffer& b = g_ws[std::make_tuple(dev, stream, who)];
    const unsigned long long id = current_context_id();
    if (b.ptr && id != 0 && b.ctx != id) {
        // allocated in a context that no longer exists (device reset): the
        // memory went with it
        b = OwnedBuffer{};
    }
    if (b.bytes < need) {
        if (b.ptr) {
            err = cudaStreamSynchronize(stream);   // the old buffer may still be in use
            if (err != cudaSuccess) return err;
            cudaFree(b.ptr);
            b = OwnedBuffer{};
        }
        size_t sz = need < (size_t(1) << 20) ? (size_t(1) << 20) : need;
        err = cudaMalloc(&b.ptr, sz);
        if (err != cudaSuccess) {
            b = OwnedBuffer{};
            return err;
        }
        // the counter region must start at zero (kernels leave it zero)
        err = cudaMemset(b.ptr, 0, sz);
        if (err != cudaSuccess) return err;
        b.bytes = sz;
        b.ctx = current_context_id();
    }
    *out = b.ptr;
    return cudaSuccess;
}

}  // namespace

int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

sfa_status check_args(const void* q, const void* k, const void* v, const int32_t* idx, int B,
                      int S1, int S2, int N1, int N2, int Dk, int Dv, int topK, float scale,
                      int layout, int causal, int dtype, const void* out, const float* lse,
                      const sfa_options* opt) {
    if (!q || !k || !v || !idx || !out) return SFA_ERR_INVALID_ARG;
    if (B < 1 || S1 < 1 || S2 < 1 || N1 < 1 || N2 < 1 || Dk < 1 || Dv < 1 || topK < 1)
        return SFA_ERR_INVALID_ARG;
    if (N1 % N2 != 0) return SFA_ERR_INVALID_ARG;               // GQA grouping (§3)
    if (Dk % 64 != 0 || Dv % 64 != 0 || Dv > Dk) return SFA_ERR_INVALID_ARG;
    if (topK > S2) return SFA_ERR_INVALID_ARG;                   // 1 <= topK <= S2
    if (causal && S1 > S2) return SFA_ERR_INVALID_ARG;           // causal needs S1 <= S2
    if (layout != SFA_LAYOUT_BSND && layout != SFA_LAYOUT_BNSD) return SFA_ERR_INVALID_ARG;
    if (dtype != SFA_DTYPE_F16 && dtype != SFA_DTYPE_BF16) return SFA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return SFA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(idx) || !aligned16(out))
        return SFA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SFA_ERR_INVALID_ARG;
    if (opt && opt->value_is_key_prefix && v != k) return SFA_ERR_INVALID_ARG;
    if (opt && (opt->num_splits < 0 || opt->ctas_per_sm < 0 || opt->ctas_per_sm > 2 ||
                opt->num_ctas < 0))
        return SFA_ERR_INVALID_ARG;
    if (opt && opt->workspace && !aligned16(opt->workspace)) return SFA_ERR_INVALID_ARG;
    if (Dk > 576 || Dv > 512) return SFA_ERR_UNSUPPORTED;
    // element offsets must fit int64 comfortably and grid.x must fit
    if ((int64_t)B * N2 * S1 > 0x7fffffffLL) return SFA_ERR_UNSUPPORTED;
    return SFA_OK;
}

void resolve_strides(SfaParams& p, int layout, bool prefix) {
    const int64_t S1 = p.S1, S2 = p.S2, N1 = p.N1, N2 = p.N2, Dk = p.Dk, Dv = p.Dv,
                  K = p.topK;
    const int64_t ldv = prefix ? Dk : Dv;
    if (layout == SFA_LAYOUT_BSND) {
        p.q_sb = S1 * N1 * Dk; p.q_ss = N1 * Dk; p.q_sh = Dk;
        p.k_sb = S2 * N2 * Dk; p.k_ss = N2 * Dk; p.k_sh = Dk;
        p.v_sb = S2 * N2 * ldv; p.v_ss = N2 * ldv; p.v_sh = ldv;
        p.i_sb = S1 * N2 * K; p.i_ss = N2 * K; p.i_sh = K;
        p.o_sb = S1 * N1 * Dv; p.o_ss = N1 * Dv; p.o_sh = Dv;
        p.l_sb = S1 * N1; p.l_ss = N1; p.l_sh = 1;
    } else {
        p.q_sb = N1 * S1 * Dk; p.q_sh = S1 * Dk; p.q_ss = Dk;
        p.k_sb = N2 * S2 * Dk; p.k_sh = S2 * Dk; p.k_ss = Dk;
        p.v_sb = N2 * S2 * ldv; p.v_sh = S2 * ldv; p.v_ss = ldv;
        p.i_sb = N2 * S1 * K; p.i_sh = S1 * K; p.i_ss = K;
        p.o_sb = N1 * S1 * Dv; p.o_sh = S1 * Dv; p.o_ss = Dv;
        p.l_sb = N1 * S1; p.l_sh = S1; p.l_ss = 1;
    }
}

}  // namespace sfa

using namespace sfa;

extern "C" {

const char* sfa_status_string(sfa_status s) {
    switch (s) {
        case SFA_OK: return "ok";
        case SFA_ERR_INVALID_ARG: return "invalid argument";
        case SFA_ERR_UNSUPPORTED: return "unsupported by this build";
        case SFA_ERR_WORKSPACE: return "workspace missing or too small";
        case SFA_ERR_INDEX_RANGE: return "sparse index outside [0, S2)";
        case SFA_ERR_CUDA: return "CUDA error";
        case SFA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    }
    return "unknown status";
}

uint64_t sfa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

sfa_status sfa_workspace_size(int B, int S1, int N1, int N2, int Dk, int Dv, int topK,
                              int num_splits, size_t* bytes) {
    if (!bytes || B < 1 || S1 < 1 || N1 < 1 || N2 < 1 || Dv < 1 || topK < 1 || num_splits < 0 ||
        Dk < Dv)
        return SFA_ERR_INVALID_ARG;
    const int splits = num_splits > 0 ? num_splits : max_splits_for(topK);
    // counter head + either split partials or the plan's own extra workspace
    const size_t split = sfa_split_ws_bytes((int64_t)B * S1 * N1, splits, Dv);
    const size_t extra = plan_extra_ws_bytes(B, S1, N1, N2, Dk, Dv, topK);
    const size_t region = split > extra ? split : extra;
    *bytes = region ? counter_region_bytes((int64_t)B * S1 * N2) + region : 0;
    return SFA_OK;
}

sfa_status sfa_run_ex(const void* q, const void* k, const void* v, const int32_t* sparse_idx,
                      int B, int S1, int S2, int N1, int N2, int Dk, int Dv, int topK,
                      float scale, sfa_layout layout, int causal, sfa_dtype dtype, void* out,
                      float* lse, sfa_stream_t stream, const sfa_options* opt) {
    sfa_status st = check_args(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale,
                               (int)layout, causal, (int)dtype, out, lse, opt);
    if (st != SFA_OK) return st;
    const bool prefix = (v == k);   // the prefix view is the only way v can alias k

    SfaParams p{};
    p.q = q; p.k = k; p.v = v; p.idx = sparse_idx; p.out = out; p.lse = lse;
    p.B = B; p.S1 = S1; p.S2 = S2; p.N1 = N1; p.N2 = N2; p.G = N1 / N2;
    p.Dk = Dk; p.Dv = Dv; p.topK = topK;
    p.causal = causal ? 1 : 0;
    p.validate = (opt && opt->validate_indices) ? 1 : 0;
    p.ctas_per_sm = opt ? opt->ctas_per_sm : 0;
    p.num_ctas = opt ? opt->num_ctas : 0;
    p.inputs_ready = (opt && opt->inputs_ready) ? 1 : 0;
    p.err_word = device_error_word();  // index checks (if validating) and wait timeouts
    if (!p.err_word) return SFA_ERR_CUDA;
    p.scale_log2 = scale * kLog2e;
    resolve_strides(p, (int)layout, prefix);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Plan plan = choose_plan(p, dtype, num_sms(), opt ? opt->num_splits : 0);
    p.splits = plan.splits;
    p.slots_per_split = plan.slots_per_split;

    // workspace: [counter head][split partials | plan's extra region]
    const size_t split_bytes = sfa_split_ws_bytes((int64_t)B * S1 * N1, p.splits, Dv);
    const size_t region = split_bytes + plan.extra_ws_bytes;
    const size_t head = counter_region_bytes((int64_t)B * S1 * N2);
    const size_t need = region ? head + region : 0;
    void* ws = nullptr;
    if (need > 0) {
        if (opt && opt->workspace) {
            if (opt->workspace_bytes < need) return SFA_ERR_WORKSPACE;
            ws = opt->workspace;
        } else {
            if (owned_workspace(need, s, &ws) != cudaSuccess) return SFA_ERR_CUDA;
        }
        p.counters = static_cast<unsigned*>(ws);
    }
    char* region_base = ws ? static_cast<char*>(ws) + head : nullptr;
    if (p.splits > 1) {
        p.ws_o = reinterpret_cast<float*>(region_base);
        p.ws_ml = p.ws_o + (int64_t)B * S1 * N1 * p.splits * Dv;
    }
    void* extra = region_base ? region_base + split_bytes : nullptr;
    cudaError_t err = run_plan(plan, p, dtype, extra, num_sms(), s);
    return err == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

sfa_status sfa_run(const void* q, const void* k, const void* v, const int32_t* sparse_idx,
                   int B, int S1, int S2, int N1, int N2, int Dk, int Dv, int topK, float scale,
                   sfa_layout layout, int causal, sfa_dtype dtype, void* out, float* lse,
                   sfa_stream_t stream) {
    return sfa_run_ex(q, k, v, sparse_idx, B, S1, S2, N1, N2, Dk, Dv, topK, scale, layout,
                      causal, dtype, out, lse, stream, nullptr);
}

sfa_status sfa_get_last_error(sfa_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SFA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int)) != cudaSuccess) return SFA_ERR_CUDA;
    if (word) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) return SFA_ERR_CUDA;
        return (word & kErrWaitTimeout) ? SFA_ERR_DEVICE_TIMEOUT : SFA_ERR_INDEX_RANGE;
    }
    return SFA_OK;
}

}  // extern "C"
