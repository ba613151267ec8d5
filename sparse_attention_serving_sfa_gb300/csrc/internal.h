// Internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sfa.h"

namespace sfa {

// Library-wide count of kernel launches (see sfa_kernel_launches()).
void count_launches(int n);

// One top-K sparse attention call, resolved to element strides.  A "row" of
// q / out is one (b, n1, s1) head vector; a row of k / v is one (b, n2, s2)
// key; a row of idx is the topK list of one (b, n2, s1).
struct SfaParams {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* idx;
    void* out;
    float* lse;
    float* ws_o;   // [rows][splits][Dv] unnormalised partial outputs
    float* ws_ml;  // [rows][splits][2]  (running max in log2 units, sum)
    int* err_word; // bit 0 set when validation sees an index outside [0, S2)
    unsigned* counters;  // per index list, zero between calls (reserved workspace head)
    int B, S1, S2, N1, N2, G, Dk, Dv, topK;
    int causal, validate, splits, slots_per_split;
    int ctas_per_sm, num_ctas;   // launch tuning of the small-group path (0 = auto)
    int inputs_ready;            // inputs not written by the preceding grid (sfa_options)
    float scale_log2;  // scale * log2(e)
    int64_t q_sb, q_ss, q_sh;
    int64_t k_sb, k_ss, k_sh;
    int64_t v_sb, v_ss, v_sh;
    int64_t i_sb, i_ss, i_sh;
    int64_t o_sb, o_ss, o_sh;
    int64_t l_sb, l_ss, l_sh;
};

// Host-side argument rules of the top-K entry points (status before launch).
sfa_status check_args(const void* q, const void* k, const void* v, const int32_t* idx, int B,
                      int S1, int S2, int N1, int N2, int Dk, int Dv, int topK, float scale,
                      int layout, int causal, int dtype, const void* out, const float* lse,
                      const sfa_options* opt);

// Fills the element strides of `p` (sizes already set) for `layout`; with
// `prefix`, value rows use the key's row length.
void resolve_strides(SfaParams& p, int layout, bool prefix);

// SM count of the current device (cached).
int num_sms();

// Every workspace starts with a fixed head of per-index-list arrival
// counters, kept zero between calls and never used for anything else.
constexpr int64_t kMaxCounters = 16384;
size_t counter_region_bytes(int64_t units);

// Bytes of split workspace for `splits` splits.
size_t sfa_split_ws_bytes(int64_t rows, int splits, int Dv);

// Small-group decode path (G <= 8, Dk == Dv in {64, 128, 256}, G * Dk <= 512):
// persistent stream-K kernel plus a combine of the ranges that share an index
// list.  decode_ws_bytes bounds the workspace it needs.
bool decode_supported(const SfaParams& p);
size_t decode_ws_bytes(const SfaParams& p);
cudaError_t launch_sfa_decode(const SfaParams& p, sfa_dtype dtype, int num_sms, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

// Small-group tensor-core path (8 < G <= 16, Dv == 128, Dk in {128, 192,
// 256}, at least four index lists per CTA of a one-per-SM grid): slots on the
// MMA M side, whole lists per CTA, no workspace.
bool group_tc_supported(const SfaParams& p, int num_sms);
cudaError_t launch_sfa_group_tc(const SfaParams& p, sfa_dtype dtype, int num_sms,
                                cudaStream_t stream);

// MLA path (G == 128 query heads per index list, Dk == 576, Dv == 512, value
// = key prefix): 2-CTA cluster tensor-core kernel, stream-K over chunks with
// an in-kernel merge of split units.  mla_ws_bytes bounds its workspace.
bool mla_supported(const SfaParams& p);
size_t mla_ws_bytes(const SfaParams& p);
cudaError_t launch_sfa_mla(const SfaParams& p, sfa_dtype dtype, int num_sms, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

// Generic warp-FMA path (any supported shape) and its split combine.
cudaError_t launch_sfa_generic(const SfaParams& p, sfa_dtype dtype, cudaStream_t stream);
cudaError_t launch_sfa_combine(const SfaParams& p, sfa_dtype dtype, cudaStream_t stream);

// One row tile of the block-sparse work list: `nrows` query rows starting at
// `row0`, all inside block row `rb`.
struct BsrTile {
    int rb, row0, nrows, pad;
};

struct BsrParams {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* lse;
    const int32_t* indptr;   // device copy, MB + 1
    const int32_t* indices;  // device copy, nnz
    const BsrTile* tiles;    // device work list
    int ntiles;
    int M, N, R, C, Hq, Hkv, d;
    float scale_log2;
    // element masking inside stored blocks: 0 none, 1 causal (bottom-right,
    // key column j visible to row i iff j <= i + N - M), 2 per-element bits
    // (`mask`: element (r, c) of the k-th stored block is bit
    // (k * R + r) * C + c, most significant bit first within each byte),
    // 3 variable blocks (HND tensors; `indptr` = key window list offsets,
    // `indices` = the key windows, 6 ints each: the first keys of four
    // 16-key quarters, then the 64-bit allowed-key mask low / high word;
    // `causal` adds the bottom-right rule)
    int mask_mode;
    const uint8_t* mask;
    int causal;
    // plan()'s logits_soft_cap times log2(e); 0 = no cap
    float softcap_log2;
    // 1: k and v are (Hkv, N, d) (HND) instead of (N, Hkv, d) (NHD); modes
    // 0-2 only (mode 3 is HND throughout)
    int kv_hnd;
    // 8-bit q / k / v: 0 no (16-bit), 1 E4M3, 2 E5M2 (the launch's dtype is
    // then the output's); per-head dequantisation scales, NULL = 1
    int f8;
    const float* scale_q;   // [Hq]
    const float* scale_k;   // [Hkv]
    const float* scale_v;   // [Hkv]
};

cudaError_t launch_bsr_generic(const BsrParams& p, sfa_dtype dtype, cudaStream_t stream);

// Tensor-core BSR path (head_dim 64 or 128, C % 64 == 0, G | 128).  A work
// item (4 ints: block row, first row, kv head, -) covers
// bsr_tc_rows_per_item() rows of one block row; in mode 3 the 4 ints are
// (key window list, first row, kv head, end of the row block).
// launch_bsr_tc runs the per-element mask mode (2) only, in 64-key blocks.
bool bsr_tc_supported(int head_dim, int C, int Hq, int Hkv);
int bsr_tc_rows_per_item(int Hq, int Hkv);
cudaError_t launch_bsr_tc(const BsrParams& p, const void* items, int nitems, int* err_word,
                          sfa_dtype dtype, cudaStream_t stream);

// Modes 0 (plain), 1 (causal) and 3 (variable blocks) on the tensor cores in
// 128-key steps; same support and work items as launch_bsr_tc.
cudaError_t launch_bsr_tc_wide(const BsrParams& p, const void* items, int nitems, int* err_word,
                               sfa_dtype dtype, cudaStream_t stream);

// TMA tiled 3-D maps, 128-byte swizzle, box 64 dims wide: over a
// [rows][heads][dim] tensor (box hb heads x rb rows) and over a
// [heads][rows][dim] tensor (box rb rows x hb heads).
bool make_map(CUtensorMap* map, const void* base, bool bf16, int dim, int heads, int rows, int hb,
              int rb);
bool make_map_hnd(CUtensorMap* map, const void* base, bool bf16, int dim, int rows, int heads,
                  int rb, int hb);
// 2-D map over `rows` rows of `width` 16-bit elements, row_stride elements
// apart; box = box_w elements x 1 row, no swizzle (tile::gather4 copies).
bool make_rows_map(CUtensorMap* map, const void* base, bool bf16, int width, int64_t rows,
                   int64_t row_stride, int box_w);
// The driver's cuTensorMapEncodeTiled (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// The same over 8-bit elements, box 128 elements (128 bytes) wide.
bool make_map8(CUtensorMap* map, const void* base, int dim, int heads, int rows, int hb, int rb);
bool make_map8_hnd(CUtensorMap* map, const void* base, int dim, int rows, int heads, int rb,
                   int hb);

// Launches `kern` with programmatic dependent launch allowed: the grid may be
// scheduled while the previous kernel in the stream finishes; the kernel must
// call griddepcontrol.wait before its first global-memory access.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same with the grid cut into thread-block clusters of `cluster` CTAs
// along x (cluster <= 1: no clusters).
template <class... KArgs, class... Args>
cudaError_t launch_pdl_clustered(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster > 1 ? cluster : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// How many clusters of `cluster` CTAs of `kern` (block threads, smem bytes of
// dynamic shared memory) can be resident at once; 0 if the query fails.
template <class... KArgs>
int max_active_clusters(void (*kern)(KArgs...), int block, size_t smem, int cluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Device address of the library's error word on the current device.
int* device_error_word();

// Id of the calling thread's current CUDA context (0 if none).
unsigned long long current_context_id();

// Device addresses of one __device__ symbol, looked up once per device and
// again whenever that device's current context differs from the one of the
// lookup (after a device reset the module is loaded anew).  address() takes
// the symbol's host-side stand-in (&symbol) and returns nullptr on failure.
constexpr int kMaxDevices = 64;
struct SymbolCache {
    std::mutex mu;
    void* ptr[kMaxDevices] = {};
    unsigned long long ctx[kMaxDevices] = {};
    void* address(const void* symbol);
};

}  // namespace sfa
