/*
 * sfa.h -- C ABI of the GB300 sparse flash attention library (libsfa_gb300.so).
 *
 * Two forms of sparse attention, both computed entirely by the library's own
 * sm_103a CUDA kernels:
 *
 *   1. Top-K index form ("SparseFlashAttention 算子 API 描述", §2 算子定义 and
 *      §3 接口规范): every (b, n2, s1) owns topK int32 key positions; the
 *      N1/N2 query heads of KV head n2 attend only to those rows of K and V.
 *   2. Block-sparse form ("flashinfer.sparse", BlockSparseAttentionWrapper):
 *      query row i attends to key column j iff block (i / R, j / C) is stored
 *      in a BSR matrix (indptr / indices), with a plan() / run() split.
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, out, lse, sparse_idx and the workspaces are
 *     DEVICE pointers owned by the caller; the library never frees them.
 *     Pointers named *_host are host memory, read during the call only.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and returns without synchronising, except sfa_get_last_error.
 *   - Host-detectable argument errors return a status before anything is
 *     launched; no kernel traps, asserts or spins on the device.
 *   - All device pointers must be 16-byte aligned.
 */
#ifndef SFA_GB300_H
#define SFA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* sfa_stream_t;

typedef enum {
    SFA_OK = 0,
    SFA_ERR_INVALID_ARG = 1,  /* shape, enum, pointer or alignment rule broken */
    SFA_ERR_UNSUPPORTED = 2,  /* legal per the spec but outside this build's limits */
    SFA_ERR_WORKSPACE = 3,    /* caller workspace missing or too small */
    SFA_ERR_INDEX_RANGE = 4,  /* a sparse index outside [0, S2) was seen (validate mode) */
    SFA_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    SFA_ERR_DEVICE_TIMEOUT = 6 /* a kernel's bounded wait gave up (reported by
                                  sfa_get_last_error); that call's output is invalid */
} sfa_status;

/* Tensor layouts ("SparseFlashAttention 算子 API 描述", §2 布局说明):
 *   BSND: q [B,S1,N1,Dk]  k [B,S2,N2,Dk]  v [B,S2,N2,Dv]
 *         sparse_idx [B,S1,N2,topK]  out [B,S1,N1,Dv]  lse [B,S1,N1]
 *   BNSD: q [B,N1,S1,Dk]  k [B,N2,S2,Dk]  v [B,N2,S2,Dv]
 *         sparse_idx [B,N2,S1,topK]  out [B,N1,S1,Dv]  lse [B,N1,S1]
 * All row-major and contiguous, except v in key-prefix mode (below). */
typedef enum { SFA_LAYOUT_BSND = 0, SFA_LAYOUT_BNSD = 1 } sfa_layout;

/* Element types.  The top-K entry points take F16 or BF16, shared by q, k,
 * v and out (§3 数据类型).  E4M3 / E5M2 are the two 8-bit floating-point
 * formats of the operator page's precision table (§4 精度要求), accepted by
 * bsr_plan_set_data_types only. */
typedef enum {
    SFA_DTYPE_F16 = 0,
    SFA_DTYPE_BF16 = 1,
    SFA_DTYPE_E4M3 = 2,   /* 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448 */
    SFA_DTYPE_E5M2 = 3    /* 1 sign, 5 exponent (bias 15), 2 mantissa bits; max 57344 */
} sfa_dtype;

/*
 * sfa_run -- top-K sparse flash attention.
 *
 * Computes, for every batch b, query head n1 (KV head n2 = n1 / (N1/N2)) and
 * query position s1, with the topK positions idx_i = sparse_idx[b, n2, s1, i]
 * (layout-mapped):
 *     s_i   = scale * <q[b,n1,s1,:Dk], k[b,n2,idx_i,:Dk]>
 *     s_i   = -inf  if causal and idx_i > s1 + (S2 - S1)      (bottom-right)
 *     out   = sum_i softmax(s)_i * v[b,n2,idx_i,:Dv]
 *     lse   = ln(sum_i exp(s_i))
 * (§2 具体子步骤 and 因果掩码).  A row whose slots are all masked writes
 * out = +0 and lse = -inf (§3 规则与约束: "softmax 输出按全 0 处理").
 * Duplicate positions in a row count once per slot, as in the spec's golden.
 *
 * Arguments
 *   q, k, v       device, dtype elements, layout above.  If v == k and
 *                 Dv <= Dk, v is read as the prefix view k[..., :Dv] (rows of
 *                 Dk elements; §3 语义约束, the MLA latent cache).
 *   sparse_idx    device int32 in [0, S2).  Out-of-range positions are never
 *                 dereferenced: their slot is treated as masked.
 *   B,S1,S2,N1,N2 sizes; N1 % N2 == 0; causal requires S1 <= S2.
 *   Dk, Dv        multiples of 64, Dv <= Dk; this build: Dk <= 576, Dv <= 512.
 *   topK          1 <= topK <= S2.
 *   scale         softmax scale (usually 1/sqrt(Dk)); any finite value.
 *   out           device, dtype, layout above.
 *   lse           device float32 or NULL.
 *   stream        CUDA stream for every launch of the call.
 * Workspace: a library-owned device workspace is allocated on first use for
 * each (device, stream) pair and grown when a larger shape needs it (the
 * growing call synchronises that stream once).  Calls on different streams
 * therefore never share a workspace and may overlap on the GPU; calls on one
 * stream share it and run in stream order.  The per-thread default stream
 * (cudaStreamPerThread) gets one workspace per host thread.  Each workspace
 * is held until the process exits.  Use sfa_run_ex to pass your own.
 * Errors: SFA_ERR_INVALID_ARG / SFA_ERR_UNSUPPORTED before any launch;
 * SFA_ERR_CUDA if a launch fails.
 */
sfa_status sfa_run(const void* q, const void* k, const void* v, const int32_t* sparse_idx,
                   int B, int S1, int S2, int N1, int N2, int Dk, int Dv, int topK, float scale,
                   sfa_layout layout, int causal, sfa_dtype dtype, void* out, float* lse,
                   sfa_stream_t stream);

/* Options of sfa_run_ex.  Zero-initialise and set what you need. */
typedef struct {
    /* Caller-owned device float workspace for split-topK partial results
     * ("flashinfer.sparse", BlockSparseAttentionWrapper.__init__: the float
     * workspace that holds split-k intermediates).  NULL = library-owned.
     * Size: sfa_workspace_size().  Its head holds per-index-list arrival
     * counters: zero-fill the buffer once before its first use; every call
     * that completes leaves the head zero again (after an
     * SFA_ERR_DEVICE_TIMEOUT, zero it again).  Must not be used by another
     * call that overlaps this one on the GPU. */
    void* workspace;
    size_t workspace_bytes;
    /* 1: v is the prefix view k[..., :Dv] (v must equal k).  0: inferred from
     * v == k. */
    int value_is_key_prefix;
    /* 1: an out-of-range index also sets the library's device error word,
     * read (and cleared) by sfa_get_last_error. */
    int validate_indices;
    /* Number of topK splits of the generic path; 0 = chosen from the SM
     * count. */
    int num_splits;
    /* Launch tuning of the small-group paths.  ctas_per_sm (G <= 8):
     * persistent CTAs per SM of the warp-MMA kernel (1 = deep shared-memory
     * ring, 2 = two CTAs with shallow rings).  num_ctas: the total number of
     * CTAs (chunk or index-list ranges) of that kernel, or of the tensor-core
     * kernel for many index lists of 9 to 16 heads.  0 = automatic. */
    int ctas_per_sm;
    int num_ctas;
    /* 1: the caller states that q, k, v and sparse_idx were not written by
     * the kernel that precedes this call in the stream (they were ready
     * before it started), so the small-group kernel (G <= 8) and the MLA
     * kernel (128 heads) may read them while that kernel is still running:
     * they wait for the preceding grid (programmatic dependent launch) only
     * before their first write of out, lse or the workspace, and a call's
     * gather overlaps the previous call's tail.  Other paths ignore it.
     * 0 = wait before the first read. */
    int inputs_ready;
} sfa_options;

sfa_status sfa_run_ex(const void* q, const void* k, const void* v, const int32_t* sparse_idx,
                      int B, int S1, int S2, int N1, int N2, int Dk, int Dv, int topK,
                      float scale, sfa_layout layout, int causal, sfa_dtype dtype, void* out,
                      float* lse, sfa_stream_t stream, const sfa_options* opt);

/* Bytes of float workspace sfa_run_ex may need for these sizes with any
 * split count it would choose (or with num_splits, if > 0).  Host only. */
sfa_status sfa_workspace_size(int B, int S1, int N1, int N2, int Dk, int Dv, int topK,
                              int num_splits, size_t* bytes);

/* Synchronises `stream`, then reads (and clears) the library's device error
 * word: SFA_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up since the
 * last check, else SFA_ERR_INDEX_RANGE if a call with validate_indices saw an
 * index outside [0, S2); SFA_ERR_CUDA on a CUDA error; else SFA_OK. */
sfa_status sfa_get_last_error(sfa_stream_t stream);

/* Static text for a status code. */
const char* sfa_status_string(sfa_status status);

/* Number of CUDA kernels this library has launched in this process, over
 * all entry points (a diagnostic for launch accounting; no paper
 * counterpart). */
uint64_t sfa_kernel_launches(void);

/*
 * sfa_gather_probe -- measurement probe (no paper counterpart): reads every
 * K row, and every V row unless v == k (the prefix view), that sfa_run with
 * the same k, v, sparse_idx, sizes and layout gathers ("SparseFlashAttention
 * 算子 API 描述", §2 具体子步骤, the sparse gather step), and does nothing
 * else.  Its duration is the floor for any kernel that must fetch those
 * bytes: the gather ceiling the attention kernels are measured against.
 *   sink        device buffer of at least 2 * SM count * 4 bytes; it may
 *               receive one word per CTA (a fold of the data read).
 * The rows are read with 16-byte loads, the lanes of a warp covering a row's
 * pieces (coalesced), many rows in flight per lane.
 * Arguments otherwise as sfa_run (16-bit elements); out-of-range indices are
 * skipped.  Errors: SFA_ERR_INVALID_ARG, SFA_ERR_WORKSPACE (sink too small),
 * SFA_ERR_UNSUPPORTED (K + V bytes per slot above 1536), SFA_ERR_CUDA.
 */
sfa_status sfa_gather_probe(const void* k, const void* v, const int32_t* sparse_idx, int B,
                            int S1, int S2, int N2, int Dk, int Dv, int topK, sfa_layout layout,
                            void* sink, size_t sink_bytes, sfa_stream_t stream);

/*
 * sfa_gather_probe_tma -- the same measurement probe with the rows moved by
 * TMA row gathers (cp.async.bulk.tensor tile::gather4: four rows of a 2-D
 * tensor map per copy, one copy per column box of up to 256 elements) into a
 * ring of shared-memory stages, one CTA per SM; nothing reads the rows.
 * k and v must be contiguous ([B][S2][N2][D] for BSND, [B][N2][S2][D] for
 * BNSD), or v == k (the prefix view: K rows only).  Arguments otherwise as
 * sfa_gather_probe, without the sink.  Errors: SFA_ERR_INVALID_ARG,
 * SFA_ERR_UNSUPPORTED (B * S2 * N2 >= 2^31 rows, or rows too long for two
 * 64-row stages), SFA_ERR_CUDA.
 */
sfa_status sfa_gather_probe_tma(const void* k, const void* v, const int32_t* sparse_idx, int B,
                                int S1, int S2, int N2, int Dk, int Dv, int topK,
                                sfa_layout layout, sfa_stream_t stream);

/* Size of the device scratch array behind sfa_run_noalloc (8 MiB). */
#define SFA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * sfa_run_noalloc -- sfa_run for callers that cannot allocate device memory.
 * (No counterpart in the operator spec or the FlashInfer pages: this is a
 * deployment variant of the same computation.)
 *
 * Some callers may not call cudaMalloc at all: a serving engine that has
 * reserved nearly all of HBM up front for its KV cache and owns every later
 * allocation, a plugin host that forbids libraries from allocating behind its
 * back, or a latency-critical loop that cannot take the device-wide
 * synchronisation cudaFree can cause.  sfa_run, by contrast, may allocate (and
 * grow) its library-owned workspace.  This entry point computes the same result
 * as sfa_run with the generic kernel and its split combine, and keeps the split
 * partials in a fixed device array of SFA_NOALLOC_SCRATCH_BYTES that is part of
 * the library image: every GPU that loads the library holds those bytes until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * Arguments, layouts and results are those of sfa_run (value-prefix mode is
 * inferred from v == k; no index validation).
 * Limits: the split partials of the largest split count the generic kernel
 * can choose for topK -- rows = B * S1 * N1 rows of (Dv + 2) floats times
 * min(ceil(topK / 64), 32) splits -- must fit SFA_NOALLOC_SCRATCH_BYTES;
 * larger shapes are rejected with SFA_ERR_WORKSPACE before anything is
 * launched (the same rule on every GPU, whatever its SM count).  Other
 * argument errors as in sfa_run.
 * Set-up: the first call on each device looks up the device address of the
 * array (cudaGetSymbolAddress) with that device current, and looks it up
 * again after the device's context has been re-created (cudaDeviceReset);
 * make the first call on a device before any stream capture.
 * Sharing: all calls on a device share the one array and it keeps the last
 * call's contents.  Nothing in it needs clearing (every split partial is
 * written before it is read), but calls whose kernels overlap on the GPU --
 * concurrent streams, or several host threads -- race on it and must be
 * serialised by the caller.
 */
sfa_status sfa_run_noalloc(const void* q, const void* k, const void* v,
                           const int32_t* sparse_idx, int B, int S1, int S2, int N1, int N2,
                           int Dk, int Dv, int topK, float scale, sfa_layout layout, int causal,
                           sfa_dtype dtype, void* out, float* lse, sfa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Block-sparse (BSR) attention ("flashinfer.sparse",
 * BlockSparseAttentionWrapper: plan() builds cached auxiliary structures,
 * run() may then be called many times). */

typedef struct bsr_plan_s* bsr_plan_t;

/*
 * bsr_plan -- validate a BSR pattern and build the device work list.
 *
 *   indptr_host   host int32[MB + 1], MB = ceil(M / R); indptr[0] == 0,
 *                 non-decreasing.
 *   indices_host  host int32[nnz] (nnz = indptr[MB]) block columns, each in
 *                 [0, NB), NB = N / C; no repeats within a block row (a mask
 *                 holds a block once).  Any order.
 *   M, N, R, C    rows / columns of the mask and block size; N % C == 0.
 *   num_qo_heads, num_kv_heads   num_qo_heads % num_kv_heads == 0; qo head h
 *                 reads kv head h / (num_qo_heads / num_kv_heads).
 *   head_dim      multiple of 64, <= 256 in this build.
 *   causal        nonzero: bottom-right causal mask on top of the block
 *                 pattern -- key column j is visible to query row i iff
 *                 j <= i + (N - M) (plan(): "causal", the same rule the
 *                 prefill page's tril example pins).  Blocks entirely above
 *                 that diagonal are dropped from the plan.
 *   sm_scale      softmax scale; <= 0 selects 1/sqrt(head_dim).
 *   dtype         element type of q, k, v and out.
 *   int_ws        device buffer the work list is copied into (on `stream`);
 *                 size from bsr_plan_int_workspace_size().
 *   float_ws      device float workspace for split partial results, or
 *                 NULL.  This build's BSR kernels keep every row block's
 *                 keys in one CTA and never touch it.
 *   plan_out      receives a handle, valid until bsr_plan_destroy(); the
 *                 workspaces must stay allocated as long as it is used.
 */
sfa_status bsr_plan(const int32_t* indptr_host, const int32_t* indices_host, int M, int N,
                    int R, int C, int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                    float sm_scale, sfa_dtype dtype, void* int_ws, size_t int_ws_bytes,
                    void* float_ws, size_t float_ws_bytes, sfa_stream_t stream,
                    bsr_plan_t* plan_out);

/* Bytes of int workspace bsr_plan needs for this pattern. Host only. */
sfa_status bsr_plan_int_workspace_size(const int32_t* indptr_host, int M, int N, int R, int C,
                                       int num_qo_heads, int num_kv_heads, int head_dim,
                                       size_t* bytes);

/*
 * bsr_plan_masked -- bsr_plan with a per-element mask inside the stored
 * blocks ("flashinfer.sparse", BlockSparseAttentionWrapper.plan(): `mask`
 * of shape (nnz, R, C) and its bit-packed form `packed_mask`).
 *
 *   packed_mask_host  host bytes, ceil(nnz * R * C / 8) of them, or NULL
 *                 (then this is bsr_plan).  Element (r, c) of the k-th
 *                 stored block (indices order) says whether query row
 *                 (i / R) * R + r may attend key column indices[k] * C + c;
 *                 the (nnz, R, C) tensor is flattened in that order and
 *                 packed most significant bit first (element e is bit
 *                 7 - e % 8 of byte e / 8; the page leaves the bit order
 *                 open).  nnz * R * C must fit in an int32
 *                 (SFA_ERR_UNSUPPORTED otherwise).
 *   causal        ignored when a mask is given (plan(): causal applies only
 *                 without a custom mask).
 *   int_ws        size from bsr_plan_masked_int_workspace_size(...,
 *                 with_mask = 1): the work list plus the mask bytes.
 * Rows whose every element is masked write out = +0 and lse = -inf.  Other
 * arguments, ownership and errors as bsr_plan.
 */
sfa_status bsr_plan_masked(const int32_t* indptr_host, const int32_t* indices_host,
                           const uint8_t* packed_mask_host, int M, int N, int R, int C,
                           int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                           float sm_scale, sfa_dtype dtype, void* int_ws, size_t int_ws_bytes,
                           void* float_ws, size_t float_ws_bytes, sfa_stream_t stream,
                           bsr_plan_t* plan_out);

/* Bytes of int workspace bsr_plan_masked needs (with_mask = 0: as
 * bsr_plan_int_workspace_size).  Host only. */
sfa_status bsr_plan_masked_int_workspace_size(const int32_t* indptr_host, int M, int N, int R,
                                              int C, int num_qo_heads, int num_kv_heads,
                                              int head_dim, int with_mask, size_t* bytes);

/* Layout of the k / v tensors of bsr_run ("flashinfer.prefill.
 * single_prefill_with_kv_cache", parameter kv_layout: NHD or HND). */
typedef enum { SFA_KV_LAYOUT_NHD = 0, SFA_KV_LAYOUT_HND = 1 } sfa_kv_layout;

/*
 * bsr_plan_set_kv_layout -- the layout of the k and v tensors of every later
 * bsr_run with this plan: SFA_KV_LAYOUT_NHD (N, num_kv_heads, head_dim), the
 * default, or SFA_KV_LAYOUT_HND (num_kv_heads, N, head_dim), as the
 * single-request prefill page's kv_layout defines them.  q and out stay
 * (M, num_qo_heads, head_dim).  Host only.
 * Errors: SFA_ERR_INVALID_ARG (NULL plan, another value).
 */
sfa_status bsr_plan_set_kv_layout(bsr_plan_t plan, sfa_kv_layout kv_layout);

/*
 * bsr_run -- block-sparse attention with a plan (bsr_run_scaled without
 * scales).
 *   q    device (M, num_qo_heads, head_dim), NHD, dtype.
 *   k, v device (N, num_kv_heads, head_dim), NHD, dtype, or
 *        (num_kv_heads, N, head_dim) after bsr_plan_set_kv_layout(HND).
 *   out  device (M, num_qo_heads, head_dim), dtype.
 *   lse  device float32 (M, num_qo_heads) or NULL: natural-log log-sum-exp
 *        of the scaled logits of the row's allowed columns.
 * Rows with no visible column (no stored block, or every element masked)
 * write out = +0 and lse = -inf.
 */
sfa_status bsr_run(bsr_plan_t plan, const void* q, const void* k, const void* v, void* out,
                   float* lse, sfa_stream_t stream);

/*
 * bsr_plan_set_logits_soft_cap -- plan()'s logits_soft_cap ("flashinfer.sparse",
 * BlockSparseAttentionWrapper.plan()): with cap > 0 every logit x (the scaled
 * score sm_scale * q.k; the page does not say whether x includes sm_scale)
 * becomes cap * tanh(x / cap) before the softmax, and lse is over the capped
 * logits.  cap <= 0 turns it off (the page's default 0).  Applies to every
 * later bsr_run with this plan.  Host only.
 * Errors: SFA_ERR_INVALID_ARG (NULL plan, non-finite cap).
 */
sfa_status bsr_plan_set_logits_soft_cap(bsr_plan_t plan, float logits_soft_cap);

/*
 * bsr_plan_set_data_types -- plan()'s q_data_type, kv_data_type and
 * o_data_type ("flashinfer.sparse", BlockSparseAttentionWrapper.plan();
 * kv_data_type defaults to q_data_type, o_data_type to half).  bsr_plan's
 * `dtype` sets all three; this changes them for every later run.
 * Combinations of this build:
 *   - q = k / v = out = the plan's dtype (F16 or BF16), as after bsr_plan;
 *   - q = k / v in {E4M3, E5M2} with out in {F16, BF16} (FP8 attention; the
 *     per-head scales of bsr_run_scaled apply), for plans of the tensor-core
 *     path with head_dim 128 and no per-element mask, without a soft cap.
 * Host only.  Errors: SFA_ERR_INVALID_ARG (NULL plan, a value outside
 * sfa_dtype), SFA_ERR_UNSUPPORTED (any other combination or plan).
 */
sfa_status bsr_plan_set_data_types(bsr_plan_t plan, sfa_dtype q_dtype, sfa_dtype kv_dtype,
                                   sfa_dtype o_dtype);

/*
 * bsr_run_scaled -- run() with its per-head scales ("flashinfer.sparse",
 * BlockSparseAttentionWrapper.run(): scale_q [num_qo_heads], scale_k and
 * scale_v [num_kv_heads], "for FP8 quantisation", 1.0 when not given).
 * They are read as dequantisation scales: element codes times their head's
 * scale are the values attention runs on, i.e. the scores of qo head h (kv
 * head g) are sm_scale * scale_q[h] * scale_k[g] * q.k and its output is
 * scale_v[g] * sum_j softmax_j * v_j; lse is over those scores.
 *   q, k, v   device, the plan's q / kv data types (bsr_run's shapes and
 *             layouts; 8-bit codes for E4M3 / E5M2).
 *   scale_q, scale_k, scale_v  device float32 arrays, 4-byte aligned, or
 *             NULL (= 1.0 for every head).  Each scale must be positive and
 *             finite; other values give unspecified numbers (never a fault).
 *   out, lse  device, out of the plan's o_data_type; lse float32 or NULL.
 * On a plan whose data types are 16-bit, every scale must be NULL
 * (SFA_ERR_UNSUPPORTED otherwise) and this is bsr_run.  An FP8 plan with a
 * soft cap set returns SFA_ERR_UNSUPPORTED.  Other errors as bsr_run.
 */
sfa_status bsr_run_scaled(bsr_plan_t plan, const void* q, const void* k, const void* v,
                          const float* scale_q, const float* scale_k, const float* scale_v,
                          void* out, float* lse, sfa_stream_t stream);

/* Frees the plan's host state.  Safe on NULL.  Does not touch the
 * caller's workspaces. */
void bsr_plan_destroy(bsr_plan_t plan);

/* ------------------------------------------------------------------------ */
/* Variable block-sparse attention ("flashinfer.sparse",
 * VariableBlockSparseAttentionWrapper: blocks of any size given per kv head
 * by block_row_sz / block_col_sz, and each kv head its own block mask). */

typedef struct varbsr_plan_s* varbsr_plan_t;

/*
 * varbsr_plan -- validate the block mask map and sizes and build the device
 * work list (plan()).
 *
 *   block_mask_map_host  host bytes (num_kv_heads, MB, NB), row-major; a
 *                 nonzero byte marks block (row block, column block) of that
 *                 kv head as attended.
 *   block_row_sz_host    host int32 (num_kv_heads, MB), each >= 0; every kv
 *                 head's row sizes sum to the same qo_len >= 1.
 *   block_col_sz_host    host int32 (num_kv_heads, NB), each >= 0; every kv
 *                 head's column sizes sum to the same kv_len >= 1.
 *                 Query row i of qo head h attends key column j iff the
 *                 block of kv head g = h / (num_qo_heads / num_kv_heads)
 *                 holding (i, j) is set: row block b spans the rows after
 *                 the first b row sizes of g, column blocks likewise.
 *   MB, NB        number of row / column blocks (>= 1).
 *   num_qo_heads, num_kv_heads   num_qo_heads % num_kv_heads == 0; this
 *                 build needs 128 % (num_qo_heads / num_kv_heads) == 0
 *                 (SFA_ERR_UNSUPPORTED otherwise).
 *   head_dim      64 or 128 in this build (SFA_ERR_UNSUPPORTED otherwise).
 *   causal        nonzero: also key j <= i + (kv_len - qo_len) (the
 *                 bottom-right rule bsr_plan uses; the page does not state
 *                 the alignment for qo_len != kv_len).
 *   sm_scale      softmax scale; <= 0 selects 1/sqrt(head_dim).
 *   dtype         element type of q, k, v and out.
 *   int_ws        device buffer, 16-byte aligned, that the key tile lists
 *                 and work list are copied into (on `stream`); size from
 *                 varbsr_plan_int_workspace_size() with the same arguments.
 *   plan_out      receives a handle, valid until varbsr_plan_destroy(); the
 *                 workspace must stay allocated as long as it is used.
 * No float workspace: each work item keeps all of its keys in one CTA.
 * Errors: SFA_ERR_INVALID_ARG (NULL pointer, negative size, sizes that do not
 * sum alike, unaligned workspace), SFA_ERR_WORKSPACE (int_ws too small),
 * SFA_ERR_UNSUPPORTED, SFA_ERR_CUDA (the upload failed).
 */
sfa_status varbsr_plan(const uint8_t* block_mask_map_host, const int32_t* block_row_sz_host,
                       const int32_t* block_col_sz_host, int MB, int NB, int num_qo_heads,
                       int num_kv_heads, int head_dim, int causal, float sm_scale,
                       sfa_dtype dtype, void* int_ws, size_t int_ws_bytes, sfa_stream_t stream,
                       varbsr_plan_t* plan_out);

/* Bytes of int workspace varbsr_plan needs for these arguments.  Host only. */
sfa_status varbsr_plan_int_workspace_size(const uint8_t* block_mask_map_host,
                                          const int32_t* block_row_sz_host,
                                          const int32_t* block_col_sz_host, int MB, int NB,
                                          int num_qo_heads, int num_kv_heads, int head_dim,
                                          int causal, size_t* bytes);

/* qo_len and kv_len (the sums of the block sizes) of a plan.  Host only. */
sfa_status varbsr_plan_dims(varbsr_plan_t plan, int* qo_len, int* kv_len);

/*
 * varbsr_run -- variable block-sparse attention with a plan (run()).
 *   q    device (num_qo_heads, qo_len, head_dim), HND, dtype, 16-byte aligned.
 *   k, v device (num_kv_heads, kv_len, head_dim), HND, dtype.
 *   out  device (num_qo_heads, qo_len, head_dim), dtype: q's own layout (the
 *        page prints the return shape as [M, num_qo_heads, head_dim] but
 *        takes q as (num_qo_heads, qo_len, head_dim); read as q's layout).
 *   lse  device float32 (num_qo_heads, qo_len) or NULL: natural-log
 *        log-sum-exp of the scaled logits of the row's allowed columns.
 * Rows with no allowed column write out = +0 and lse = -inf.
 */
sfa_status varbsr_run(varbsr_plan_t plan, const void* q, const void* k, const void* v,
                      void* out, float* lse, sfa_stream_t stream);

/* varbsr_plan_set_logits_soft_cap -- plan()'s logits_soft_cap
 * (VariableBlockSparseAttentionWrapper.plan()), as
 * bsr_plan_set_logits_soft_cap.  Host only. */
sfa_status varbsr_plan_set_logits_soft_cap(varbsr_plan_t plan, float logits_soft_cap);

/* Frees the plan's host state.  Safe on NULL. */
void varbsr_plan_destroy(varbsr_plan_t plan);

#ifdef __cplusplus
}
#endif

#endif /* SFA_GB300_H */
