// Generic top-K sparse flash attention: warp-level FMA path.
//
// "SparseFlashAttention 算子 API 描述", §2 具体子步骤: gather the selected K/V
// rows, scaled dot product, bottom-right causal mask, softmax over the topK
// slots, weighted sum.  This kernel evaluates the softmax online (running
// max and sum per query head, rescaling the partial output), which is the
// same function in exact arithmetic, and can split the topK slots of a row
// across CTAs; sfa_combine_kernel merges the split partials.
//
// CTA = one (b, n2, s1) index list x one block of HB query heads x one slot
// range.  4 warps.  Per 32-slot chunk: the selected K (and V) rows are copied
// into shared memory with 16-byte cp.async (two stages, so the gather of
// chunk c+1 overlaps the math of chunk c); lane j of each warp scores slot j
// against the warp's heads; each warp then updates its heads' softmax state
// and accumulates P.V with lanes owning output columns.
#include "common.cuh"
#include "internal.h"

namespace sfa {
namespace {

constexpr int kChunk = 32;     // slots per pipeline stage (one per lane)
constexpr int kWarps = 4;
constexpr int kPad = 8;        // elements of padding per smem row (16 bytes)
constexpr int kMaxDk = 576;
constexpr int kMaxDv = 512;

struct GenericSmem {
    // byte offsets inside dynamic shared memory
    int q, k, v, idx, p, total;
};

__host__ __device__ inline GenericSmem generic_smem(int HB, int Dk, int Dv, bool v_in_k) {
    GenericSmem s;
    int off = 0;
    s.q = off;   off += HB * Dk * 4;
    s.k = off;   off += 2 * kChunk * (Dk + kPad) * 2;
    s.v = off;   off += v_in_k ? 0 : 2 * kChunk * (Dv + kPad) * 2;
    s.idx = off; off += 2 * kChunk * 4;
    s.p = off;   off += HB * kChunk * 4;
    s.total = off;
    return s;
}

template <class E, int HPW>
__global__ void __launch_bounds__(kWarps * 32)
sfa_generic_kernel(const SfaParams p, const int v_in_k) {
    using T = typename E::T;
    constexpr int HB = HPW * kWarps;
    extern __shared__ __align__(16) unsigned char smem[];
    const GenericSmem L = generic_smem(HB, p.Dk, p.Dv, v_in_k);
    float* q_s = reinterpret_cast<float*>(smem + L.q);
    T* k_s = reinterpret_cast<T*>(smem + L.k);
    T* v_s = reinterpret_cast<T*>(smem + L.v);
    int* idx_s = reinterpret_cast<int*>(smem + L.idx);
    float* p_s = reinterpret_cast<float*>(smem + L.p);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // unit = (b, n2, s1)
    const int unit = blockIdx.x;
    const int s1 = unit % p.S1;
    const int n2 = (unit / p.S1) % p.N2;
    const int b = unit / (p.S1 * p.N2);
    const int g0 = blockIdx.y * HB;                      // first head of the block (in group)
    const int nh = min(HB, p.G - g0);
    const int split = blockIdx.z;
    const int slot_begin = split * p.slots_per_split;
    const int slot_end = min(p.topK, slot_begin + p.slots_per_split);
    const int diag = s1 + (p.S2 - p.S1);

    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k) + b * p.k_sb + n2 * p.k_sh;
    const T* vg = static_cast<const T*>(p.v) + b * p.v_sb + n2 * p.v_sh;
    const int32_t* ig = p.idx + b * p.i_sb + n2 * p.i_sh + s1 * p.i_ss;
    const int ks_ld = p.Dk + kPad;
    const int vs_ld = v_in_k ? ks_ld : p.Dv + kPad;

    // q rows of the block's heads, scaled by scale*log2(e), as fp32.
    for (int e = tid; e < HB * p.Dk; e += blockDim.x) {
        int h = e / p.Dk, d = e % p.Dk;
        float x = 0.f;
        if (h < nh) {
            int n1 = n2 * p.G + g0 + h;
            x = E::to_f(qg[b * p.q_sb + n1 * p.q_sh + s1 * p.q_ss + d]) * p.scale_log2;
        }
        q_s[e] = x;
    }

    // Gather of one chunk into stage `st`.
    auto load_chunk = [&](int c, int st) {
        const int base = slot_begin + c * kChunk;
        if (tid < kChunk) {
            int slot = base + tid;
            int id = -1;
            if (slot < slot_end) {
                id = ig[slot];
                if (id < 0 || id >= p.S2) {
                    if (p.validate) atomicOr(p.err_word, 1);
                    id = -1;
                }
            }
            idx_s[st * kChunk + tid] = id;
        }
        const int kpr = p.Dk / 8;                       // 16-byte pieces per K row
        for (int e = tid; e < kChunk * kpr; e += blockDim.x) {
            int j = e / kpr, piece = e % kpr;
            int slot = base + j;
            int id = (slot < slot_end) ? ig[slot] : -1;
            bool ok = id >= 0 && id < p.S2;
            const T* src = kg + (ok ? (int64_t)id * p.k_ss : 0) + piece * 8;
            cp_async_16_zfill(k_s + (st * kChunk + j) * ks_ld + piece * 8, src, ok ? 16 : 0);
        }
        if (!v_in_k) {
            const int vpr = p.Dv / 8;
            for (int e = tid; e < kChunk * vpr; e += blockDim.x) {
                int j = e / vpr, piece = e % vpr;
                int slot = base + j;
                int id = (slot < slot_end) ? ig[slot] : -1;
                bool ok = id >= 0 && id < p.S2;
                const T* src = vg + (ok ? (int64_t)id * p.v_ss : 0) + piece * 8;
                cp_async_16_zfill(v_s + (st * kChunk + j) * vs_ld + piece * 8, src, ok ? 16 : 0);
            }
        }
        cp_async_commit();
    };

    // Per-warp softmax state and output accumulators (lane owns columns
    // 2*lane + 64*t, t < Dv/64).
    constexpr int kMaxPairs = kMaxDv / 64;
    float m[HPW], l[HPW];
    float2 o[HPW][kMaxPairs];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxPairs; ++t) o[hh][t] = make_float2(0.f, 0.f);
    }
    const int npairs = p.Dv / 64;

    const int nslots = max(slot_end - slot_begin, 0);
    const int nchunks = (nslots + kChunk - 1) / kChunk;
    if (nchunks > 0) load_chunk(0, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        if (c + 1 < nchunks) {
            load_chunk(c + 1, st ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // ---- scores: lane = slot ----
        const T* krow = k_s + (st * kChunk + lane) * ks_ld;
        float acc[HPW];
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) acc[hh] = 0.f;
        for (int d = 0; d < p.Dk; d += 8) {
            uint4 kv = *reinterpret_cast<const uint4*>(krow + d);
            float2 k0 = E::unpack2(kv.x), k1 = E::unpack2(kv.y);
            float2 k2 = E::unpack2(kv.z), k3 = E::unpack2(kv.w);
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) {
                const float* qr = q_s + (warp * HPW + hh) * p.Dk + d;
                float4 qa = *reinterpret_cast<const float4*>(qr);
                float4 qb = *reinterpret_cast<const float4*>(qr + 4);
                acc[hh] += qa.x * k0.x + qa.y * k0.y + qa.z * k1.x + qa.w * k1.y +
                           qb.x * k2.x + qb.y * k2.y + qb.z * k3.x + qb.w * k3.y;
            }
        }
        const int id = idx_s[st * kChunk + lane];
        const bool visible = id >= 0 && !(p.causal && id > diag);

        // ---- online softmax per head, then P.V ----
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const float s = visible ? acc[hh] : -INFINITY;
            const float m_new = fmaxf(m[hh], warp_max(s));
            const float alpha = rescale_factor(m[hh], m_new);
            const float pj = visible ? fast_exp2(s - m_new) : 0.f;
            l[hh] = l[hh] * alpha + warp_sum(pj);
            m[hh] = m_new;
            p_s[(warp * HPW + hh) * kChunk + lane] = pj;
#pragma unroll
            for (int t = 0; t < kMaxPairs; ++t) {
                o[hh][t].x *= alpha;
                o[hh][t].y *= alpha;
            }
        }
        __syncwarp();
        const T* vbase = (v_in_k ? k_s : v_s) + (st * kChunk) * vs_ld + 2 * lane;
        for (int j = 0; j < kChunk; ++j) {
            const T* vrow = vbase + j * vs_ld;
            float pj[HPW];
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) pj[hh] = p_s[(warp * HPW + hh) * kChunk + j];
#pragma unroll
            for (int t = 0; t < kMaxPairs; ++t) {
                if (t < npairs) {
                    float2 vv = E::unpack2(*reinterpret_cast<const uint32_t*>(vrow + 64 * t));
#pragma unroll
                    for (int hh = 0; hh < HPW; ++hh) {
                        o[hh][t].x += pj[hh] * vv.x;
                        o[hh][t].y += pj[hh] * vv.y;
                    }
                }
            }
        }
        __syncthreads();   // stage st is refilled by the next iteration's load
    }

    // ---- epilogue ----
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int h = warp * HPW + hh;
        if (h >= nh) continue;
        const int g = g0 + h;
        const int n1 = n2 * p.G + g;
        if (p.splits == 1) {
            T* orow = static_cast<T*>(p.out) + b * p.o_sb + n1 * p.o_sh + s1 * p.o_ss;
            const float inv = (l[hh] > 0.f) ? 1.f / l[hh] : 0.f;
#pragma unroll
            for (int t = 0; t < kMaxPairs; ++t) {
                if (t < npairs) {
                    uint32_t packed = (l[hh] > 0.f) ? E::pack2(o[hh][t].x * inv, o[hh][t].y * inv)
                                                    : 0u;
                    *reinterpret_cast<uint32_t*>(orow + 2 * lane + 64 * t) = packed;
                }
            }
            if (p.lse && lane == 0) {
                p.lse[b * p.l_sb + n1 * p.l_sh + s1 * p.l_ss] =
                    (l[hh] > 0.f) ? (m[hh] + __log2f(l[hh])) * kLn2 : -INFINITY;
            }
        } else {
            const int64_t row = (int64_t)unit * p.G + g;
            float* wo = p.ws_o + (row * p.splits + split) * p.Dv;
#pragma unroll
            for (int t = 0; t < kMaxPairs; ++t)
                if (t < npairs) *reinterpret_cast<float2*>(wo + 2 * lane + 64 * t) = o[hh][t];
            if (lane == 0) {
                p.ws_ml[(row * p.splits + split) * 2 + 0] = m[hh];
                p.ws_ml[(row * p.splits + split) * 2 + 1] = l[hh];
            }
        }
    }
}

// Merge of the split partials of one output row:
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p O_p / sum_p w_p l_p,
//   lse = (M + log2 sum_p w_p l_p) * ln 2.  No visible slot in any split: +0, -inf.
template <class E>
__global__ void __launch_bounds__(128) sfa_combine_kernel(const SfaParams p) {
    using T = typename E::T;
    const int64_t row = blockIdx.x;                 // ((b*N2 + n2)*S1 + s1)*G + g
    const int g = row % p.G;
    const int64_t unit = row / p.G;
    const int s1 = unit % p.S1;
    const int n2 = (unit / p.S1) % p.N2;
    const int b = unit / ((int64_t)p.S1 * p.N2);
    const int n1 = n2 * p.G + g;
    const float* ml = p.ws_ml + row * p.splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, ml[2 * s]);
    float Lsum = 0.f;
    for (int s = 0; s < p.splits; ++s) Lsum += rescale_factor(ml[2 * s], M) * ml[2 * s + 1];
    const bool empty = !(Lsum > 0.f);
    const float inv = empty ? 0.f : 1.f / Lsum;
    T* orow = static_cast<T*>(p.out) + b * p.o_sb + n1 * p.o_sh + s1 * p.o_ss;
    const float* wo = p.ws_o + row * p.splits * p.Dv;
    for (int e = threadIdx.x; e < p.Dv; e += blockDim.x) {
        float acc = 0.f;
        if (!empty)
            for (int s = 0; s < p.splits; ++s)
                acc += rescale_factor(ml[2 * s], M) * wo[(int64_t)s * p.Dv + e];
        orow[e] = empty ? E::from_f(0.f) : E::from_f(acc * inv);
    }
    if (p.lse && threadIdx.x == 0)
        p.lse[b * p.l_sb + n1 * p.l_sh + s1 * p.l_ss] =
            empty ? -INFINITY : (M + __log2f(Lsum)) * kLn2;
}

template <class E, int HPW>
cudaError_t launch_generic_t(const SfaParams& p, cudaStream_t stream) {
    const bool v_in_k = (p.v == p.k) && (p.v_ss == p.k_ss);
    const GenericSmem L = generic_smem(HPW * kWarps, p.Dk, p.Dv, v_in_k);
    auto kern = sfa_generic_kernel<E, HPW>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)(p.B * p.N2 * p.S1), (unsigned)((p.G + HPW * kWarps - 1) / (HPW * kWarps)),
              (unsigned)p.splits);
    kern<<<grid, kWarps * 32, L.total, stream>>>(p, v_in_k ? 1 : 0);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

size_t counter_region_bytes(int64_t) {
    // fixed size, so that calls of different shapes sharing a workspace never
    // place other data where another call keeps its counters
    return (size_t)kMaxCounters * sizeof(unsigned);
}

size_t sfa_split_ws_bytes(int64_t rows, int splits, int Dv) {
    if (splits <= 1) return 0;
    return (size_t)rows * splits * ((size_t)Dv + 2) * sizeof(float);
}

cudaError_t launch_sfa_generic(const SfaParams& p, sfa_dtype dtype, cudaStream_t stream) {
    if (p.Dk > kMaxDk || p.Dv > kMaxDv) return cudaErrorInvalidValue;
    const bool two = p.G > 4;
    if (dtype == SFA_DTYPE_BF16)
        return two ? launch_generic_t<BF16, 2>(p, stream) : launch_generic_t<BF16, 1>(p, stream);
    return two ? launch_generic_t<F16, 2>(p, stream) : launch_generic_t<F16, 1>(p, stream);
}

cudaError_t launch_sfa_combine(const SfaParams& p, sfa_dtype dtype, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.N2 * p.S1 * p.G;
    if (dtype == SFA_DTYPE_BF16)
        sfa_combine_kernel<BF16><<<(unsigned)rows, 128, 0, stream>>>(p);
    else
        sfa_combine_kernel<F16><<<(unsigned)rows, 128, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sfa
