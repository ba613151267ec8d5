// Block-sparse (BSR) attention: register-tiled FMA path for any block shape.
//
// "flashinfer.sparse", BlockSparseAttentionWrapper: query row i attends to
// key column j iff block (i / R, j / C) is stored (scipy bsr_matrix
// convention), GQA with qo head h reading kv head h / (Hq / Hkv).
//
// CTA = one row tile (<= 64 query rows of one block row) x one qo head,
// 256 threads as a 16 x 16 grid.  The block row's keys are the concatenation
// of its stored blocks' column ranges; they are processed in chunks of 64
// keys (any C: a chunk may span several blocks).  Per chunk: S = Q K^T as a
// 64 x 64 register-tiled product (each thread 4 x 4), online softmax per row
// (row max / sum across the 16 threads of a row), O += P V (each thread 4
// rows x d/16 columns).  plan()'s causal (bottom-right) and per-element mask
// set the masked scores to -inf before the softmax.
#include "common.cuh"
#include "internal.h"

namespace sfa {
namespace {

constexpr int kRows = 64;      // query rows per tile
constexpr int kKeys = 64;      // keys per chunk
constexpr int kThreads = 256;
constexpr int kSPad = 4;       // float padding of transposed tiles

struct BsrSmem {
    int q, k, v, p, cols, ecols, total;
};

__host__ __device__ inline BsrSmem bsr_smem(int d) {
    BsrSmem s;
    int off = 0;
    s.q = off;    off += d * (kRows + kSPad) * 4;   // q^T  [d][64 rows]
    s.k = off;    off += d * (kKeys + kSPad) * 4;   // k^T  [d][64 keys]
    s.v = off;    off += kKeys * d * 4;             // v    [64 keys][d]
    s.p = off;    off += kKeys * (kRows + kSPad) * 4;  // p^T [64 keys][64 rows]
    s.cols = off; off += kKeys * 4;
    s.ecols = off; off += kKeys * 4;   // mask bit of (row 0 of the block, key)
    s.total = off;
    return s;
}

template <class E, int D>
__global__ void __launch_bounds__(kThreads) bsr_generic_kernel(const BsrParams p) {
    using T = typename E::T;
    constexpr int CPT = D / 16;                 // output columns per thread
    extern __shared__ __align__(16) unsigned char smem[];
    const BsrSmem L = bsr_smem(D);
    float* qT = reinterpret_cast<float*>(smem + L.q);
    float* kT = reinterpret_cast<float*>(smem + L.k);
    float* vs = reinterpret_cast<float*>(smem + L.v);
    float* pT = reinterpret_cast<float*>(smem + L.p);
    int* cols = reinterpret_cast<int*>(smem + L.cols);
    int* ecols = reinterpret_cast<int*>(smem + L.ecols);
    constexpr int QLD = kRows + kSPad, KLD = kKeys + kSPad, PLD = kRows + kSPad;

    const BsrTile tile = p.tiles[blockIdx.x];
    const int h = blockIdx.y;
    const int kvh = h / (p.Hq / p.Hkv);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const T* qg = static_cast<const T*>(p.q);
    const T* kg = static_cast<const T*>(p.k);
    const T* vg = static_cast<const T*>(p.v);

    // Q tile, transposed, scaled by scale*log2(e); rows past the tile are 0.
    for (int e = tid; e < kRows * D; e += kThreads) {
        int r = e / D, dd = e % D;
        float x = 0.f;
        if (r < tile.nrows)
            x = E::to_f(qg[((int64_t)(tile.row0 + r) * p.Hq + h) * D + dd]) * p.scale_log2;
        qT[dd * QLD + r] = x;
    }

    const int blk0 = p.indptr[tile.rb], blk1 = p.indptr[tile.rb + 1];
    const int nkeys = (blk1 - blk0) * p.C;

    float m[4], l[4], o[4][CPT];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < CPT; ++c) o[i][c] = 0.f;
    }

    for (int k0 = 0; k0 < nkeys; k0 += kKeys) {
        const int nk = min(kKeys, nkeys - k0);
        __syncthreads();   // previous chunk fully consumed
        if (tid < kKeys) {
            int col = -1, ecol = 0;
            if (tid < nk) {
                const int pos = k0 + tid;
                const int kb = blk0 + pos / p.C, cc = pos % p.C;
                col = p.indices[kb] * p.C + cc;
                ecol = kb * p.R * p.C + cc;
            }
            cols[tid] = col;
            ecols[tid] = ecol;
        }
        __syncthreads();
        // K (transposed) and V chunk as fp32; missing keys are zero.
        for (int e = tid; e < kKeys * (D / 8); e += kThreads) {
            int j = e / (D / 8), piece = e % (D / 8);
            int col = cols[j];
            uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            if (col >= 0) {
                const int64_t off = (p.kv_hnd ? (int64_t)kvh * p.N + col
                                              : (int64_t)col * p.Hkv + kvh) * D + piece * 8;
                kv = *reinterpret_cast<const uint4*>(kg + off);
                vv = *reinterpret_cast<const uint4*>(vg + off);
            }
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
            const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float2 kf = E::unpack2(kw[w]);
                float2 vf = E::unpack2(vw[w]);
                int dd = piece * 8 + 2 * w;
                kT[dd * KLD + j] = kf.x;
                kT[(dd + 1) * KLD + j] = kf.y;
                vs[j * D + dd] = vf.x;
                vs[j * D + dd + 1] = vf.y;
            }
        }
        __syncthreads();

        // S tile: rows ty*4 .. +4, keys tx*4 .. +4
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
        for (int dd = 0; dd < D; ++dd) {
            float4 a = *reinterpret_cast<const float4*>(qT + dd * QLD + ty * 4);
            float4 bk = *reinterpret_cast<const float4*>(kT + dd * KLD + tx * 4);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {bk.x, bk.y, bk.z, bk.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] += av[i] * bv[j];
        }
        // online softmax per row (16 threads share a row group)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float cm = -INFINITY;
            const int rl = ty * 4 + i;                    // row of the tile
            const int rin = tile.row0 + rl - tile.rb * p.R;    // row inside its block
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kj = tx * 4 + j;
                // logits soft cap (scores are already in log2 units)
                if (p.softcap_log2 > 0.f)
                    s[i][j] = soft_cap_log2(s[i][j], p.softcap_log2, 1.f / p.softcap_log2);
                if (kj >= nk) {
                    s[i][j] = -INFINITY;
                } else if (p.mask_mode != 0 && rl < tile.nrows) {
                    bool ok;
                    if (p.mask_mode == 1) {
                        ok = (int64_t)cols[kj] <= (int64_t)(tile.row0 + rl) + (p.N - p.M);
                    } else {
                        const int e = ecols[kj] + rin * p.C;
                        ok = ((p.mask[e >> 3] >> (7 - (e & 7))) & 1) != 0;
                    }
                    if (!ok) s[i][j] = -INFINITY;
                }
                cm = fmaxf(cm, s[i][j]);
            }
#pragma unroll
            for (int o2 = 8; o2 > 0; o2 >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
            const float m_new = fmaxf(m[i], cm);
            const float alpha = rescale_factor(m[i], m_new);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float pj = (s[i][j] == -INFINITY) ? 0.f : fast_exp2(s[i][j] - m_new);
                rs += pj;
                pT[(tx * 4 + j) * PLD + ty * 4 + i] = pj;
            }
#pragma unroll
            for (int o2 = 8; o2 > 0; o2 >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o2);
            l[i] = l[i] * alpha + rs;
            m[i] = m_new;
#pragma unroll
            for (int c = 0; c < CPT; ++c) o[i][c] *= alpha;
        }
        __syncthreads();
        // O += P V : rows ty*4 .. +4, columns tx*CPT .. +CPT
        for (int j = 0; j < nk; ++j) {
            float4 pa = *reinterpret_cast<const float4*>(pT + j * PLD + ty * 4);
            const float pv[4] = {pa.x, pa.y, pa.z, pa.w};
            const float* vrow = vs + j * D + tx * CPT;
#pragma unroll
            for (int c = 0; c < CPT; c += 4) {
                float4 vv = *reinterpret_cast<const float4*>(vrow + c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[i][c] += pv[i] * vv.x;
                    o[i][c + 1] += pv[i] * vv.y;
                    o[i][c + 2] += pv[i] * vv.z;
                    o[i][c + 3] += pv[i] * vv.w;
                }
            }
        }
    }

    // epilogue
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= tile.nrows) continue;
        const int64_t row = tile.row0 + r;
        T* orow = static_cast<T*>(p.out) + (row * p.Hq + h) * D + tx * CPT;
        const bool empty = !(l[i] > 0.f);
        const float inv = empty ? 0.f : 1.f / l[i];
#pragma unroll
        for (int c = 0; c < CPT; c += 2) {
            uint32_t packed = empty ? 0u : E::pack2(o[i][c] * inv, o[i][c + 1] * inv);
            *reinterpret_cast<uint32_t*>(orow + c) = packed;
        }
        if (p.lse && tx == 0)
            p.lse[row * p.Hq + h] = empty ? -INFINITY : (m[i] + __log2f(l[i])) * kLn2;
    }
}

template <class E, int D>
cudaError_t launch_bsr_t(const BsrParams& p, cudaStream_t stream) {
    const BsrSmem L = bsr_smem(D);
    auto kern = bsr_generic_kernel<E, D>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)p.ntiles, (unsigned)p.Hq);
    kern<<<grid, kThreads, L.total, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

template <class E>
cudaError_t launch_bsr_e(const BsrParams& p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_bsr_t<E, 64>(p, stream);
        case 128: return launch_bsr_t<E, 128>(p, stream);
        case 192: return launch_bsr_t<E, 192>(p, stream);
        case 256: return launch_bsr_t<E, 256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_bsr_generic(const BsrParams& p, sfa_dtype dtype, cudaStream_t stream) {
    if (p.ntiles == 0) return cudaSuccess;
    return dtype == SFA_DTYPE_BF16 ? launch_bsr_e<BF16>(p, stream) : launch_bsr_e<F16>(p, stream);
}

}  // namespace sfa
