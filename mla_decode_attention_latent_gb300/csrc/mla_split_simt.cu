// Split-KV MLA decode, SIMT form: one warp per query row, fp32 online softmax.
//
// This is the plain CUDA-core formulation of the split-KV step (no tensor
// cores).  It walks the same work partition and writes the same outputs and
// partials as the tensor-core kernel, and serves as a second, independent GPU
// implementation of the step.
//
// Per (part, 8-row block): for each segment (sequence b, pages [p0, p1)) of
// the part, every warp owns one query row r = i * h_q + h and streams the keys
// j < min(64 * p1, T_row), T_row = T_b (or T_b - s_q + i + 1 when causal):
//   s    = scale * log2(e) * <q_r, k_j>           (warp-reduced dot product)
//   m'   = max(m, s);  l = l * 2^(m - m') + 2^(s - m');  acc = acc * 2^(m - m') + 2^(s - m') * v_j
// and at the end of the segment writes O = acc / l and LSE = ln 2 * (m + log2 l),
// to the output when the sequence is not split, else to the partial slot
// num_splits[b] + split index.  Lane l holds dims [16 l, 16 l + 16) of the
// latent part (also its V dims) and RoPE dims 512 + [2 l, 2 l + 2).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kSimtWarps = 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kSimtWarps * 32)
split_kv_simt_kernel(const DecodeParams p) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.y * kSimtWarps + (threadIdx.x >> 5);
    if (r >= p.rows) return;
    const int part = blockIdx.x;
    const int32_t *md = p.metadata + (size_t)part * kMdInts;
    const int bb = md[0], bp = md[1], eb = md[2], ep = md[3], bs = md[4];
    if (bb == eb && bp == ep) return;
    const int qi = r / p.h_q;  // query token index within the step

    for (int b = bb; b < p.batch; ++b) {
        if (b == eb && ep == 0) break;
        int T = p.seqlens[b];
        if (T < 0 || T > p.max_blocks * kPage) {
            if (lane == 0) atomicOr(p.status, MLA_DEVERR_SEQLEN);
            T = T < 0 ? 0 : p.max_blocks * kPage;
        }
        const int n_pages = (T + kPage - 1) / kPage;
        const int p0 = (b == bb) ? bp : 0;
        const int p1 = (b == eb) ? ep : n_pages;
        const int split = (b == bb) ? bs : 0;
        const int n_split = p.num_splits[b + 1] - p.num_splits[b];
        const int T_row = p.causal ? T - p.s_q + qi + 1 : T;
        const int j_end = min(p1 * kPage, T_row);

        // query row: 16 latent dims + 2 RoPE dims per lane, as fp32
        const uint16_t *qrow = p.q + ((size_t)b * p.rows + r) * kDqk;
        float qv[18];
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(qrow + 16 * lane);
            const uint4 a = src[0], c = src[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                qv[2 * k] = bf16_lo(w[k]);
                qv[2 * k + 1] = bf16_hi(w[k]);
            }
            const uint32_t rw = *reinterpret_cast<const uint32_t *>(qrow + 512 + 2 * lane);
            qv[16] = bf16_lo(rw);
            qv[17] = bf16_hi(rw);
        }

        float m = -CUDART_INF_F, l = 0.f;
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;

        for (int j = p0 * kPage; j < j_end; ++j) {
            const int blk = p.block_table[(size_t)b * p.max_blocks + j / kPage];
            if (blk < 0 || blk >= p.num_blocks) {
                if (lane == 0) atomicOr(p.status, MLA_DEVERR_BLOCK_ID);
                continue;
            }
            const uint16_t *krow = p.kcache + ((size_t)blk * kPage + (j % kPage)) * kDqk;
            const uint4 *src = reinterpret_cast<const uint4 *>(krow + 16 * lane);
            const uint4 a = src[0], c = src[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
            const uint32_t rw = *reinterpret_cast<const uint32_t *>(krow + 512 + 2 * lane);
            float kv[16];
            float dot = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                kv[2 * k] = bf16_lo(w[k]);
                kv[2 * k + 1] = bf16_hi(w[k]);
                dot = fmaf(qv[2 * k], kv[2 * k], dot);
                dot = fmaf(qv[2 * k + 1], kv[2 * k + 1], dot);
            }
            dot = fmaf(qv[16], bf16_lo(rw), dot);
            dot = fmaf(qv[17], bf16_hi(rw), dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float s = dot * p.scale_log2;
            const float m_new = fmaxf(m, s);
            const float alpha = exp2f(m - m_new);  // m = -inf on the first key: alpha = 0
            const float pj = exp2f(s - m_new);
            l = l * alpha + pj;
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = fmaf(pj, kv[k], acc[k] * alpha);
            m = m_new;
        }

        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse_row = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
        if (n_split <= 1) {
            const size_t out = (size_t)b * p.rows + r;
            uint4 pk[2];
            uint32_t *pw = reinterpret_cast<uint32_t *>(pk);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * k] * inv_l, acc[2 * k + 1] * inv_l);
                pw[k] = *reinterpret_cast<uint32_t *>(&h2);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + out * kDv + 16 * lane);
            dst[0] = pk[0];
            dst[1] = pk[1];
            if (lane == 0) p.lse[out] = lse_row;
        } else {
            const int slot = p.num_splits[b] + split;
            if (slot < 0 || slot >= p.max_splits) {
                if (lane == 0) atomicOr(p.status, MLA_DEVERR_SEQLEN);
            } else {
                const size_t idx = (size_t)slot * p.rows + r;
                float4 *dst = reinterpret_cast<float4 *>(p.o_accum + idx * kDv + 16 * lane);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dst[k] = make_float4(acc[4 * k] * inv_l, acc[4 * k + 1] * inv_l, acc[4 * k + 2] * inv_l,
                                         acc[4 * k + 3] * inv_l);
                if (lane == 0) p.lse_accum[idx] = lse_row;
            }
        }
        if (b == eb) break;
    }
}

}  // namespace

cudaError_t launch_split_kv_simt(const DecodeParams &p, cudaStream_t stream) {
    dim3 grid(p.num_parts, (p.rows + kSimtWarps - 1) / kSimtWarps);
    split_kv_simt_kernel<<<grid, kSimtWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mla
