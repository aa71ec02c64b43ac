// Combine: merges the split-KV partial results of a sequence, weighted by
// their log-sum-exp.
//
// A sequence cut into k parts (num_splits[b+1] - num_splits[b] = k > 1, see
// mla_get_metadata) leaves, for every query row, k partial outputs O_s (each
// normalised by its own softmax sum) and partial LSEs L_s.  The exact result
// is
//   L = ln sum_s exp(L_s)            (computed with the max shifted out)
//   O = sum_s exp(L_s - L) * O_s
// which is the decode call's o and lse ("FlashMLA란 무엇인가?", section
// "FlashMLA 설치 및 사용", step 3: the call returns o_i and lse_i; num_splits is
// the scheduler output of step 2).  Partials with L_s = -inf (no visible key in
// that part) carry weight 0; a row with no visible key anywhere gets O = 0 and
// L = -inf.
//
// One warp per (sequence, row).  Lane s holds the partial LSE of partial s,
// so the LSEs are read once; the weights travel by shuffle.  Each lane owns
// 16 of the 512 output dims as four float4 groups at lane*4 + 128*k, so every
// warp load is 512 contiguous bytes, and the loads of two partials are in
// flight together.  Memory-bound: reads k * 2 KB of partials, writes 1 KB of
// bf16.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mla_sm103.cuh"

namespace mla {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineUnroll = 2;  // partials whose loads are in flight together

__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float *__restrict__ o_accum, const float *__restrict__ lse_accum,
               const int32_t *__restrict__ num_splits, int rows, int max_splits,
               uint16_t *__restrict__ o, float *__restrict__ lse, unsigned int *status) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    const int b = blockIdx.y;
    sm103::griddep_wait();  // the split-KV kernel's partials (programmatic launch)
    if (row >= rows) return;
    const int first = num_splits[b];
    const int n = num_splits[b + 1] - first;
    if (n <= 1) return;  // written directly by the split-KV kernel
    if (first < 0 || first + n > max_splits) {
        if (lane == 0) atomicOr(status, MLA_DEVERR_SEQLEN);
        return;
    }

    // lane s keeps L_s of partial s (partials past 32 are read again below)
    const float l_own = lane < n ? lse_accum[(size_t)(first + lane) * rows + row] : -CUDART_INF_F;
    float m = l_own;
    for (int s = lane + 32; s < n; s += 32) m = fmaxf(m, lse_accum[(size_t)(first + s) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

    const size_t out_row = (size_t)b * rows + row;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float total_lse = -CUDART_INF_F;
    if (m != -CUDART_INF_F) {
        float sum = lane < n ? __expf(l_own - m) : 0.f;
        for (int s = lane + 32; s < n; s += 32) sum += __expf(lse_accum[(size_t)(first + s) * rows + row] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        total_lse = m + __logf(sum);
        const float w_own = lane < n ? __expf(l_own - total_lse) : 0.f;
        for (int s0 = 0; s0 < n; s0 += kCombineUnroll) {
            float w[kCombineUnroll];
            float4 v[kCombineUnroll][4];
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u) {
                const int s = s0 + u;  // uniform across the warp
                const size_t slot = (size_t)(first + (s < n ? s : 0)) * rows + row;
                w[u] = s < 32 ? __shfl_sync(0xffffffffu, w_own, s & 31) : __expf(lse_accum[slot] - total_lse);
                if (s >= n) w[u] = 0.f;
                const float4 *src = reinterpret_cast<const float4 *>(o_accum + slot * kDv);
#pragma unroll
                for (int k = 0; k < 4; ++k) v[u][k] = s < n ? src[lane + 32 * k] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[k].x += w[u] * v[u][k].x;
                    acc[k].y += w[u] * v[u][k].y;
                    acc[k].z += w[u] * v[u][k].z;
                    acc[k].w += w[u] * v[u][k].w;
                }
        }
    }
    uint2 *dst = reinterpret_cast<uint2 *>(o + out_row * kDv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        dst[lane + 32 * k] = pk;
    }
    if (lane == 0) lse[out_row] = total_lse;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.rows + kCombineWarps - 1) / kCombineWarps, p.batch, 1);
    cfg.blockDim = dim3(kCombineWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // launch overlaps the split kernel's tail
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, (const float *)p.o_accum, (const float *)p.lse_accum,
                              (const int32_t *)p.num_splits, p.rows, p.max_splits, p.o, p.lse, p.status);
}

}  // namespace mla
