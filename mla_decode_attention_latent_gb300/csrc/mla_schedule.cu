// Tile scheduler: cuts the (sequence, page) range of a decode batch into
// contiguous split-KV parts of near-equal cost.
//
// The usage page "FlashMLA란 무엇인가?" (section "FlashMLA 설치 및 사용", step 2
// "MLA 메타데이터 가져오기") computes tile_scheduler_metadata and num_splits
// from cache_seqlens once per decode step; every layer then reuses them.  The
// page names the outputs only; the partition below is this library's:
//   n_b   = ceil(T_b / 64),  cost = sum_b (n_b + F),  F = fixed segment cost
//   quota = ceil(cost / parts) + F
//   walk the sequences with a cursor; a part finishes whole sequences while
//   (remaining pages + F) fits its budget, then takes (budget - F) pages of the
//   next sequence if that is positive; the last part takes the rest.
// Metadata row: {begin_seq, begin_page, end_seq, end_page, begin_split, 0, 0, 0}.
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kSchedThreads = 256;

__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const int32_t *__restrict__ seqlens, int batch, int num_parts,
                int32_t *__restrict__ metadata, int32_t *__restrict__ num_splits,
                unsigned int *status) {
    __shared__ long long s_cost[kSchedThreads];
    __shared__ int s_bad[kSchedThreads];

    // total cost, reduced over the block
    long long cost = 0;
    int bad = 0;
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int t = seqlens[b];
        if (t < 0) { bad = 1; t = 0; }
        cost += (t + kPage - 1) / kPage + kFixedCost;
    }
    s_cost[threadIdx.x] = cost;
    s_bad[threadIdx.x] = bad;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            s_cost[threadIdx.x] += s_cost[threadIdx.x + w];
            s_bad[threadIdx.x] |= s_bad[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x != 0) return;
    if (s_bad[0]) atomicOr(status, MLA_DEVERR_SEQLEN);

    const long long quota = (s_cost[0] + num_parts - 1) / num_parts + kFixedCost;
    int b = 0, page = 0, parts_on_b = 0;
    int splits_so_far = 0;
    num_splits[0] = 0;
    for (int p = 0; p < num_parts; ++p) {
        int32_t *row = metadata + (size_t)p * kMdInts;
        row[0] = b;
        row[1] = page;
        row[4] = parts_on_b;
        const bool last = (p == num_parts - 1);
        long long budget = quota;
        while (b < batch) {
            int t = seqlens[b];
            if (t < 0) t = 0;
            const long long remaining = (t + kPage - 1) / kPage - page;
            if (last || remaining + kFixedCost <= budget) {
                budget -= remaining + kFixedCost;
                splits_so_far += parts_on_b + 1;
                num_splits[b + 1] = splits_so_far;
                ++b;
                page = 0;
                parts_on_b = 0;
            } else {
                const long long take = budget - kFixedCost;
                if (take > 0) {
                    page += (int)take;
                    ++parts_on_b;
                }
                break;
            }
        }
        row[2] = b;
        row[3] = page;
        row[5] = 0;
        row[6] = 0;
        row[7] = 0;
    }
}

}  // namespace

cudaError_t launch_schedule(const int32_t *seqlens, int batch, int num_parts, int32_t *metadata,
                            int32_t *num_splits, unsigned int *status, cudaStream_t stream) {
    schedule_kernel<<<1, kSchedThreads, 0, stream>>>(seqlens, batch, num_parts, metadata, num_splits,
                                                     status);
    return cudaGetLastError();
}

}  // namespace mla
