// Tile scheduler: cuts the (sequence, page) range of a decode batch into
// contiguous split-KV parts of near-equal cost.
//
// The usage page "FlashMLA란 무엇인가?" (section "FlashMLA 설치 및 사용", step 2
// "MLA 메타데이터 가져오기") computes tile_scheduler_metadata and num_splits
// from cache_seqlens once per decode step; every layer then reuses them.  The
// page names the outputs only; the partition below is this library's:
//   lay the sequences on one line of cost units, sequence b taking
//   c_b = F + n_b units (F = fixed cost of a segment, a call argument; n_b = ceil(T_b / 64)
//   pages) from S_b = c_0 + ... + c_{b-1}; Q = ceil(total / parts); part p
//   starts at unit p * Q.  A unit in a sequence's first F units maps to its
//   page 0, a later one to page (x - S_b - F); the last part ends at
//   (batch, 0).  A part that starts inside a sequence's pages pays F beyond
//   its Q units, so no part costs more than Q + F.
// Every part's bounds are independent of the others' (two binary searches
// over the prefix sums), so the whole partition is computed in parallel.
// Metadata row: {begin_seq, begin_page, end_seq, end_page, begin_split, 0, 0, 0}.
#include "mla_internal.h"
#include "mla_sm103.cuh"

namespace mla {
namespace {

constexpr int kSchedThreads = 512;

__device__ __forceinline__ int pages_of(int t) { return t <= 0 ? 0 : t / kPage + (t % kPage != 0); }

// Exclusive prefix sum over the block; *total receives the block total.
template <typename T>
__device__ T block_exclusive_scan(T v, T *s_warp, T *total) {
    constexpr int kWarps = kSchedThreads / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        T y = lane < kWarps ? s_warp[lane] : T(0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const T z = __shfl_up_sync(0xffffffffu, y, off);
            if (lane >= off) y += z;
        }
        if (lane < kWarps) s_warp[lane] = y;
    }
    __syncthreads();
    const T base = w > 0 ? s_warp[w - 1] : T(0);
    *total = s_warp[kWarps - 1];
    __syncthreads();  // s_warp may be reused right after
    return base + x - v;
}

// One CTA.  Thread t owns the contiguous chunk of sequences
// [t * chunk, (t + 1) * chunk); a scan of the chunk costs gives every chunk's
// first unit, so a unit is located by a binary search over the chunks and a
// short walk inside one.
__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const int32_t *__restrict__ seqlens, int batch, int num_parts, int fixed_cost, int combine_cost,
                int32_t *__restrict__ metadata, int32_t *__restrict__ num_splits,
                unsigned int *status) {
    __shared__ long long s_start[kSchedThreads + 1];  // first unit of every chunk; [kSchedThreads] = total
    __shared__ long long s_warp64[kSchedThreads / 32];
    __shared__ int s_warp32[kSchedThreads / 32];

    // the split-KV launch that follows may start its prologue now; it waits
    // for this grid to complete before it reads the partition
    if (threadIdx.x == 0) sm103::griddep_launch_dependents();
    const int chunk = (batch + kSchedThreads - 1) / kSchedThreads;
    const int i0 = min(threadIdx.x * chunk, batch), i1 = min(i0 + chunk, batch);
    long long cost = 0;
    bool bad = false;
    for (int i = i0; i < i1; ++i) {
        const int t = seqlens[i];
        bad |= t < 0;
        cost += pages_of(t) + fixed_cost;
    }
    if (bad) atomicOr(status, MLA_DEVERR_SEQLEN);
    long long total;
    const long long first_unit = block_exclusive_scan(cost, s_warp64, &total);
    s_start[threadIdx.x] = first_unit;
    if (threadIdx.x == 0) s_start[kSchedThreads] = total;

    // how many parts get work: all of them, or one per sequence when the
    // batch is smaller and that is estimated to finish sooner.  A candidate
    // with quota q costs q, plus F + C when a part would start strictly
    // inside some sequence's pages (a multiple of q in (S_b + F, S_{b+1})).
    const long long q_all = (total + num_parts - 1) / num_parts;  // total >= batch * F > 0
    const long long q_seq = (total + batch - 1) / batch;
    bool cut_all = false, cut_seq = false;
    if (batch < num_parts) {
        long long u = first_unit;
        for (int i = i0; i < i1; ++i) {
            const int n = pages_of(seqlens[i]);
            const long long next = u + n + fixed_cost;
            if (n > 0) {
                cut_all |= (next - 1) / q_all > (u + fixed_cost) / q_all;
                cut_seq |= (next - 1) / q_seq > (u + fixed_cost) / q_seq;
            }
            u = next;
        }
    }
    cut_all = __syncthreads_or(cut_all);
    cut_seq = __syncthreads_or(cut_seq);
    const long long est_all = q_all + (cut_all ? fixed_cost + combine_cost : 0);
    const long long est_seq = q_seq + (cut_seq ? fixed_cost + combine_cost : 0);
    const long long quota = (batch < num_parts && est_seq < est_all) ? q_seq : q_all;

    // cursor of unit x: sequence b, page, and S_b
    auto cursor = [&](long long x, int &b, int &pg, long long &sb) {
        if (x >= total) {
            b = batch;
            pg = 0;
            sb = total;
            return;
        }
        int lo = 0, hi = kSchedThreads;  // s_start[lo] <= x < s_start[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_start[mid] <= x) lo = mid;
            else hi = mid;
        }
        long long u = s_start[lo];
        int i = lo * chunk;
        while (true) {
            const long long c = pages_of(seqlens[i]) + fixed_cost;
            if (x < u + c) break;
            u += c;
            ++i;
        }
        b = i;
        sb = u;
        const long long off = x - u;
        pg = off <= fixed_cost ? 0 : (int)(off - fixed_cost);
    };

    for (int p = threadIdx.x; p < num_parts; p += kSchedThreads) {
        int b0, pg0, b1 = batch, pg1 = 0;
        long long s0, s1;
        cursor((long long)p * quota, b0, pg0, s0);
        if (p + 1 < num_parts) cursor((long long)(p + 1) * quota, b1, pg1, s1);
        // parts touching b0 before p: the one holding its page 0, then every
        // part that started inside its pages (the first at floor((S + F) / Q) + 1)
        const int split0 = pg0 > 0 ? (int)(p - (s0 + fixed_cost) / quota) : 0;
        int32_t *row = metadata + (size_t)p * kMdInts;  // 4-byte alignment is all the caller promises
        row[0] = b0;
        row[1] = pg0;
        row[2] = b1;
        row[3] = pg1;
        row[4] = split0;
        row[5] = 0;
        row[6] = 0;
        row[7] = 0;
    }

    // parts touching sequence b: 1 + the part starts strictly inside its pages
    int segs = 0;
    {
        long long u = first_unit;
        for (int i = i0; i < i1; ++i) {
            const int n = pages_of(seqlens[i]);
            const long long next = u + n + fixed_cost;
            segs += 1 + (n > 0 ? (int)((next - 1) / quota - (u + fixed_cost) / quota) : 0);
            u = next;
        }
    }
    int all;
    int run = block_exclusive_scan(segs, s_warp32, &all);
    {
        long long u = first_unit;
        for (int i = i0; i < i1; ++i) {
            const int n = pages_of(seqlens[i]);
            const long long next = u + n + fixed_cost;
            run += 1 + (n > 0 ? (int)((next - 1) / quota - (u + fixed_cost) / quota) : 0);
            num_splits[i + 1] = run;
            u = next;
        }
    }
    if (threadIdx.x == 0) num_splits[0] = 0;
}

}  // namespace

cudaError_t launch_schedule(const int32_t *seqlens, int batch, int num_parts, int fixed_cost, int combine_cost,
                            int32_t *metadata, int32_t *num_splits, unsigned int *status, cudaStream_t stream) {
    schedule_kernel<<<1, kSchedThreads, 0, stream>>>(seqlens, batch, num_parts, fixed_cost, combine_cost, metadata,
                                                     num_splits, status);
    return cudaGetLastError();
}

}  // namespace mla
