// C ABI of the MLA decode library: argument validation, workspace layout and
// kernel launches.  See include/mla_decode.h for the contract of each call.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// Device status word: kernels OR MLA_DEVERR_* bits into it instead of
// trapping.  Host code reaches it through its per-device address.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
unsigned int *g_status_addr[kMaxDevices] = {};
std::mutex g_status_mutex;

int status_address(unsigned int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return MLA_ERR_CUDA;
        g_status_addr[dev] = static_cast<unsigned int *>(ptr);
    }
    *out = g_status_addr[dev];
    return MLA_OK;
}

// NVTX range over a call's host side (argument checks and launches), so that
// a profiler timeline ties the kernels to the call that enqueued them; free
// when no tool is attached
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
};

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kRowsPerTile = 128;  // query rows per tensor-core tile

std::mutex g_timing_mutex;
// sparse decode: pair-split gathers with cluster multicast (1) or local gathers (0)
std::atomic<int> g_cluster_multicast{1};
cudaEvent_t g_split_begin = nullptr, g_split_end = nullptr;
constexpr int kMaxRows = 65536;

}  // namespace

size_t workspace_bytes(int batch, int rows, int num_parts) {
    const size_t splits = (size_t)batch + (size_t)num_parts;
    return align_up(splits * rows * kDv * sizeof(float)) + align_up(splits * rows * sizeof(float));
}

void carve_workspace(void *ws, int batch, int rows, int num_parts, float **o_accum, float **lse_accum) {
    const size_t splits = (size_t)batch + (size_t)num_parts;
    char *base = static_cast<char *>(ws);
    *o_accum = reinterpret_cast<float *>(base);
    *lse_accum = reinterpret_cast<float *>(base + align_up(splits * rows * kDv * sizeof(float)));
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_num_sm_parts(int device, int num_q_rows, int h_kv, int *num_parts) {
    if (!num_parts || num_q_rows < 1 || h_kv < 1) return MLA_ERR_INVALID_ARG;
    if (h_kv != 1) return MLA_ERR_UNSUPPORTED;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
    if (device != prev && cudaSetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
    // one CTA pair (two SMs) per part and row tile: as many pairs as fit at once
    int pairs = 0;
    cudaError_t e = split_kv_tc_max_pairs<576, false>(&pairs);  // every variant fits one CTA per SM
    if (device != prev) cudaSetDevice(prev);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    if (pairs < 1) pairs = 1;
    const int tiles = (num_q_rows + kRowsPerTile - 1) / kRowsPerTile;
    const int parts = pairs / tiles;
    *num_parts = parts > 0 ? parts : 1;
    return MLA_OK;
}

int mla_get_metadata_costs(const int32_t *cache_seqlens, int batch, int num_q_rows, int h_kv, int num_parts,
                           int fixed_cost, int combine_cost, int32_t *tile_scheduler_metadata, int32_t *num_splits,
                           struct CUstream_st *stream) {
    if (!cache_seqlens || !tile_scheduler_metadata || !num_splits) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || num_q_rows < 1 || h_kv < 1 || num_parts < 1) return MLA_ERR_INVALID_ARG;
    if (fixed_cost < 1 || fixed_cost > MLA_SCHED_MAX_COST || combine_cost < 0 || combine_cost > MLA_SCHED_MAX_COST)
        return MLA_ERR_INVALID_ARG;
    if (h_kv != 1) return MLA_ERR_UNSUPPORTED;
    Range range("mla_get_metadata");
    unsigned int *status = nullptr;
    if (status_address(&status) != MLA_OK) return MLA_ERR_CUDA;
    cudaError_t e = launch_schedule(cache_seqlens, batch, num_parts, fixed_cost, combine_cost, tile_scheduler_metadata,
                                    num_splits, status, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_get_metadata(const int32_t *cache_seqlens, int batch, int num_q_rows, int h_kv, int num_parts,
                     int32_t *tile_scheduler_metadata, int32_t *num_splits, struct CUstream_st *stream) {
    return mla_get_metadata_costs(cache_seqlens, batch, num_q_rows, h_kv, num_parts, kFixedCost, kCombineCost,
                                  tile_scheduler_metadata, num_splits, stream);
}

size_t mla_workspace_bytes(int batch, int s_q, int h_q, int h_kv, int dv, int num_parts) {
    if (batch < 1 || s_q < 1 || h_q < 1 || h_kv < 1 || num_parts < 1 || dv != kDv) return 0;
    if (h_q % h_kv) return 0;
    const long long rows = (long long)s_q * h_q / h_kv;
    if (rows > kMaxRows) return 0;
    return workspace_bytes(batch, (int)rows, num_parts);
}

}  // extern "C"

namespace {

enum class Kind { kBf16, kE4m3, kSparse };

// Index lists of the sparse decode (unused otherwise).
struct Lists {
    const int32_t *indices = nullptr;  // [batch][s_q][topk]
    int topk = 0;
    const int32_t *list_lens = nullptr;  // [batch]: the lengths the work partition was computed on
};

// The decode behind every cache format: validation, then split + combine.
int decode(const void *q, const void *kcache, Kind kind, int64_t num_blocks, const int32_t *block_table,
           int max_blocks_per_seq, const int32_t *cache_seqlens, int batch, int s_q, int h_q, int h_kv, int d, int dv,
           const int32_t *tile_scheduler_metadata, const int32_t *num_splits, int num_parts, float softmax_scale,
           int causal, void *o, float *lse, void *workspace, size_t ws_bytes, struct CUstream_st *stream,
           const Lists &lists = Lists()) {
    const bool e4m3 = kind == Kind::kE4m3, sparse = kind == Kind::kSparse;
    Range range(sparse ? "mla_decode_kvcache_sparse" : e4m3 ? "mla_decode_kvcache_fp8" : "mla_decode_kvcache");
    if (!q || !kcache || !block_table || !cache_seqlens || !tile_scheduler_metadata || !num_splits || !o || !lse ||
        !workspace)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || batch > 65535 || s_q < 1 || h_q < 1 || h_kv < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || num_parts < 1 || d < 1 || dv < 1)
        return MLA_ERR_INVALID_ARG;
    if (!(softmax_scale == softmax_scale)) return MLA_ERR_INVALID_ARG;
    if ((d != kDqk && d != kDv) || dv != kDv || h_kv != 1) return MLA_ERR_UNSUPPORTED;
    if (e4m3 && d != kDqk) return MLA_ERR_UNSUPPORTED;
    if (sparse) {
        if (!lists.indices || !lists.list_lens || lists.topk < 1) return MLA_ERR_INVALID_ARG;
        // a 128-row tile must hold the heads of one query token
        if (d != kDqk || (s_q > 1 && h_q != kRowsPerTile)) return MLA_ERR_UNSUPPORTED;
        // the gathers address cache rows with 32-bit coordinates
        if (num_blocks > 0x7fffffffLL / kPage) return MLA_ERR_UNSUPPORTED;
    }
    if ((long long)s_q * h_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * kPage > 0x7fffffffLL) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(o) || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
    const int rows = s_q * h_q;
    if (ws_bytes < workspace_bytes(batch, rows, num_parts)) return MLA_ERR_WORKSPACE;

    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.kcache = static_cast<const uint16_t *>(kcache);
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.max_blocks = max_blocks_per_seq;
    p.seqlens = sparse ? lists.list_lens : cache_seqlens;
    p.batch = batch;
    p.s_q = s_q;
    p.h_q = h_q;
    p.rows = rows;
    p.metadata = tile_scheduler_metadata;
    p.num_splits = num_splits;
    p.num_parts = num_parts;
    p.max_splits = batch + num_parts;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = (causal != 0 && s_q > 1 && !sparse) ? 1 : 0;
    p.indices = lists.indices;
    p.topk = lists.topk;
    p.kv_lens = cache_seqlens;
    p.o = static_cast<uint16_t *>(o);
    p.lse = lse;
    carve_workspace(workspace, batch, rows, num_parts, &p.o_accum, &p.lse_accum);
    if (status_address(&p.status) != MLA_OK) return MLA_ERR_CUDA;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t ev_begin, ev_end;
    {
        std::lock_guard<std::mutex> lock(g_timing_mutex);
        ev_begin = g_split_begin;
        ev_end = g_split_end;
    }
    if (ev_begin && cudaEventRecord(ev_begin, s) != cudaSuccess) return MLA_ERR_CUDA;
    cudaError_t e = sparse ? (g_cluster_multicast.load() ? launch_split_kv_tc_sparse(p, s)
                                                         : launch_split_kv_tc_sparse_local(p, s))
                    : e4m3 ? launch_split_kv_tc<576, true>(p, s)
                           : (d == kDqk ? launch_split_kv_tc<576, false>(p, s) : launch_split_kv_tc<512, false>(p, s));
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    if (ev_end && cudaEventRecord(ev_end, s) != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_combine(p, s);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_decode_kvcache(const void *q, const void *kcache, int64_t num_blocks, const int32_t *block_table,
                       int max_blocks_per_seq, const int32_t *cache_seqlens, int batch, int s_q, int h_q,
                       int h_kv, int d, int dv, const int32_t *tile_scheduler_metadata,
                       const int32_t *num_splits, int num_parts, float softmax_scale, int causal, void *o,
                       float *lse, void *workspace, size_t ws_bytes, struct CUstream_st *stream) {
    return decode(q, kcache, Kind::kBf16, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, batch, s_q, h_q,
                  h_kv, d, dv, tile_scheduler_metadata, num_splits, num_parts, softmax_scale, causal, o, lse, workspace,
                  ws_bytes, stream);
}

int mla_decode_kvcache_fp8(const void *q, const void *kv_pages, int64_t num_blocks, const int32_t *block_table,
                           int max_blocks_per_seq, const int32_t *cache_seqlens, int batch, int s_q, int h_q,
                           int h_kv, int d, int dv, const int32_t *tile_scheduler_metadata,
                           const int32_t *num_splits, int num_parts, float softmax_scale, int causal, void *o,
                           float *lse, void *workspace, size_t ws_bytes, struct CUstream_st *stream) {
    return decode(q, kv_pages, Kind::kE4m3, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, batch, s_q,
                  h_q, h_kv, d, dv, tile_scheduler_metadata, num_splits, num_parts, softmax_scale, causal, o, lse, workspace,
                  ws_bytes, stream);
}

int mla_decode_kvcache_sparse(const void *q, const void *kcache, int64_t num_blocks, const int32_t *block_table,
                              int max_blocks_per_seq, const int32_t *cache_seqlens, const int32_t *indices, int topk,
                              const int32_t *list_lens, int batch, int s_q, int h_q, int h_kv, int d, int dv,
                              const int32_t *tile_scheduler_metadata, const int32_t *num_splits, int num_parts,
                              float softmax_scale, void *o, float *lse, void *workspace, size_t ws_bytes,
                              struct CUstream_st *stream) {
    Lists lists;
    lists.indices = indices;
    lists.topk = topk;
    lists.list_lens = list_lens;
    return decode(q, kcache, Kind::kSparse, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, batch, s_q,
                  h_q, h_kv, d, dv, tile_scheduler_metadata, num_splits, num_parts, softmax_scale, 0, o, lse,
                  workspace, ws_bytes, stream, lists);
}

int mla_device_status(int *status, int clear) {
    if (!status) return MLA_ERR_INVALID_ARG;
    unsigned int *addr = nullptr;
    if (status_address(&addr) != MLA_OK) return MLA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, addr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    if (clear && v) {
        const unsigned int zero = 0;
        if (cudaMemcpy(addr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ERR_CUDA;
    }
    *status = (int)v;
    return MLA_OK;
}

int mla_set_timing_events(void *split_begin, void *split_end) {
    if ((split_begin == nullptr) != (split_end == nullptr)) return MLA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    g_split_begin = static_cast<cudaEvent_t>(split_begin);
    g_split_end = static_cast<cudaEvent_t>(split_end);
    return MLA_OK;
}

int mla_set_cluster_multicast(int enabled) {
    if (enabled != 0 && enabled != 1) return MLA_ERR_INVALID_ARG;
    g_cluster_multicast.store(enabled);
    return MLA_OK;
}

const char *mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape or device";
        case MLA_ERR_WORKSPACE: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA runtime error";
        case MLA_ERR_DEVICE: return "a kernel reported a device-side error";
        default: return "unknown status";
    }
}

}  // extern "C"
