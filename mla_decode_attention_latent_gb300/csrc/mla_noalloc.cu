// mla_decode_kvcache_noalloc: the decode call for callers that cannot
// allocate device memory themselves.
//
// Some callers of a decode kernel may not call cudaMalloc (or any allocating
// routine) at the point where they decode: a serving runtime that hands out
// every byte of device memory from its own pre-planned arena, a plugin
// interface that provides the call with its inputs and outputs but no
// workspace, or a hot loop that must not risk the implicit device
// synchronisation and fragmentation an allocation can bring.  They still own
// and pass the inputs and outputs; only the split-KV scratch (the fp32 partial
// outputs and partial LSEs of split sequences) is the library's problem.
//
// Here that scratch is one file-scope device array of fixed size.  Every GPU
// that loads the library holds it until the process exits.  All calls share
// it and it keeps whatever the previous call left; nothing in it needs to
// start at zero, because every slot the combine kernel reads is written
// earlier in the same call.  Two calls whose kernels overlap on the GPU (for
// example on two streams) race on the array: callers must order them.
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// fixed capacity of the shared scratch, bytes
constexpr size_t kNoAllocScratchBytes = (size_t)MLA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the real address is
// asked for once per device, with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return MLA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" int mla_decode_kvcache_noalloc(const void *q, const void *kcache, int64_t num_blocks,
                                          const int32_t *block_table, int max_blocks_per_seq,
                                          const int32_t *cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                                          int d, int dv, const int32_t *tile_scheduler_metadata,
                                          const int32_t *num_splits, int num_parts, float softmax_scale,
                                          int causal, void *o, float *lse, struct CUstream_st *stream) {
    if (!q || !kcache || !block_table || !cache_seqlens || !tile_scheduler_metadata || !num_splits || !o || !lse)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || s_q < 1 || h_q < 1 || h_kv < 1 || num_parts < 1 || d < 1 || dv < 1) return MLA_ERR_INVALID_ARG;
    if ((d != MLA_HEAD_DIM && d != MLA_V_DIM) || dv != MLA_V_DIM || h_kv != 1 || (long long)s_q * h_q > 65536)
        return MLA_ERR_UNSUPPORTED;
    const size_t need = mla_workspace_bytes(batch, s_q, h_q, h_kv, dv, num_parts);
    if (need == 0) return MLA_ERR_INVALID_ARG;
    if (need > mla::kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // beyond the fixed scratch
    void *scratch = nullptr;
    if (mla::scratch_address(&scratch) != MLA_OK) return MLA_ERR_CUDA;
    return mla_decode_kvcache(q, kcache, num_blocks, block_table, max_blocks_per_seq, cache_seqlens, batch, s_q, h_q,
                              h_kv, d, dv, tile_scheduler_metadata, num_splits, num_parts, softmax_scale, causal, o,
                              lse, scratch, mla::kNoAllocScratchBytes, stream);
}
