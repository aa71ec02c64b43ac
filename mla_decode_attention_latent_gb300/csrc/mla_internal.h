// Internal host-side interface between the C-ABI layer (mla_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mla_decode.h"

namespace mla {

constexpr int kPage = MLA_PAGE_SIZE;       // tokens per cache page
constexpr int kDqk = MLA_HEAD_DIM;         // 512 latent + 64 RoPE dims
constexpr int kDv = MLA_V_DIM;             // value dims = first 512 dims of a row
constexpr int kMdInts = MLA_METADATA_INTS;
constexpr int kFixedCost = MLA_SCHED_FIXED_COST_PAGES;
constexpr int kCombineCost = MLA_SCHED_COMBINE_COST_PAGES;

// Everything a split-KV kernel needs for one decode call.
struct DecodeParams {
    const uint16_t *q;            // [batch][s_q][h_q][576] bf16
    const uint16_t *kcache;       // [num_blocks][64][1][576] bf16, or packed e4m3 pages (read as bytes)
    int64_t num_blocks;
    const int32_t *block_table;   // [batch][max_blocks]
    int max_blocks;
    const int32_t *seqlens;       // [batch]
    int batch, s_q, h_q;
    int rows;                     // s_q * h_q query rows per sequence
    const int32_t *metadata;      // [num_parts][8]
    const int32_t *num_splits;    // [batch + 1]
    int num_parts;
    int max_splits;               // batch + num_parts: capacity of the workspace
    float scale_log2;             // softmax_scale * log2(e)
    int causal;
    uint16_t *o;                  // [batch][s_q][h_q][512] bf16
    float *lse;                   // [batch][s_q][h_q]
    float *o_accum;               // [max_splits][rows][512] fp32 partial outputs
    float *lse_accum;             // [max_splits][rows] partial LSE (natural log)
    unsigned int *status;         // device status word (MLA_DEVERR_* bits)
    // sparse top-k decode only (seqlens then holds each sequence's list length)
    const int32_t *indices;       // [batch][s_q][topk] token positions per query token
    int topk;
    const int32_t *kv_lens;       // [batch] cache lengths: positions >= kv_lens[b] are ignored
};

// Workspace carve-up shared by the API, the split kernel and the combine.
size_t workspace_bytes(int batch, int rows, int num_parts);
void carve_workspace(void *ws, int batch, int rows, int num_parts, float **o_accum, float **lse_accum);

cudaError_t launch_schedule(const int32_t *seqlens, int batch, int num_parts, int fixed_cost, int combine_cost,
                            int32_t *metadata, int32_t *num_splits, unsigned int *status, cudaStream_t stream);
// the tensor-core split-KV kernel for cached rows of width D (576 or 512), bf16
// rows or (E4M3, D = 576) packed e4m3 pages with per-token scales
template <int D, bool E4M3>
cudaError_t launch_split_kv_tc(const DecodeParams &p, cudaStream_t stream);
// the sparse top-k variant (576-wide bf16 rows gathered from index lists):
// the CTA pair splits each page's gathers with cluster multicast, or (local)
// each CTA gathers its own rows
cudaError_t launch_split_kv_tc_sparse(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_split_kv_tc_sparse_local(const DecodeParams &p, cudaStream_t stream);
int split_kv_tc_tile_rows();
// CTA pairs of the split-KV kernel that fit on the current device at once
template <int D, bool E4M3>
cudaError_t split_kv_tc_max_pairs(int *pairs);
cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream);

}  // namespace mla
