/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * Multi-head Latent Attention decoding over a paged latent KV cache.  Every
 * query head attends to one shared latent KV head: a cached row of
 * d = 576 bf16 values (512 latent + 64 decoupled-RoPE dims) serves as the key,
 * and its first dv = 512 dims as the value.  Pages hold 64 tokens and are
 * addressed through a per-sequence block table.
 *
 * Sources for the operations declared here:
 *  - "Novita AI, H100 및 H200에서 FlashMLA 평가", section "MLA란 무엇인가요?",
 *    table "MHA vs MQA vs GQA vs MLA": all heads share a compressed latent KV
 *    vector per token, with RoPE decoupled.
 *  - "FlashMLA란 무엇인가?" (topnet.top article 5338), section "FlashMLA의 주요
 *    특성": bf16 and a paged KV cache with block size 64.
 *  - same page, section "FlashMLA 설치 및 사용":
 *      step 2 "MLA 메타데이터 가져오기": get_mla_metadata(cache_seqlens,
 *        s_q * h_q // h_kv, h_kv) -> (tile_scheduler_metadata, num_splits),
 *        computed once and reused by every layer;
 *      step 3 "MLA 디코딩 실행": flash_mla_with_kvcache(q, kvcache, block_table,
 *        cache_seqlens, dv, tile_scheduler_metadata, num_splits, causal)
 *        -> (o, lse).
 *  - same page, section "FlashMLA의 기술 구현" ("병렬 디코딩"): several query
 *    tokens per step, read here as s_q > 1 with a causal mask: query i of a
 *    sequence of length T sees cached positions < T - s_q + i + 1.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    the caller allocates, owns and frees them.  The library never allocates,
 *    frees or retains caller memory and keeps no per-call state.
 *  - `stream` is a CUDA stream (cudaStream_t / CUstream; NULL = legacy default).
 *    Calls that launch work enqueue it on `stream` and return without waiting.
 *  - Return value: MLA_OK (0) or a negative MLA_ERR_* code.  Arguments are
 *    validated on the host before anything is launched; on an argument error
 *    nothing is launched and no output is touched.
 *  - bf16 tensors are raw IEEE bfloat16 bit patterns (2 bytes per element),
 *    row-major and densely packed in the shapes given.
 *  - The library looks up the device addresses of its own device arrays (the
 *    status word, the scratch of mla_decode_kvcache_noalloc) once per device
 *    and keeps them for the life of the process.  cudaDeviceReset invalidates
 *    them: do not call the library on a device after resetting it in the same
 *    process.
 *
 * Supported on the GPU path: d = 576 or 512 (bf16 cache) or 576 (packed
 * e4m3 cache, mla_decode_kvcache_fp8), dv = 512, page size 64,
 * h_kv = 1, any batch >= 1, any s_q >= 1 and h_q >= 1 with
 * s_q * h_q <= 65536.  d = 512 is the d_qk = 512 variant that the
 * "[FlashInfer] ... SM120 sparse MLA" page names for DSv4, read as a
 * 512-dim cached row that is both key and value (no separate RoPE part).
 * Other shapes return MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

/* status codes */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1)   /* null pointer, negative size, inconsistent shapes */
#define MLA_ERR_UNSUPPORTED (-2)   /* shape or device outside what the GPU path implements */
#define MLA_ERR_WORKSPACE (-3)     /* workspace smaller than mla_workspace_bytes() */
#define MLA_ERR_CUDA (-4)          /* a CUDA runtime call or kernel launch failed */
#define MLA_ERR_DEVICE (-5)        /* a kernel reported an error (see mla_device_status) */

/* fixed shape constants of the GPU path */
#define MLA_PAGE_SIZE 64
#define MLA_HEAD_DIM 576
#define MLA_V_DIM 512
#define MLA_METADATA_INTS 8
/* fixed cost of one split-KV segment, in pages, used by the work partition */
#define MLA_SCHED_FIXED_COST_PAGES 8
/* cost, in pages, that the partition charges for needing the combine pass */
#define MLA_SCHED_COMBINE_COST_PAGES 4
/* the same two costs for the sparse decode, in 64-entry list chunks: a list
   chunk's row gathers take about four times a dense page, so the per-segment
   costs come to a quarter or less (measured on GB300: topk 2048 over b = 64
   sequences, split + combine 170 us with the dense costs, 156 us with a
   fixed cost of 2 chunks, 153 us with 1) */
#define MLA_SCHED_SPARSE_FIXED_COST_CHUNKS 1
#define MLA_SCHED_SPARSE_COMBINE_COST_CHUNKS 1
/* largest cost mla_get_metadata_costs accepts */
#define MLA_SCHED_MAX_COST (1 << 20)

/* device-side error bits reported through mla_device_status() */
#define MLA_DEVERR_TIMEOUT 0x1     /* a bounded wait inside a kernel gave up */
#define MLA_DEVERR_BLOCK_ID 0x2    /* a block_table entry was outside [0, num_blocks) */
#define MLA_DEVERR_SEQLEN 0x4      /* a cache_seqlens entry was negative or beyond the table */
#define MLA_DEVERR_SCALE 0x8       /* an e4m3 page held a scale with |c| >= 255 (or NaN) for a token
                                      inside its sequence (mla_decode_kvcache_fp8) */

/*
 * mla_num_sm_parts — number of split-KV work parts for one decode call.
 *
 * Host-only query.  The caller uses it to size tile_scheduler_metadata
 * ([num_parts * MLA_METADATA_INTS] int32) before mla_get_metadata.
 *   device      CUDA device ordinal the decode will run on
 *   num_q_rows  query rows per KV head: s_q * h_q / h_kv (the pages' second
 *               argument of get_mla_metadata)
 *   h_kv        KV heads (must be 1)
 *   num_parts   out: number of parts (>= 1)
 * Errors: MLA_ERR_INVALID_ARG (null out pointer, num_q_rows < 1),
 *         MLA_ERR_UNSUPPORTED (h_kv != 1), MLA_ERR_CUDA (device query failed).
 */
MLA_API int mla_num_sm_parts(int device, int num_q_rows, int h_kv, int *num_parts);

/*
 * mla_get_metadata — split-KV work partition ("MLA 메타데이터 가져오기").
 *
 * Launches the tile-scheduler kernel on `stream`.  It reads the sequence
 * lengths and cuts the (sequence, page) range into `num_parts` contiguous
 * parts of near-equal cost (pages plus MLA_SCHED_FIXED_COST_PAGES per
 * segment); a sequence may be cut across several parts (split-KV).  When
 * the batch is smaller than num_parts and one part per sequence is
 * estimated to finish sooner (no sequence cut, so no combine, charged
 * MLA_SCHED_COMBINE_COST_PAGES), only `batch` parts get work and the
 * others are empty.
 *   cache_seqlens            device int32 [batch]; entries >= 0
 *   batch                    number of sequences (>= 1)
 *   num_q_rows, h_kv         as for mla_num_sm_parts
 *   num_parts                parts to produce (>= 1; normally mla_num_sm_parts)
 *   tile_scheduler_metadata  device int32 [num_parts][MLA_METADATA_INTS], out:
 *                            per part {begin_seq, begin_page, end_seq,
 *                            end_page, begin_split, 0, 0, 0}; the part covers
 *                            the (sequence, page) cursor range [begin, end)
 *   num_splits               device int32 [batch + 1], out: prefix sum over
 *                            sequences of the number of parts touching each
 * The outputs stay valid for every decode call with the same cache_seqlens
 * values, num_q_rows and num_parts (one computation serves all layers).
 * A negative length sets MLA_DEVERR_SEQLEN in the device status word.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (h_kv != 1), MLA_ERR_CUDA.
 */
MLA_API int mla_get_metadata(const int32_t *cache_seqlens, int batch, int num_q_rows, int h_kv,
                     int num_parts, int32_t *tile_scheduler_metadata, int32_t *num_splits,
                     struct CUstream_st *stream);

/*
 * mla_get_metadata_costs — the same partition with the two costs given.
 *
 * mla_get_metadata is this call with fixed_cost = MLA_SCHED_FIXED_COST_PAGES
 * and combine_cost = MLA_SCHED_COMBINE_COST_PAGES.  The costs are in units
 * of one page of the lengths the partition is computed on (for the sparse
 * decode: one 64-entry list chunk; MLA_SCHED_SPARSE_*_CHUNKS are its
 * measured values).  They change only how the work is cut, never what a
 * decode computes.
 *   fixed_cost    cost of one segment (>= 1, <= MLA_SCHED_MAX_COST)
 *   combine_cost  cost charged for needing the combine (>= 0, <= MLA_SCHED_MAX_COST)
 * Other arguments, outputs and errors: as mla_get_metadata.
 */
MLA_API int mla_get_metadata_costs(const int32_t *cache_seqlens, int batch, int num_q_rows, int h_kv,
                           int num_parts, int fixed_cost, int combine_cost, int32_t *tile_scheduler_metadata,
                           int32_t *num_splits, struct CUstream_st *stream);

/*
 * mla_workspace_bytes — device scratch that mla_decode_kvcache needs for the
 * partial results of split sequences: fp32 partial outputs and their LSE for
 * at most (batch + num_parts) splits.  Returns 0 on invalid arguments.
 */
MLA_API size_t mla_workspace_bytes(int batch, int s_q, int h_q, int h_kv, int dv, int num_parts);

/*
 * mla_decode_kvcache — MLA decode over the paged latent cache ("MLA 디코딩 실행").
 *
 * For batch b, query token i, head h (all heads share KV head 0):
 *   T    = cache_seqlens[b]                 (causal == 0, or s_q == 1)
 *   T    = cache_seqlens[b] - s_q + i + 1   (causal != 0)
 *   k_j  = kcache[block_table[b][j / 64]][j % 64][0][0..d),     j < T
 *   s_j  = softmax_scale * <q[b][i][h], k_j>
 *   lse  = ln sum_j exp(s_j)
 *   o    = sum_j exp(s_j - lse) * k_j[0..512)
 * Rows with T <= 0 get o = 0 and lse = -inf.
 *
 *   q              device bf16 [batch][s_q][h_q][d]
 *   kcache         device bf16 [num_blocks][64][h_kv][d]; 16-byte aligned.
 *                  Rows past a sequence's end may hold any bits (NaN too).
 *   num_blocks     physical pages in kcache
 *   block_table    device int32 [batch][max_blocks_per_seq]; the first
 *                  ceil(T_b / 64) entries of row b must lie in [0, num_blocks)
 *   cache_seqlens  device int32 [batch]; 0 <= T_b <= 64 * max_blocks_per_seq
 *   d, dv          576 (or 512) and 512
 *   tile_scheduler_metadata, num_splits, num_parts
 *                  from mla_get_metadata with the same cache_seqlens
 *   softmax_scale  multiplies q.k before the softmax (e.g. 1/sqrt(576))
 *   causal         nonzero: the causal rule above (only matters for s_q > 1)
 *   o              device bf16 [batch][s_q][h_q][dv], out
 *   lse            device fp32 [batch][s_q][h_q], out (natural log)
 *   workspace      device scratch of at least mla_workspace_bytes(...) bytes,
 *                  256-byte aligned; its contents on entry do not matter
 * Out-of-range block ids or lengths found on the device are skipped and set
 * bits in the device status word (mla_device_status); they never fault.
 * Stream order: two kernels are enqueued on `stream` (split-KV, then the
 * combine), both as programmatic dependent launches.  Each may be scheduled
 * while the kernel before it is finishing, but reads and writes no global
 * memory until that kernel has completed, so the call observes every earlier
 * write on the stream exactly as an ordinary launch would.  The launches can
 * be captured in a CUDA graph once the first call on a device has set the
 * kernel attributes.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE,
 *         MLA_ERR_CUDA (launch failure).
 */
MLA_API int mla_decode_kvcache(const void *q, const void *kcache, int64_t num_blocks,
                       const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                       int d, int dv, const int32_t *tile_scheduler_metadata,
                       const int32_t *num_splits, int num_parts, float softmax_scale,
                       int causal, void *o, float *lse, void *workspace,
                       size_t workspace_bytes, struct CUstream_st *stream);

/*
 * mla_decode_kvcache_fp8 — the same decode over a cache of packed e4m3 pages
 * with per-token scales.
 *
 * The page "[flashinfer] FlashInfer, SM120 GPU를 위한 희소 MLA 커널 추가로 LLM
 * 추론 속도 향상" (item 5, flashinfer/mla/trtllm.py) says that the MLA decode
 * API takes a `kv_scale_format` for a packed KV cache with scales, and the page
 * "[vllm] Blackwell을 위한 새로운 MLA 백엔드: TOKENSPEED_MLA 분석" (section
 * "들어가며") runs the Blackwell decode on an FP8 KV cache; neither gives the
 * layout.  This library's reading: a page of the cache is one packed
 * record of MLA_FP8_PAGE_BYTES(d) bytes,
 *   bytes [0, 64 d)          64 rows of d OCP e4m3 codes (row j, dim c at j d + c)
 *   bytes [64 d, 64 d + 256) 64 fp32 per-token scales c_j (little endian)
 * and cached row j dequantizes to k_j[c] = c_j * e4m3(code[j][c]).  The call
 * then computes exactly what mla_decode_kvcache computes on the dequantized
 * rows (V = their first 512 dims).
 *
 *   kv_pages       device bytes [num_blocks][MLA_FP8_PAGE_BYTES(d)]; 16-byte
 *                  aligned.  Codes and scales of rows past a sequence's end
 *                  may hold any bits.
 *   d              576 only (other values: MLA_ERR_UNSUPPORTED)
 *   everything else as for mla_decode_kvcache (q, o and lse stay bf16/fp32).
 * Precision: the kernel computes in f16 on the tensor cores.  The e4m3 codes
 * widen to f16 exactly; q is rounded to f16 (exact for |q| in [2^-17, 65504]);
 * the softmax weights times c_j are rounded to f16, so |c_j| must stay below
 * 255 for every token inside a sequence (a larger one can overflow f16).  A
 * scale with |c_j| >= 255, or a NaN scale, of a token inside its sequence
 * sets MLA_DEVERR_SCALE in the device status word, and the outputs of that
 * sequence are then undefined.  Scales of rows past a sequence's end are
 * never read.
 * Stream order, graph capture and errors: as for mla_decode_kvcache.
 */
#define MLA_FP8_PAGE_BYTES(d) (MLA_PAGE_SIZE * (d) + MLA_PAGE_SIZE * 4)
MLA_API int mla_decode_kvcache_fp8(const void *q, const void *kv_pages, int64_t num_blocks,
                                   const int32_t *block_table, int max_blocks_per_seq,
                                   const int32_t *cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                                   int d, int dv, const int32_t *tile_scheduler_metadata,
                                   const int32_t *num_splits, int num_parts, float softmax_scale,
                                   int causal, void *o, float *lse, void *workspace,
                                   size_t workspace_bytes, struct CUstream_st *stream);

/*
 * mla_decode_kvcache_sparse — sparse top-k decode: each query token attends
 * only to the cached tokens its index list names.
 *
 * The page "[flashinfer] FlashInfer, SM120 GPU를 위한 희소 MLA 커널 추가로 LLM
 * 추론 속도 향상" (section "왜 이게 좋은가?", item 2) describes sparse MLA as
 * attention over only the top-k selected tokens of a paged cache; it gives no
 * interface.  This library's reading: query token i of sequence b carries
 * indices[b][i][0 .. topk) (token positions, shared by all its heads); an
 * entry is ignored when it is outside [0, cache_seqlens[b]) (-1 pads short
 * lists) or at or past list_lens[b]; every other entry is one term of the
 * softmax (a position listed twice counts twice); no causal mask applies:
 *   s_t = softmax_scale * <q, k_{indices[t]}>,  lse = ln sum_t exp(s_t),
 *   o   = sum_t exp(s_t - lse) * k_{indices[t]}[0..512)   over valid entries t.
 * A row with no valid entry gets o = 0 and lse = -inf.
 *
 *   kcache, block_table, cache_seqlens, q, o, lse, workspace
 *                  as for mla_decode_kvcache (bf16 cache, d = 576 only)
 *   indices        device int32 [batch][s_q][topk]
 *   topk           entries per list, >= 1
 *   list_lens      device int32 [batch]: the lengths the work partition was
 *                  computed on (tile_scheduler_metadata and num_splits come
 *                  from mla_get_metadata_costs on this array with
 *                  MLA_SCHED_SPARSE_FIXED_COST_CHUNKS and
 *                  MLA_SCHED_SPARSE_COMBINE_COST_CHUNKS, or from
 *                  mla_get_metadata; normally topk for every sequence)
 * A 128-row tile holds one query token's heads: s_q must be 1, or h_q 128
 * (MLA_ERR_UNSUPPORTED otherwise).  Rows are gathered one by one from the
 * cache (TMA gathers over the cache viewed as num_blocks * 64 rows, which
 * must stay below 2^31: MLA_ERR_UNSUPPORTED otherwise), so any positions may
 * be listed.
 * Stream order, graph capture and errors: as for mla_decode_kvcache.
 */
MLA_API int mla_decode_kvcache_sparse(const void *q, const void *kcache, int64_t num_blocks,
                                      const int32_t *block_table, int max_blocks_per_seq,
                                      const int32_t *cache_seqlens, const int32_t *indices, int topk,
                                      const int32_t *list_lens, int batch, int s_q, int h_q, int h_kv,
                                      int d, int dv, const int32_t *tile_scheduler_metadata,
                                      const int32_t *num_splits, int num_parts, float softmax_scale,
                                      void *o, float *lse, void *workspace, size_t workspace_bytes,
                                      struct CUstream_st *stream);

/*
 * mla_decode_kvcache_noalloc — mla_decode_kvcache for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart of this call; it exists for callers that may
 * not allocate at decode time: runtimes that plan every byte of device memory
 * up front in their own arena, plugin interfaces that pass a call its inputs
 * and outputs but no workspace, and hot loops that must avoid an
 * allocation's implicit synchronisation.  The arguments and results are those
 * of mla_decode_kvcache without `workspace` / `workspace_bytes`: the split-KV
 * scratch comes from one fixed device array of MLA_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  No call allocates (no cudaMalloc, cudaFree or allocating
 * library routine).
 *  - The first call on a device looks up the array's device address with that
 *    device current (a one-time set-up per device); make that first call
 *    before any stream capture.
 *  - Every call shares the array and it keeps the previous call's contents;
 *    nothing in it needs to start at zero.  Calls whose kernels overlap on the
 *    GPU (e.g. on two streams) race on it: order them on one stream.
 * Errors: those of mla_decode_kvcache, and MLA_ERR_WORKSPACE when
 * mla_workspace_bytes() for the shape exceeds MLA_NOALLOC_SCRATCH_BYTES
 * (nothing is launched then).
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
MLA_API int mla_decode_kvcache_noalloc(const void *q, const void *kcache, int64_t num_blocks,
                                       const int32_t *block_table, int max_blocks_per_seq,
                                       const int32_t *cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                                       int d, int dv, const int32_t *tile_scheduler_metadata,
                                       const int32_t *num_splits, int num_parts, float softmax_scale,
                                       int causal, void *o, float *lse, struct CUstream_st *stream);

/*
 * mla_device_status — read the device status word of the current device.
 *
 * Synchronizes the device, stores the OR of the MLA_DEVERR_* bits raised by
 * kernels since the last clear into *status, and clears the word if `clear`
 * is nonzero.  Returns MLA_OK, MLA_ERR_INVALID_ARG or MLA_ERR_CUDA.
 */
MLA_API int mla_device_status(int *status, int clear);

/*
 * mla_set_timing_events — profiling aid: time the split-KV kernel alone.
 *
 * While set, every mla_decode_kvcache call records `split_begin` on its
 * stream just before the split-KV kernel and `split_end` just after it, so
 * that cudaEventElapsedTime gives that kernel's duration (the combine kernel
 * is outside the pair).  Both are cudaEvent_t handles created by the caller
 * on the device the decode runs on; pass NULL, NULL to stop.  The setting is
 * process-wide.  Returns MLA_OK, or MLA_ERR_INVALID_ARG if only one is NULL.
 */
MLA_API int mla_set_timing_events(void *split_begin, void *split_end);

/*
 * mla_set_cluster_multicast — how mla_decode_kvcache_sparse gathers rows.
 *
 * With 1 (the default) the two CTAs of a cluster split each list chunk's row
 * gathers between them and write every gathered row into both CTAs with a
 * TMA cluster multicast (within this GPU's own memory).  With 0 each CTA
 * gathers every row chunk it uses itself and nothing is multicast; the
 * results are bit-identical, the decode about 1.3x slower.  A process that
 * runs one job across several GPUs sets 0 before its first call.  The
 * setting is process-wide.  Returns MLA_OK, or MLA_ERR_INVALID_ARG unless
 * `enabled` is 0 or 1.
 */
MLA_API int mla_set_cluster_multicast(int enabled);

/* mla_status_string — static description of a status code (never NULL). */
MLA_API const char *mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
