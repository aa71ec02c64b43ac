// Split-KV MLA decode on sm_103a tensor cores: one CTA pair per (part, row tile).
//
// Implementation shared by the translation units that instantiate it for one
// cached row width D = MLA_SPLIT_D: 576 (512 latent + 64 RoPE dims, the
// DeepSeek-style latent cache) or 512 (the d_qk = 512 variant that the
// "[FlashInfer] ... SM120 sparse MLA" page names for DSv4: read here as a
// 512-dim row that is both key and value, with no separate RoPE part).
//
// What is computed (per query row r = i * h_q + h of sequence b, over the keys
// of the part's page range; see include/mla_decode.h):
//   s_j = scale * <q_r, k_j>,  p_j = 2^(s_j log2 e - m),  O = sum_j p_j v_j / l
// with an fp32 online softmax (running max m, running sum l), and at the end
// of the range either the final O (bf16) and LSE, or an fp32 partial O and
// partial LSE for the combine kernel when the sequence is split.  Sources:
// "FlashMLA란 무엇인가?" (topnet.top article 5338), sections "FlashMLA의 주요
// 특성" (bf16, paged cache, block 64) and "FlashMLA 설치 및 사용" step 3 (the
// decode call returns o and lse); "Novita AI, H100 및 H200에서 FlashMLA 평가",
// table "MHA vs MQA vs GQA vs MLA" (every head shares the latent KV row, so
// QK^T and PV are dense contractions over all heads of a tile).
//
// Design (GB300-first; the pages' kernel is a Hopper design and only prior art):
// a 128 x 512 fp32 output accumulator fills a whole SM's tensor memory, so the
// work of one tile is split across the two CTAs of a cluster by role:
//
//   score CTA (rank 0)                       value CTA (rank 1)
//   ------------------                       ------------------
//   Q latent [128 x 512] bf16 in TMEM,       O tile [128 x 512] fp32 in TMEM
//     Q RoPE [128 x 64] in smem (D = 576)    TMA: page dims 0..511 (8 chunks)
//   TMA: 16 KB chunk slots, each holding       into a 2-stage ring
//     one 64-dim chunk of two pages          tcgen05 O += P V  (N = 2 x 256)
//   tcgen05 S = Q K^T over two pages at      4 warps: zero the tail rows of V,
//     once (N = 128), A from TMEM (the         lazy O rescale, epilogue staged
//     RoPE chunk's from smem), two issuers     through smem
//     alternating steps
//   4 warps: mask + online softmax; P and
//     row factors -> local staging -> bulk
//     copies into the value CTA
//
// Loads: the chunk loads of the score CTA come from HBM (the value CTA's load
// of the same page then hits L2).  P and the row factors (17 KB per page) go
// to the value CTA as one bulk copy per row warp, completing on the value
// CTA's barrier; the value CTA's MMA commit hands the buffer back through a
// multicast commit.  The running max is rescaled lazily: O is only corrected
// when a page's maximum exceeds the current one by more than 2^8.
//
// Warp roles (256 threads): warp 0 issues TMA, warp 1 allocates TMEM and
// issues MMAs (one elected lane), warps 2..5 are the row warps (thread t of
// warp w owns TMEM lane / tile row 32 * (w % 4) + t); in the score CTA warp 6
// is the second MMA issuer and warp 7 the second TMA producer.
//
// Every wait is bounded (mla_sm103.cuh); on a timeout the kernel raises
// MLA_DEVERR_TIMEOUT, tells its peer CTA to stop, and unwinds.
//
// e4m3 cache (MLA_SPLIT_FP8 = 1, D = 576): a page holds 64 rows of e4m3 codes
// followed by 64 fp32 per-token scales, and row j dequantizes to c_j * code_j
// (include/mla_decode.h).  Scores run on the fp8 tensor cores: each q row is
// split into three e4m3 parts (q / sigma_r ~ h + m + l, sigma_r = max |q_r| /
// 448), and every part is contracted with the codes as they land (nine
// 64-byte-swizzled chunks per page); the row warps sum the three and multiply
// by sigma_r, the softmax scale and the token's scale.  The value CTA widens
// its page's value codes to f16 (exact for every e4m3 value) in place in the
// upper half of each V stage, zeroing the rows past a sequence's end, and runs
// P V in f16 with P multiplied by the token's scale, so the accumulators see
// c_j * code_j as the dequantized row.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <mutex>

#include "mla_internal.h"
#include "mla_sm103.cuh"

#ifndef MLA_SPLIT_D
#error "define MLA_SPLIT_D (the cached row width: 576 or 512) before including this file"
#endif

namespace mla {
namespace {

using namespace sm103;

constexpr int kD = MLA_SPLIT_D;                // cached row width: key dims, the first kDv of them the value
static_assert(kD == 576 || kD == 512, "supported cached row widths");
constexpr bool kHasRope = kD > kDv;            // a RoPE part beyond the value dims (one more 64-dim chunk)
#ifndef MLA_SPLIT_FP8
#define MLA_SPLIT_FP8 0
#endif
constexpr bool kFp8 = MLA_SPLIT_FP8 != 0;      // e4m3 cache pages with per-token scales
#ifndef MLA_SPLIT_SPARSE
#define MLA_SPLIT_SPARSE 0
#endif
constexpr bool kSparse = MLA_SPLIT_SPARSE != 0;  // keys gathered row by row from per-query-token index lists
#ifndef MLA_SPARSE_MULTICAST
#define MLA_SPARSE_MULTICAST 1
#endif
// sparse lists: the CTA pair splits each page's row gathers and multicasts
// them to both CTAs (1), or each CTA gathers every chunk it uses itself (0)
constexpr bool kPairGather = kSparse && MLA_SPARSE_MULTICAST != 0;
static_assert(!(kSparse && kFp8) && (!kSparse || MLA_SPLIT_D == 576), "sparse decode: 576-wide bf16 rows");
constexpr bool kRing = kFp8 || kSparse;          // a per-step side ring (e4m3: token scales; sparse: key masks)

constexpr int kThreads = 256;                  // 8 warps: TMA, MMA, 4 row warps, second score MMA issuer and TMA producer
constexpr int kTileRows = 128;                 // query rows per tile = TMEM lanes
constexpr int kScoreIssuers = 2;               // score-CTA MMA issuers (and TMA producers), alternating steps
// Pages per score step: two for bf16 rows (one tcgen05 MMA with N = 128
// covers both), one for e4m3 pages, whose scores are three fp8 contractions
// (see below) and whose S buffers are therefore one page wide, and one for
// sparse lists, whose gathered pages both CTAs share (below).
constexpr int kStepPages = (kFp8 || kSparse) ? 1 : 2;
// score CTA: MMA operand slots, one ring per issuer: for bf16 rows 5 each of
// 16 KB (one 64-dim chunk of two pages); for e4m3 pages 2 each of 36 KB (the
// nine 64-code chunks of one page, each a 64-byte-swizzled [64 x 64 B] tile).
// Sparse lists use no ring: both CTAs hold the same two page buffers (all nine
// 64-dim chunks of a gathered page, 72 KB each) at the same offsets, filled by
// gathers that each CTA issues for part of the chunks and multicasts to both,
// so that each SM's gather engine moves about half of a page's rows.
constexpr int kKSlots = kFp8 ? 4 : (kSparse ? 2 : 10);
constexpr int kRingSlots = kKSlots / kScoreIssuers;  // slots per score-MMA issuer's ring
constexpr int kVStages = 2;                    // value CTA ring: whole pages (dims 0..511)
constexpr int kSBufs = 2;                      // S buffers in TMEM (score CTA), one per step
constexpr int kPBufs = 2;                      // P buffers (staging in the score CTA, landing in the value CTA)
constexpr int kKChunks = kD / 64;              // 9 (or 8) chunks of 64 dims (128 B rows)
constexpr int kVChunks = kDv / 64;             // 8
constexpr int kLatChunks = kDv / 64;           // 8 latent chunks: the Q part kept in TMEM
constexpr uint32_t kChunkBytes = kPage * 128;  // 64 tokens x 128 B = 8 KB
constexpr uint32_t kE4ChunkBytes = kPage * 64;             // one 64-code chunk of one e4m3 page: 4 KB
constexpr uint32_t kSlotBytes = kFp8 ? kKChunks * kE4ChunkBytes : 2 * kChunkBytes;  // 36 KB / 16 KB
constexpr uint32_t kVStageBytes = (kSparse ? kKChunks : kVChunks) * kChunkBytes;  // 64 KB (sparse: 72 KB page buffers)
constexpr uint32_t kPBytes = kTileRows * 128;             // 16 KB: 128 rows x 64 bf16, 128B-swizzled
constexpr uint32_t kFacOff = kPBytes;                      // then fac[128] (fp32)
constexpr uint32_t kInvLOff = kPBytes + kTileRows * 4;     // then inv_l[128] (fp32)
constexpr uint32_t kPMsgBytes = kPBytes + 2 * kTileRows * 4;  // 17 KB, a multiple of 1 KB
// e4m3 pages: q is split per row into three e4m3 parts, q / sigma_r ~ h + m + l
// (sigma_r = max |q_r| / 448), each contracted with the codes in fp8 on the
// tensor cores; the latent dims of the three parts sit in TMEM (four codes
// per column), their RoPE dims in 64-byte-swizzled shared tiles
constexpr int kQParts = kFp8 ? 3 : 1;
constexpr uint32_t kQPartCols = kDv / 4;                   // e4m3: one part's 512 latent codes = 128 columns
constexpr uint32_t kQCols = kFp8 ? kQParts * kQPartCols : kDv / 2;  // bf16: 256 columns of bf16 pairs
constexpr uint32_t kSCol0 = kQCols;                        // S buffers follow Q
constexpr uint32_t kSCols = kStepPages * kPage;            // an S buffer holds the scores of one step
constexpr uint32_t kTmemCols = 512;
static_assert(kSCol0 + kSBufs * kSCols <= kTmemCols, "tensor memory of the score CTA");
constexpr float kRescaleLog2 = 8.0f;                       // lazy rescale threshold (log2 units)
constexpr uint32_t kEpiCols = 64;                          // epilogue chunk: 64 fp32 columns
constexpr uint32_t kEpiStride = kEpiCols * 4 + 16;         // padded row stride (conflict-free v4 stores)

static_assert(!kFp8 || kD == kDqk, "the e4m3 cache holds 576-wide rows");
constexpr uint32_t kE4PageBytes = kPage * kD + kPage * 4;  // 64 rows of codes, then 64 fp32 scales
constexpr uint32_t kE4ScaleOff = kPage * kD;               // the scales' byte offset in a page
constexpr uint32_t kVLandOff = kVStageBytes / 2;           // e4m3 page landing inside a V stage (upper 32 KB)
constexpr float kE4ScaleLimit = 255.f;                     // |scale| bound: P (< 2^8) times it stays in f16 range
constexpr float kE4Max = 448.f;                            // largest finite e4m3 value
constexpr int kScSlots = 8;                                // side ring: one slot per step (a producer waits on
                                                           // the rows of 8 steps back: never in practice)
constexpr uint32_t kScBytes = kStepPages * kPage * 4;      // e4m3: the step's token scales; sparse: key masks
static_assert(kE4PageBytes % 16 == 0 && kE4ScaleOff % 16 == 0, "TMA and bulk-copy alignment of e4m3 pages");

// shared-memory layout (offsets from the 1024-byte aligned base)
// score CTA: [K operand rings 2 x 5 x 16 KB][Q RoPE tile 16 KB][P staging 2 x 17 KB];
// e4m3: [operand rings 2 x 2 x 36 KB][Q RoPE tiles 3 x 8 KB][P staging][scales 8 x 256 B];
// sparse: [page buffers 2 x 72 KB][Q RoPE][P staging][key masks 8 x 256 B]
constexpr uint32_t kKRingOff = 0;
constexpr uint32_t kQRopeOff = kKRingOff + (kSparse ? kVStages * kVStageBytes : kKSlots * kSlotBytes);
constexpr uint32_t kQRopePartBytes = kTileRows * (kFp8 ? 64 : 128);  // one part's [128 rows] RoPE tile
constexpr uint32_t kStageOff = kQRopeOff + (kHasRope ? kQParts * kQRopePartBytes : 0);
constexpr uint32_t kScaleOff = kStageOff + kPBufs * kPMsgBytes;   // the side ring of the steps in flight
constexpr uint32_t kScoreEnd = kScaleOff + (kRing ? kScSlots * kScBytes : 0);
// value CTA: [V ring 2 x 64 KB (sparse: the page buffers)][P landing 2 x 17 KB][epilogue staging 34 KB]
constexpr uint32_t kVRingOff = 0;
constexpr uint32_t kPBufOff = kVRingOff + kVStages * kVStageBytes;
constexpr uint32_t kEpiOff = kPBufOff + kPBufs * kPMsgBytes;
constexpr uint32_t kValueEnd = kEpiOff + kTileRows * kEpiStride;
// barriers at the same offset in both CTAs (the peer arrives on some of them)
constexpr uint32_t kBarOff = ((kScoreEnd > kValueEnd ? kScoreEnd : kValueEnd) + 1023u) & ~1023u;
static_assert(kQRopeOff % 1024 == 0 && kStageOff % 1024 == 0 && kPBufOff % 1024 == 0 && kPMsgBytes % 1024 == 0 &&
                  kSlotBytes % 1024 == 0,
              "swizzled tiles need 1 KB alignment");

enum Bar {
    // score CTA
    B_KFULL = 0, B_KEMPTY = B_KFULL + kKSlots, B_SFULL = B_KEMPTY + kKSlots, B_SEMPTY = B_SFULL + kSBufs,
    B_QFULL = B_SEMPTY + kSBufs, B_QACK = B_QFULL + 1, B_PFREE = B_QACK + 1,
    // value CTA
    B_VFULL = B_PFREE + kPBufs, B_VEMPTY = B_VFULL + kVStages, B_PFULL = B_VEMPTY + kVStages,
    B_PREADY = B_PFULL + kPBufs, B_PVDONE = B_PREADY + kPBufs, B_ODONE = B_PVDONE + 1, B_OEMPTY = B_ODONE + 1,
    // both
    B_FINAL = B_OEMPTY + 1, B_BASE_COUNT = B_FINAL + 1
};
// e4m3 pages and sparse lists: landing of the value CTA's codes (its row warps
// then widen them and arrive on B_VFULL), the score CTA's side ring, and the
// value CTA's read-before-write barrier of the in-place widening
constexpr int B_VLAND = B_BASE_COUNT, B_SCFULL = B_VLAND + kVStages, B_SCEMPTY = B_SCFULL + kScSlots,
              B_VREAD = B_SCEMPTY + kScSlots;
// sparse lists: one barrier per 64-dim chunk of each page buffer, at the same
// offset in both CTAs, so that the score MMAs can start on a page's first
// chunks while the rest are still being gathered
constexpr int B_CHUNK = B_VREAD + 1;
constexpr int B_COUNT = kSparse ? B_CHUNK + kVStages * kKChunks : (kRing ? B_VREAD + 1 : B_BASE_COUNT);
constexpr uint32_t kTmemSlotOff = kBarOff + B_COUNT * 8;
constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
constexpr uint32_t kSmemUsed = kAbortOff + 4;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack of the dynamic base
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kRingSlots * kScoreIssuers == kKSlots && kSBufs % kScoreIssuers == 0, "one K ring per score-MMA issuer");

// -------------------------------------------------------------- work walk
struct Segment {
    int b, T, n_pages, p0, p1, split, n_split;
};

struct PartWalk {
    int bb, bp, eb, ep, bs, b;
    __device__ void init(const DecodeParams &p, int part) {
        const int32_t *md = p.metadata + (size_t)part * kMdInts;
        bb = md[0];
        bp = md[1];
        eb = md[2];
        ep = md[3];
        bs = md[4];
        b = (bb == eb && bp == ep) ? p.batch : bb;  // an empty part walks nothing
        if (b < 0) b = p.batch;
    }
    __device__ bool next(const DecodeParams &p, Segment &s) {
        if (b >= p.batch || b > eb || (b == eb && ep == 0)) return false;
        int T = p.seqlens[b];  // sparse decode: the length of the sequence's lists
        if (T < 0) T = 0;
        if (!kSparse && T > p.max_blocks * kPage) T = p.max_blocks * kPage;
        s.b = b;
        s.T = T;
        s.n_pages = (T + kPage - 1) / kPage;
        s.p1 = (b == eb) ? min(ep, s.n_pages) : s.n_pages;
        s.p0 = (b == bb) ? min(bp, s.p1) : 0;
        s.split = (b == bb) ? bs : 0;
        s.n_split = p.num_splits[b + 1] - p.num_splits[b];
        ++b;
        return true;
    }
};

struct Ctx {
    uint8_t *base;
    uint64_t *bars;
    volatile int *abort_flag;
    unsigned int *status;
    uint32_t peer;  // the other CTA's rank
    __device__ uint64_t *bar(int i) const { return bars + i; }
};

// bounded wait that also gives up when this CTA was told to abort
template <bool kCluster = false>
__device__ __forceinline__ bool wait(const Ctx &c, int bar_idx, uint32_t parity) {
    const uint32_t a = smem_u32(c.bar(bar_idx));
    if (kCluster ? mbar_test_cluster(a, parity) : mbar_test(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (kCluster ? mbar_test_cluster(a, parity) : mbar_test(a, parity)) return true;
        if (*c.abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(c.status, MLA_DEVERR_TIMEOUT);
            *c.abort_flag = 1;
            // tell the peer CTA to stop waiting on us
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(smem_u32((const void *)c.abort_flag), c.peer)),
                         "r"(1)
                         : "memory");
            return false;
        }
    }
}

// the same wait taken by every lane of a warp, with one outcome for all of
// them (the row warps run warp-collective tcgen05.ld/st after their waits)
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(const Ctx &c, int bar_idx, uint32_t parity) {
    return __all_sync(0xffffffffu, wait<kCluster>(c, bar_idx, parity));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int safe_block(const DecodeParams &p, int b, int page) {
    const int blk = p.block_table[(size_t)b * p.max_blocks + page];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        atomicOr(p.status, MLA_DEVERR_BLOCK_ID);
        return 0;
    }
    return blk;
}

// instruction descriptor of both MMAs: bf16 operands, or f16 for the e4m3 cache
__host__ __device__ constexpr uint32_t idesc_op(int m, int n, bool a_mn_major, bool b_mn_major) {
    return kFp8 ? idesc_f16(m, n, a_mn_major, b_mn_major) : idesc_bf16(m, n, a_mn_major, b_mn_major);
}

// In-place widening of e4m3 codes to f16 MMA operand rows.  Row R's 64 codes
// sit at land + 64 R, as the TMA left them (no swizzle); its 64 f16 values go
// to base + 128 R with the 128-byte swizzle of the operand descriptors (16-byte
// piece c of row R at piece c ^ (R % 8)).  The landing area is the upper half
// of the same buffer, so writing the upper rows overwrites codes: each of the
// group's kGroup threads reads all of its kItems 16-byte items first (item
// g = i * kGroup + tid: row g / 4, codes 16 (g % 4) .. + 15), then `sync()`
// must order every read of the group before any write, then the rows are
// written.  Rows R with R % 64 >= keep are written as zeros.  Returns false,
// having written nothing, when `sync()` does.
template <int kItems, int kGroup, typename Sync>
__device__ __forceinline__ bool widen_e4m3(uint32_t base, uint32_t land, int tid, int keep, Sync sync) {
    uint4 x[kItems];
#pragma unroll
    for (int i = 0; i < kItems; ++i) x[i] = lds128(land + 16u * (uint32_t)(i * kGroup + tid));
    if (!sync()) return false;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const int g = i * kGroup + tid;
        const int R = g >> 2, piece = g & 3;
        const uint32_t row = base + 128u * (uint32_t)R;
        uint32_t w[8] = {e4m3x2_to_f16x2(x[i].x), e4m3x2_to_f16x2(x[i].x >> 16), e4m3x2_to_f16x2(x[i].y),
                         e4m3x2_to_f16x2(x[i].y >> 16), e4m3x2_to_f16x2(x[i].z), e4m3x2_to_f16x2(x[i].z >> 16),
                         e4m3x2_to_f16x2(x[i].w), e4m3x2_to_f16x2(x[i].w >> 16)};
        if ((R & (kPage - 1)) >= keep) {
#pragma unroll
            for (int t = 0; t < 8; ++t) w[t] = 0u;
        }
        sts128(row + 16u * (uint32_t)((2 * piece) ^ (R & 7)), w[0], w[1], w[2], w[3]);
        sts128(row + 16u * (uint32_t)((2 * piece + 1) ^ (R & 7)), w[4], w[5], w[6], w[7]);
    }
    return true;
}

// -------------------------------------------------------------- roles
// Score-CTA TMA producers (one lane each, one per MMA issuer's ring `r`,
// taking the steps of parity r).  A step is up to two consecutive pages
// of a segment; each of a step's 9 64-dim chunks is one 16 KB ring slot
// holding 128 token rows (first page rows 0-63, second page rows 64-127), so
// that one tcgen05 MMA with N = 128 covers both pages.  Producer 0 asks L2 for
// each segment's Q rows as it reaches the segment.  (Streaming whole pages into L2 ahead
// of the chunk loads, from either CTA and at any distance tried, measured
// slower on GB300 than letting the chunk loads fetch them.)
__device__ void score_producer(const DecodeParams &p, const Ctx &c, const CUtensorMap *map, int part, int tile,
                               int r) {
    PartWalk walk;
    Segment s;
    {
        // the block-table line of the part's first page travels while the
        // walk reads the sequence lengths (one dependent round trip fewer
        // before the first chunk load)
        const int32_t *md = p.metadata + (size_t)part * kMdInts;
        const int bb = md[0], bp = md[1];
        if (bb >= 0 && bb < p.batch && bp >= 0 && bp < p.max_blocks)
            prefetch_line_l1(p.block_table + (size_t)bb * p.max_blocks + bp);
    }
    const int rows = min(kTileRows, p.rows - tile * kTileRows);
    walk.init(p, part);
    uint32_t ring_it = 0;  // chunks issued into this producer's ring
    uint32_t step = 0;
    bool ok = true;
    while (ok && walk.next(p, s)) {
        // producer 0 asks L2 for the segment's Q rows as it reaches the
        // segment, a few pages before the row warps load them (a prefetch at
        // the part's start would be evicted by the pages streamed meanwhile)
        if (r == 0 && s.p1 > s.p0 && rows > 0)
            prefetch_l2(p.q + ((size_t)s.b * p.rows + (size_t)tile * kTileRows) * kD, (uint32_t)rows * kD * 2);
        for (int pg = s.p0; ok && pg < s.p1; pg += 2, ++step) {
            const int npg = min(2, s.p1 - pg);
            if ((int)(step % kScoreIssuers) != r) continue;  // the other ring's step
            const int blk0 = safe_block(p, s.b, pg);
            const int blk1 = npg > 1 ? safe_block(p, s.b, pg + 1) : 0;
            for (int ch = 0; ch < kKChunks; ++ch) {
                const uint32_t k = ring_it++;
                const int sl = r * kRingSlots + (int)(k % kRingSlots);
                if (!wait(c, B_KEMPTY + sl, ((k / kRingSlots) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
#ifdef MLA_TEST_SKIP_ONE_LOAD
                // test builds only: part 0 never loads its third chunk, so the
                // slot's barrier never completes and the MMA issuer's bounded
                // wait must run out (MLA_DEVERR_TIMEOUT) and unwind the pair
                if (part == 0 && tile == 0 && r == 0 && k == 2) continue;
#endif
                uint8_t *dst = c.base + kKRingOff + sl * kSlotBytes;
                mbar_arrive_expect_tx(c.bar(B_KFULL + sl), npg * kChunkBytes);
                tma_load_3d(dst, map, c.bar(B_KFULL + sl), 64 * ch, 0, blk0);
                if (npg > 1) tma_load_3d(dst + kChunkBytes, map, c.bar(B_KFULL + sl), 64 * ch, 0, blk1);
            }
        }
    }
    // the last loads must have landed before this CTA may exit (already true
    // on the normal path, where the MMAs consumed them)
    for (uint32_t k = ring_it > (uint32_t)kRingSlots ? ring_it - kRingSlots : 0; k < ring_it; ++k)
        mbar_wait(c.bar(B_KFULL + r * kRingSlots + (int)(k % kRingSlots)), (k / kRingSlots) & 1, c.status);
}

// Score-CTA TMA producer for e4m3 pages (one lane per issuer's ring `r`,
// taking the steps of parity r).  A step is one page: its slot receives the
// page's nine 64-code chunks as 64-byte-swizzled [64 x 64 B] tiles, which the
// fp8 MMAs read as they are, and the page's 64 per-token scales go to the side
// ring (one 256 B bulk copy).
__device__ void score_producer_e4m3(const DecodeParams &p, const Ctx &c, const CUtensorMap *map, int part, int r) {
    const uint8_t *kv = reinterpret_cast<const uint8_t *>(p.kcache);
    PartWalk walk;
    Segment s;
    walk.init(p, part);
    uint32_t ring_it = 0, step = 0, own = 0;
    bool ok = true;
    while (ok && walk.next(p, s)) {
        for (int pg = s.p0; ok && pg < s.p1; ++pg, ++step) {
            if ((int)(step % kScoreIssuers) != r) continue;  // the other ring's step
            const int blk = safe_block(p, s.b, pg);
            const int sc = (int)(step % kScSlots);
            if (!wait(c, B_SCEMPTY + sc, ((step / kScSlots) & 1) ^ 1)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(c.bar(B_SCFULL + sc), kPage * 4);
            bulk_load(c.base + kScaleOff + sc * kScBytes, kv + (size_t)blk * kE4PageBytes + kE4ScaleOff, kPage * 4,
                      c.bar(B_SCFULL + sc));
            ++own;
            const uint32_t k = ring_it;
            const int sl = r * kRingSlots + (int)(k % kRingSlots);
            if (!wait(c, B_KEMPTY + sl, ((k / kRingSlots) & 1) ^ 1)) {
                ok = false;
                break;
            }
            uint8_t *dst = c.base + kKRingOff + sl * kSlotBytes;
            mbar_arrive_expect_tx(c.bar(B_KFULL + sl), kSlotBytes);
            for (int ch = 0; ch < kKChunks; ++ch)
                tma_load_3d(dst + ch * kE4ChunkBytes, map, c.bar(B_KFULL + sl), 64 * ch, 0, blk);
            ++ring_it;
        }
    }
    // the last loads must have landed before this CTA may exit (already true
    // on the normal path, where the MMAs and the row warps consumed them)
    for (uint32_t k = ring_it > (uint32_t)kRingSlots ? ring_it - kRingSlots : 0; k < ring_it; ++k)
        mbar_wait(c.bar(B_KFULL + r * kRingSlots + (int)(k % kRingSlots)), (k / kRingSlots) & 1, c.status);
    const uint32_t back = own < (uint32_t)(kScSlots / kScoreIssuers) ? own : (uint32_t)(kScSlots / kScoreIssuers);
    for (uint32_t i = own - back; i < own; ++i) {
        const uint32_t st = (uint32_t)kScoreIssuers * i + (uint32_t)r;  // this ring's steps: every other step
        mbar_wait(c.bar(B_SCFULL + (int)(st % kScSlots)), (st / kScSlots) & 1, c.status);
    }
}

// -------------------------------------------------------------- sparse top-k gathers
// A part walks list chunks instead of pages: "page" pg of sequence b is list
// entries 64 pg .. 64 pg + 63 of the tile's query token, and entry e names a
// token position; positions outside [0, kv_lens[b]) and entries past the
// list's length are invalid.  Rows are gathered with TMA four at a time
// (tile::gather4 over the cache viewed as a 2-D tensor of 64 num_blocks rows
// of d elements), straight into the 128-byte-swizzled operand layout; an
// invalid entry is given the row just past the cache, which the gather reads
// as zeros (its score column is masked by the row warps, its V row adds 0).

__device__ __forceinline__ int sparse_cache_len(const DecodeParams &p, int b) {
    int T = p.kv_lens[b];
    return T < 0 ? 0 : (T > p.max_blocks * kPage ? p.max_blocks * kPage : T);
}

// Cache rows of list entries e0 .. e0 + 3 of `list` (y[j], or the row past the
// cache), and bit j of the result set when entry e0 + j is valid.  Lanes with
// `on` false get four invalid entries.
__device__ __forceinline__ uint32_t sparse_rows(const DecodeParams &p, const int32_t *list, int list_len, int T, int b,
                                               int e0, bool on, int (&y)[4]) {
    const int past = (int)(p.num_blocks * kPage);
    int pos[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pos[j] = (on && e0 + j < list_len) ? list[e0 + j] : -1;
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        y[j] = past;
        if (pos[j] >= 0 && pos[j] < T) {
            const int blk = p.block_table[(size_t)b * p.max_blocks + pos[j] / kPage];
            if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                atomicOr(p.status, MLA_DEVERR_BLOCK_ID);
            } else {
                y[j] = blk * kPage + pos[j] % kPage;
                valid |= 1u << j;
            }
        }
    }
    return valid;
}

// bit i of x (i < 16) to bit 4 i
__device__ __forceinline__ uint64_t spread4(uint32_t x) {
    uint64_t v = x & 0xFFFFu;
    v = (v | (v << 24)) & 0x000000FF000000FFull;
    v = (v | (v << 12)) & 0x000F000F000F000Full;
    v = (v | (v << 6)) & 0x0303030303030303ull;
    v = (v | (v << 3)) & 0x1111111111111111ull;
    return v;
}

// Sparse decode: the gathers of a page are split between the two CTAs of the
// pair.  Both CTAs resolve the page's list entries to cache rows (lane i < 16:
// entries 4 i .. 4 i + 3) and gather four rows per lane and 64-dim chunk into
// page buffer it % 2: the score CTA chunks 0..2 and rows 0..31 of chunk 3,
// multicast to both CTAs, and the RoPE chunk 8 into its own buffer only; the
// value CTA rows 32..63 of chunk 3 and chunks 4..7, multicast to both (4.5
// chunks each).  Each CTA's barrier of the buffer expects the bytes that
// land in that CTA (72 KB, 64 KB); a peer's bytes may complete on it before
// the CTA has armed it, which the barrier's transaction count allows.  A
// buffer is refilled only after the value CTA's P V of the page two earlier,
// which follows the score CTA's MMAs of that page: the value producer waits
// for it on its own barrier, the score producer on the P-free barrier that
// the same MMA commit arrives on.  The variant built with
// MLA_SPARSE_MULTICAST = 0 keeps the buffers, barriers and hand-offs but has
// each CTA gather every chunk it uses itself, with no multicast: processes
// that run one job across several GPUs select it (mla_set_cluster_multicast).
constexpr int kSparseSplitChunk = 3;   // chunks below: the score CTA's; above: the value CTA's; this one by halves
constexpr uint16_t kPairMask = 0x3;    // both CTAs of the cluster

// Score-CTA producer of the sparse decode (the whole warp).  The validity mask
// of each page's list chunk goes to the side ring for the row warps.  (The
// gathers run at the TMA engine's rate for 128-byte row pieces, about 10 GB/s
// per SM on GB300, which bounds this decode.)
__device__ void score_producer_sparse(const DecodeParams &p, const Ctx &c, const CUtensorMap *map, int part,
                                      int tile) {
    const int lane = threadIdx.x & 31;
    const int qtok = p.s_q == 1 ? 0 : tile;  // the tile's query token (h_q = 128 when s_q > 1)
    PartWalk walk;
    Segment s;
    walk.init(p, part);
    uint32_t it = 0;
    bool ok = true;
    while (ok && walk.next(p, s)) {
        const int T = sparse_cache_len(p, s.b);
        const int32_t *list = p.indices + ((size_t)s.b * p.s_q + qtok) * p.topk;
        const int list_len = min(s.T, p.topk);
        for (int pg = s.p0; ok && pg < s.p1; ++pg, ++it) {
            const int b = (int)(it % kVStages);
            int y[4];
            const uint32_t v = sparse_rows(p, list, list_len, T, s.b, kPage * pg + 4 * lane, lane < 16, y);
            const uint32_t b0 = __ballot_sync(0xffffffffu, v & 1u), b1 = __ballot_sync(0xffffffffu, v & 2u),
                           b2 = __ballot_sync(0xffffffffu, v & 4u), b3 = __ballot_sync(0xffffffffu, v & 8u);
            const int sc = (int)(it % kScSlots);
            if (!warp_wait(c, B_SCEMPTY + sc, ((it / kScSlots) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                // row 4 i + j of the page is bit i of ballot j
                const uint64_t ma = spread4(b0) | spread4(b1) << 1 | spread4(b2) << 2 | spread4(b3) << 3;
                sts128(smem_u32(c.base + kScaleOff + sc * kScBytes), (uint32_t)ma, (uint32_t)(ma >> 32), 0u, 0u);
                mbar_arrive(c.bar(B_SCFULL + sc));
            }
            // page buffer b is free in both CTAs once the P V of page it - 2 is done
            if (!warp_wait<true>(c, B_PFREE + b, ((it / kPBufs) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane < kKChunks) mbar_arrive_expect_tx(c.bar(B_CHUNK + b * kKChunks + lane), kChunkBytes);
            __syncwarp();
            if (lane < 16) {
                const uint32_t buf = smem_u32(c.base + kKRingOff + b * kVStageBytes) + 512u * (uint32_t)lane;
                tma_gather4(buf + (uint32_t)kLatChunks * kChunkBytes, map, c.bar(B_CHUNK + b * kKChunks + kLatChunks),
                            64 * kLatChunks, y[0], y[1], y[2], y[3]);
#pragma unroll
                for (int ch = 0; ch < kLatChunks; ++ch) {
                    if constexpr (kPairGather) {
                        if (ch < kSparseSplitChunk || (ch == kSparseSplitChunk && lane < 8))
                            tma_gather4_multicast(buf + (uint32_t)ch * kChunkBytes, map,
                                                  c.bar(B_CHUNK + b * kKChunks + ch), 64 * ch, y[0], y[1], y[2], y[3],
                                                  kPairMask);
                    } else {
                        tma_gather4(buf + (uint32_t)ch * kChunkBytes, map, c.bar(B_CHUNK + b * kKChunks + ch), 64 * ch,
                                    y[0], y[1], y[2], y[3]);
                    }
                }
            }
        }
    }
    // the last pages' bytes (ours and the peer's) must have landed before
    // this CTA may exit (already true on the normal path, where the MMAs
    // waited for them)
    if (lane < kKChunks)
        for (uint32_t k = it > (uint32_t)kVStages ? it - kVStages : 0; k < it; ++k)
            mbar_wait(c.bar(B_CHUNK + (int)(k % kVStages) * kKChunks + lane), (k / kVStages) & 1, c.status);
    __syncwarp();
}

// Value-CTA producer of the sparse decode (the whole warp): rows 32..63 of
// chunk 3 and chunks 4..7 of each page, multicast to both CTAs.
__device__ void value_producer_sparse(const DecodeParams &p, const Ctx &c, const CUtensorMap *map, int part,
                                      int tile) {
    const int lane = threadIdx.x & 31;
    const int qtok = p.s_q == 1 ? 0 : tile;
    PartWalk walk;
    Segment s;
    walk.init(p, part);
    uint32_t it = 0;
    bool ok = true;
    while (ok && walk.next(p, s)) {
        const int T = sparse_cache_len(p, s.b);
        const int32_t *list = p.indices + ((size_t)s.b * p.s_q + qtok) * p.topk;
        const int list_len = min(s.T, p.topk);
        for (int pg = s.p0; pg < s.p1; ++pg, ++it) {
            const int b = (int)(it % kVStages);
            int y[4];
            sparse_rows(p, list, list_len, T, s.b, kPage * pg + 4 * lane, lane < 16, y);
            if (!warp_wait(c, B_VEMPTY + b, ((it / kVStages) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane < kVChunks) mbar_arrive_expect_tx(c.bar(B_CHUNK + b * kKChunks + lane), kChunkBytes);
            __syncwarp();
            if (lane < 16) {
                const uint32_t buf = smem_u32(c.base + kVRingOff + b * kVStageBytes) + 512u * (uint32_t)lane;
#pragma unroll
                for (int ch = 0; ch < kVChunks; ++ch) {
                    if constexpr (kPairGather) {
                        if (ch > kSparseSplitChunk || (ch == kSparseSplitChunk && lane >= 8))
                            tma_gather4_multicast(buf + (uint32_t)ch * kChunkBytes, map,
                                                  c.bar(B_CHUNK + b * kKChunks + ch), 64 * ch, y[0], y[1], y[2], y[3],
                                                  kPairMask);
                    } else {
                        tma_gather4(buf + (uint32_t)ch * kChunkBytes, map, c.bar(B_CHUNK + b * kKChunks + ch), 64 * ch,
                                    y[0], y[1], y[2], y[3]);
                    }
                }
            }
        }
    }
    if (lane < kVChunks)
        for (uint32_t k = it > (uint32_t)kVStages ? it - kVStages : 0; k < it; ++k)
            mbar_wait(c.bar(B_CHUNK + (int)(k % kVStages) * kKChunks + lane), (k / kVStages) & 1, c.status);
    __syncwarp();
}

// Value-CTA TMA producer (one lane): whole pages (dims 0..511) through the V
// ring (e4m3 cache: the page's 32 KB of codes into the upper half of the stage,
// completing on B_VLAND; the row warps widen them and arrive on B_VFULL).
__device__ void value_producer(const DecodeParams &p, const Ctx &c, const CUtensorMap *map, int part) {
    PartWalk walk;
    Segment s;
    walk.init(p, part);
    uint32_t it = 0;
    bool ok = true;
    while (ok && walk.next(p, s)) {
        for (int pg = s.p0; pg < s.p1; ++pg, ++it) {
            const int st = it % kVStages;
            if (!wait(c, B_VEMPTY + st, ((it / kVStages) & 1) ^ 1)) {
                ok = false;
                break;
            }
            const int blk = safe_block(p, s.b, pg);
            uint8_t *dst = c.base + kVRingOff + st * kVStageBytes;
            if constexpr (kFp8) {
                mbar_arrive_expect_tx(c.bar(B_VLAND + st), kVChunks * kE4ChunkBytes);
                for (int ch = 0; ch < kVChunks; ++ch)
                    tma_load_3d(dst + kVLandOff + ch * kE4ChunkBytes, map, c.bar(B_VLAND + st), 64 * ch, 0, blk);
            } else {
                mbar_arrive_expect_tx(c.bar(B_VFULL + st), kVStageBytes);
                for (int ch = 0; ch < kVChunks; ++ch)
                    tma_load_3d(dst + ch * kChunkBytes, map, c.bar(B_VFULL + st), 64 * ch, 0, blk);
            }
        }
    }
    constexpr int land = kFp8 ? B_VLAND : B_VFULL;  // the barrier the loads complete on
    for (uint32_t k = it > (uint32_t)kVStages ? it - kVStages : 0; k < it; ++k)
        mbar_wait(c.bar(land + (int)(k % kVStages)), (k / kVStages) & 1, c.status);
}

// Score-CTA MMA issuers: S[buf] = Q K^T for every step of (up to) two pages:
// the 512 latent dims with A = Q from TMEM, the 64 RoPE dims with A = the
// Q RoPE tile in shared memory; B = the 128 (or 64) token rows of each slot.
// A tcgen05.mma holds its issuing thread for about its own execution time, so
// whatever that thread does between MMAs (barrier waits, commits, loop
// bookkeeping) leaves the tensor pipe idle.  Two issuers therefore alternate
// steps by global step index (`lane` 0: even steps into S buffer 0, 1: odd
// steps into buffer 1): one's bookkeeping overlaps the other's MMAs.  Each
// issuer has its own ring of chunk slots, filled in step order by the
// producer and consumed in order by its only consumer: with a shared ring, an
// issuer could test a slot's barrier for a later phase while the other
// issuer's earlier chunk in that slot had not landed, which parity waits
// cannot tell apart.  Both issuers also wait for every segment's Q, so that
// their view of the Q barrier's phases stays exact.
__device__ void score_mma(const DecodeParams &p, const Ctx &c, uint32_t tmem, int part, int lane) {
    PartWalk walk;
    walk.init(p, part);
    Segment s;
    uint32_t step = 0, seg = 0, ring_it = 0;  // ring_it: chunks consumed from this issuer's own ring
    const uint32_t ring = smem_u32(c.base + kKRingOff);
    const uint64_t rope_desc = desc_sw128(smem_u32(c.base + kQRopeOff), 16, 1024);
    while (walk.next(p, s)) {
        const int nsteps = (s.p1 - s.p0 + kStepPages - 1) / kStepPages;
        if (!wait(c, B_QFULL, seg & 1)) return;  // Q of this segment is in TMEM and smem
        tc_fence_after();
        mbar_arrive(c.bar(B_QACK));              // the row warps may load the next Q only after both issuers saw this one
        ++seg;
        for (int j = 0; j < nsteps; ++j) {
            const uint32_t st = step + j;       // global step index
            if ((int)(st % kScoreIssuers) != lane) continue;
            const int sb = (int)(st % kSBufs);
            const uint32_t d = tmem + kSCol0 + sb * kSCols;
            const int npg = min(kStepPages, s.p1 - (s.p0 + kStepPages * j));
            const uint32_t idesc = npg == 2 ? idesc_op(kTileRows, 2 * kPage, false, false)
                                            : idesc_op(kTileRows, kPage, false, false);
            if (!wait(c, B_SEMPTY + sb, ((st / kSBufs) & 1) ^ 1)) return;
            tc_fence_after();  // the row warps' reads of this S buffer come first
            if constexpr (kFp8) {
                // one page: S = sum over Q's three e4m3 parts t and the nine
                // 64-code chunks of (part t) x (codes)^T, two K = 32 MMAs per
                // chunk and part; A from TMEM (latent) or the part's RoPE tile
                const uint32_t sl = lane * kRingSlots + ring_it % kRingSlots;
                if (!wait(c, B_KFULL + sl, (ring_it / kRingSlots) & 1)) return;
                const uint32_t slot = ring + sl * kSlotBytes;
                constexpr uint32_t id8 = idesc_e4m3(kTileRows, kPage);
#pragma unroll 1
                for (int ch = 0; ch < kKChunks; ++ch) {
                    const uint32_t b = slot + ch * kE4ChunkBytes;
#pragma unroll
                    for (int t = 0; t < kQParts; ++t) {
                        if (ch < kLatChunks) {
                            const uint32_t a = tmem + t * kQPartCols + ch * 16;
                            mma_ts_f8(d, a, desc_sw64(b), id8, (ch | t) ? 1u : 0u);
                            mma_ts_f8(d, a + 8, desc_sw64(b + 32), id8, 1u);
                        } else {
                            const uint32_t ar = smem_u32(c.base + kQRopeOff) + t * kQRopePartBytes;
                            mma_ss_f8(d, desc_sw64(ar), desc_sw64(b), id8, 1u);
                            mma_ss_f8(d, desc_sw64(ar + 32), desc_sw64(b + 32), id8, 1u);
                        }
                    }
                }
                mma_commit(c.bar(B_KEMPTY + sl));
                ++ring_it;
                mma_commit(c.bar(B_SFULL + sb));
                continue;
            }
            if constexpr (kSparse) {
                // one page from page buffer st % 2, each chunk as soon as it
                // has landed, in the order the two CTAs' gathers complete
                const int pb = (int)(st % kVStages);
                const uint32_t buf = ring + pb * kVStageBytes;
#pragma unroll 1
                for (int i = 0; i < kKChunks; ++i) {
                    // 8, then 0, 4, 1, 5, 2, 6, 3, 7: the two CTAs' gather queues interleaved
                    const int ch = i == 0 ? kLatChunks : (((i - 1) & 1) ? 4 + ((i - 1) >> 1) : ((i - 1) >> 1));
                    if (!wait(c, B_CHUNK + pb * kKChunks + ch, (st / kVStages) & 1)) return;
                    const uint64_t bd = desc_sw128(buf + ch * kChunkBytes, 16, 1024);
                    if (ch < kLatChunks) {
                        const uint32_t a = tmem + ch * 32;
                        mma_ts(d, a, bd, idesc, i != 0);
                        mma_ts(d, a + 8, bd + 2, idesc, 1u);
                        mma_ts(d, a + 16, bd + 4, idesc, 1u);
                        mma_ts(d, a + 24, bd + 6, idesc, 1u);
                    } else {
                        mma_ss(d, rope_desc, bd, idesc, i != 0);
                        mma_ss(d, rope_desc + 2, bd + 2, idesc, 1u);
                        mma_ss(d, rope_desc + 4, bd + 4, idesc, 1u);
                        mma_ss(d, rope_desc + 6, bd + 6, idesc, 1u);
                    }
                }
                mma_commit(c.bar(B_SFULL + sb));
                continue;
            }
            for (int ch = 0; ch < kKChunks; ++ch, ++ring_it) {
                const uint32_t sl = lane * kRingSlots + ring_it % kRingSlots;
                // TMA data: the barrier's completion already orders it before
                // the MMA's reads (no tcgen05 fence here: it would drain the pipe)
                if (!wait(c, B_KFULL + sl, (ring_it / kRingSlots) & 1)) return;
                const uint64_t bd = desc_sw128(ring + sl * kSlotBytes, 16, 1024);
                if (!kHasRope || ch < kLatChunks) {
                    const uint32_t a = tmem + ch * 32;
                    mma_ts(d, a, bd, idesc, ch != 0);
                    mma_ts(d, a + 8, bd + 2, idesc, 1u);   // +32 B along K: descriptor address field +2
                    mma_ts(d, a + 16, bd + 4, idesc, 1u);
                    mma_ts(d, a + 24, bd + 6, idesc, 1u);
                } else {
                    mma_ss(d, rope_desc, bd, idesc, 1u);
                    mma_ss(d, rope_desc + 2, bd + 2, idesc, 1u);
                    mma_ss(d, rope_desc + 4, bd + 4, idesc, 1u);
                    mma_ss(d, rope_desc + 6, bd + 6, idesc, 1u);
                }
                mma_commit(c.bar(B_KEMPTY + sl));
            }
            mma_commit(c.bar(B_SFULL + sb));
        }
        step += nsteps;
    }
}

// Value-CTA MMA issuer: O (+)= P V for every page.  Only segments with pages
// touch O, so only they count on the O barriers: the epilogue of a segment
// without pages never waits on this thread, and counting it would let the row
// warps complete two phases of the O-free barrier between two of its waits.
__device__ void value_mma(const DecodeParams &p, const Ctx &c, uint32_t tmem, int part) {
    constexpr uint32_t idesc = idesc_op(kTileRows, 256, false, true);
    PartWalk walk;
    walk.init(p, part);
    Segment s;
    uint32_t it = 0, oseg = 0;  // oseg: segments with pages so far
    while (walk.next(p, s)) {
        if (s.p1 <= s.p0) continue;
        if (!wait(c, B_OEMPTY, (oseg & 1) ^ 1)) return;  // previous segment's epilogue has read O
        ++oseg;
        for (int pg = s.p0; pg < s.p1; ++pg, ++it) {
            const int st = it % kVStages, pb = it % kPBufs;
            if constexpr (kSparse) {
                // every value chunk of the page buffer (gathered by both CTAs)
                for (int ch = 0; ch < kVChunks; ++ch)
                    if (!wait(c, B_CHUNK + st * kKChunks + ch, (it / kVStages) & 1)) return;
            } else if (!wait(c, B_VFULL + st, (it / kVStages) & 1)) {
                return;
            }
            if (!wait(c, B_PREADY + pb, (it / kPBufs) & 1)) return;
            tc_fence_after();
            const uint32_t vtile = smem_u32(c.base + kVRingOff + st * kVStageBytes);
            const uint32_t ptile = smem_u32(c.base + kPBufOff + pb * kPMsgBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < kPage / 16; ++k) {
                    const uint64_t ad = desc_sw128(ptile + k * 32, 16, 1024);
                    const uint64_t bd = desc_sw128(vtile + h * 4 * kChunkBytes + k * 2048, kChunkBytes, 1024);
                    mma_ss(tmem + h * 256, ad, bd, idesc, (pg > s.p0 || k > 0) ? 1u : 0u);
                }
            mma_commit(c.bar(B_VEMPTY + st));
            mma_commit(c.bar(B_PVDONE));
            if (pg == s.p1 - 1) mma_commit(c.bar(B_ODONE));  // O of the segment is complete
            mma_commit_multicast(c.bar(B_PFREE + pb), (uint16_t)(1u << c.peer));
        }
    }
}

// Score-CTA row warps: Q -> TMEM and smem, masked online softmax, P and row
// factors -> staging -> bulk copies into the value CTA, each warp sending its
// own 32 rows as soon as they are staged.
__device__ void score_rows(const DecodeParams &p, const Ctx &c, uint32_t tmem, int part, int tile) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 32 * (warp & 3) + lane;                // tile row = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int gr = tile * kTileRows + r;                 // row within the sequence's rows
    const bool row_ok = gr < p.rows;
    const int qi = row_ok ? gr / p.h_q : 0;              // query token index
    const uint32_t peer_buf = mapa(smem_u32(c.base + kPBufOff), c.peer);
    const uint32_t peer_pfull = mapa(smem_u32(c.bar(B_PFULL)), c.peer);
    PartWalk walk;
    walk.init(p, part);
    Segment s;
    uint32_t it = 0, step = 0, seg = 0;
    while (walk.next(p, s)) {
        const int T_row = p.causal ? s.T - p.s_q + qi + 1 : s.T;
        // both MMA issuers have seen the previous segment's Q (and, having
        // consumed all its S buffers, the MMAs reading it are done)
        if (seg > 0 && !warp_wait(c, B_QACK, (seg - 1) & 1)) return;
        ++seg;
        float qsig = 1.f;  // e4m3 pages: this row's Q scale (q ~ qsig * (h + m + l))
        if (s.p1 > s.p0) {
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + ((size_t)s.b * p.rows + (row_ok ? gr : 0)) * kD);
            if constexpr (kFp8) {
                // Q row r as three e4m3 parts of q / qsig (qsig = max |q| / 448):
                // h = e4m3(x), m = e4m3(x - h), l = e4m3(x - h - m); latent dims
                // into TMEM lane r (part t at columns 128 t + dim / 4), RoPE dims
                // into row r of part t's 64-byte-swizzled tile
                float amax = 0.f;
#pragma unroll 1
                for (int j0 = 0; j0 < kD / 8; j0 += 24) {
                    uint4 x[24];
#pragma unroll
                    for (int j = 0; j < 24; ++j) x[j] = row_ok ? __ldg(qrow + j0 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < 24; ++j) {
                        const uint32_t w4[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            amax = max3f(amax, fabsf(__uint_as_float(w4[e] << 16)),
                                         fabsf(__uint_as_float(w4[e] & 0xffff0000u)));
                    }
                }
                qsig = amax > 0.f ? amax / kE4Max : 1.f;
                const float inv = 1.f / qsig;
                // one 64-dim chunk: three parts of 16 words (four codes each)
                auto split = [&](const uint4 (&x)[8], uint32_t (&ph)[16], uint32_t (&pm)[16], uint32_t (&pl)[16]) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t w4[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
                        for (int hw = 0; hw < 2; ++hw) {
                            float v[4];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                v[2 * e] = __uint_as_float(w4[2 * hw + e] << 16) * inv;
                                v[2 * e + 1] = __uint_as_float(w4[2 * hw + e] & 0xffff0000u) * inv;
                            }
                            uint32_t code[3];
#pragma unroll
                            for (int t = 0; t < 3; ++t) {
                                const uint32_t c01 = pack_e4m3x2(v[0], v[1]), c23 = pack_e4m3x2(v[2], v[3]);
                                code[t] = c01 | (c23 << 16);
                                if (t < 2) {
                                    float d0, d1, d2, d3;
                                    f16x2_to_f32(e4m3x2_to_f16x2(c01), d0, d1);
                                    f16x2_to_f32(e4m3x2_to_f16x2(c23), d2, d3);
                                    v[0] -= d0;
                                    v[1] -= d1;
                                    v[2] -= d2;
                                    v[3] -= d3;
                                }
                            }
                            ph[2 * j + hw] = code[0];
                            pm[2 * j + hw] = code[1];
                            pl[2 * j + hw] = code[2];
                        }
                    }
                };
#pragma unroll 1
                for (int ch = 0; ch < kKChunks; ++ch) {
                    // three chunks' loads per round (the first pass brought the row into L1)
                    uint4 x[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = row_ok ? __ldg(qrow + ch * 8 + j) : make_uint4(0, 0, 0, 0);
                    if (ch % 3 == 0 && ch + 2 < kKChunks && row_ok) {
                        prefetch_line_l1(qrow + (ch + 1) * 8);
                        prefetch_line_l1(qrow + (ch + 1) * 8 + 4);
                        prefetch_line_l1(qrow + (ch + 2) * 8);
                        prefetch_line_l1(qrow + (ch + 2) * 8 + 4);
                    }
                    uint32_t ph[16], pm[16], pl[16];
                    split(x, ph, pm, pl);
                    if (ch < kLatChunks) {
                        tmem_st16(tmem + lane_base + 0 * kQPartCols + ch * 16, ph);
                        tmem_st16(tmem + lane_base + 1 * kQPartCols + ch * 16, pm);
                        tmem_st16(tmem + lane_base + 2 * kQPartCols + ch * 16, pl);
                    } else {
                        // 64 B per row; 16-byte piece q of row r at q ^ ((r >> 1) & 3)
                        const uint32_t rope = smem_u32(c.base + kQRopeOff) + (uint32_t)r * 64u;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t off = 16u * (uint32_t)(q ^ ((r >> 1) & 3));
                            sts128(rope + off, ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
                            sts128(rope + kQRopePartBytes + off, pm[4 * q], pm[4 * q + 1], pm[4 * q + 2], pm[4 * q + 3]);
                            sts128(rope + 2 * kQRopePartBytes + off, pl[4 * q], pl[4 * q + 1], pl[4 * q + 2],
                                   pl[4 * q + 3]);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tmem_wait_st();
            } else {
            // Q row r: latent dims 0..511 into TMEM lane r (columns 0..255,
            // bf16 pairs), RoPE dims 512..575 into row r of the swizzled smem
            // tile.  Two rounds of loads: the RoPE chunk with latent chunks
            // 0..3 (40 loads in flight), then chunks 4..7.
            uint4 y[kHasRope ? 8 : 1];
            if constexpr (kHasRope) {
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] = row_ok ? __ldg(qrow + kLatChunks * 8 + j) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll 1
            for (int ch0 = 0; ch0 < kLatChunks; ch0 += 4) {
                uint4 x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = row_ok ? __ldg(qrow + ch0 * 8 + j) : make_uint4(0, 0, 0, 0);
                if (kHasRope && ch0 == 0) {
                    const uint32_t rope = smem_u32(c.base + kQRopeOff) + (uint32_t)r * 128u;
#pragma unroll
                    for (int j = 0; j < (kHasRope ? 8 : 0); ++j)
                        sts128(rope + 16u * (uint32_t)(j ^ (r & 7)), y[j].x, y[j].y, y[j].z, y[j].w);
                    fence_proxy_async_smem();
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t v[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[4 * j] = x[8 * k + j].x;
                        v[4 * j + 1] = x[8 * k + j].y;
                        v[4 * j + 2] = x[8 * k + j].z;
                        v[4 * j + 3] = x[8 * k + j].w;
                    }
                    tmem_st32(tmem + lane_base + (ch0 + k) * 32, v);
                }
            }
            tmem_wait_st();
            }
        }
        tc_fence_before();
        mbar_arrive(c.bar(B_QFULL));

        float m = -CUDART_INF_F, l = 0.f;
        for (int pg = s.p0; pg < s.p1; ++pg, ++it) {
            const int pb = it % kPBufs;
            const int q2 = (pg - s.p0) % kStepPages;  // position of this page in its step
            const int sb = step % kSBufs;
            const int scs = (int)(step % kScSlots);  // e4m3: this step's slot in the scale ring
            if (q2 == 0 && !warp_wait(c, B_SFULL + sb, (step / kSBufs) & 1)) return;
            if (kRing && q2 == 0 && !warp_wait(c, B_SCFULL + scs, (step / kScSlots) & 1)) return;
            if (kFp8 && (warp & 3) == 0) {
                // one warp checks the scales of the sequence's tokens on this
                // page against the f16 limit, lane i tokens i and i + 32 (a
                // NaN scale fails the test too)
                const uint32_t sc_s = smem_u32(c.base + kScaleOff) + (uint32_t)scs * kScBytes + (uint32_t)q2 * kPage * 4;
                const int nseq = min(kPage, s.T - pg * kPage);
                const float a = lane < nseq ? fabsf(__uint_as_float(lds32(sc_s + 4 * lane))) : 0.f;
                const float b = lane + 32 < nseq ? fabsf(__uint_as_float(lds32(sc_s + 4 * (lane + 32)))) : 0.f;
                if (__any_sync(0xffffffffu, !(a < kE4ScaleLimit) || !(b < kE4ScaleLimit)) && lane == 0)
                    atomicOr(p.status, MLA_DEVERR_SCALE);
            }
            tc_fence_after();
            uint32_t sr[64];
            {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                tmem_ld32(tmem + lane_base + kSCol0 + sb * kSCols + q2 * kPage, lo);
                tmem_ld32(tmem + lane_base + kSCol0 + sb * kSCols + q2 * kPage + 32, hi);
            }
            // keys of this page visible to this row
            int nvalid = row_ok ? T_row - pg * kPage : 0;
            nvalid = nvalid < 0 ? 0 : (nvalid > kPage ? kPage : nvalid);
            // sparse decode: the page's valid list entries (gathered rows)
            uint64_t vmask = ~0ull;
            if constexpr (kSparse) {
                const uint32_t ms = smem_u32(c.base + kScaleOff) + (uint32_t)scs * kScBytes + (uint32_t)q2 * 8;
                vmask = (uint64_t)lds32(ms) | ((uint64_t)lds32(ms + 4) << 32);
                if (nvalid < kPage) vmask &= nvalid > 0 ? (~0ull >> (kPage - nvalid)) : 0ull;
            }
            // e4m3 cache: the page's per-token scales (those of keys past the
            // visible ones, whatever the page holds there, read as 0)
            float cs[kFp8 ? kPage : 1];
            if constexpr (kFp8) {
                const uint32_t sc_s =
                    smem_u32(c.base + kScaleOff) + (uint32_t)scs * kScBytes + (uint32_t)q2 * kPage * 4;
#pragma unroll
                for (int j = 0; j < kPage / 4; ++j) {
                    const uint4 c4 = lds128(sc_s + 16 * j);
                    cs[4 * j] = __uint_as_float(c4.x);
                    cs[4 * j + 1] = __uint_as_float(c4.y);
                    cs[4 * j + 2] = __uint_as_float(c4.z);
                    cs[4 * j + 3] = __uint_as_float(c4.w);
                }
                if (nvalid < kPage) {
#pragma unroll
                    for (int j = 0; j < kPage; ++j) cs[j] = j < nvalid ? cs[j] : 0.f;
                }
            }
            tmem_wait_ld();
            if (q2 == kStepPages - 1 || pg == s.p1 - 1) {  // last page of the step: release its S buffer
                tc_fence_before();
                mbar_arrive(c.bar(B_SEMPTY + sb));
                if constexpr (kRing) mbar_arrive(c.bar(B_SCEMPTY + scs));  // the scales / masks are in registers
                ++step;
            }
            if constexpr (kFp8) {
                // score of key j times its token's scale: the dequantized key
                const uint64_t zero2 = f2_pack(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float xa, xb;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])),
                                     f2_pack(cs[2 * j], cs[2 * j + 1]), zero2),
                              xa, xb);
                    sr[2 * j] = __float_as_uint(xa);
                    sr[2 * j + 1] = __float_as_uint(xb);
                }
            }
            const float sc = p.scale_log2 * qsig;  // e4m3 pages: the row's Q scale folded in
            // page maximum of scale * log2(e) * s over the visible keys, four
            // independent chains to keep the dependency depth short.  A full
            // page with a positive scale takes the maximum of the raw scores
            // (scaling is monotone there) and folds the scale into one FMA per
            // exponent below; otherwise the scaled, masked scores (-inf past
            // the visible keys) replace the raw ones and the FMA scale is 1.
            const bool raw = nvalid == kPage && sc > 0.f && (!kSparse || vmask == ~0ull);
            const float fsc = raw ? sc : 1.f;
            float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
            if (!raw) {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const bool vis = kSparse ? ((vmask >> j) & 1ull) != 0 : j < nvalid;
                    sr[j] = __float_as_uint(vis ? __uint_as_float(sr[j]) * sc : -CUDART_INF_F);
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
                mx4[j & 3] = max3f(mx4[j & 3], __uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1]));
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * fsc;
            float fac = 1.f;
            if (mx > m + kRescaleLog2 || (m == -CUDART_INF_F && mx > -CUDART_INF_F)) {
                fac = ex2(m - mx);  // 0 when m was -inf
                m = mx;
            }
            // exponent inputs and the row sum two lanes per instruction
            uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[32];
            if (m == -CUDART_INF_F) {
#pragma unroll
                for (int j = 0; j < 32; ++j) pk[j] = 0u;
            } else {
                const uint64_t sc2 = f2_pack(fsc, fsc), nm2 = f2_pack(-m, -m);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float xa, xb;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])), sc2, nm2), xa, xb);
                    const float a = ex2(xa), b = ex2(xb);
                    sum2[j & 3] = f2_add(sum2[j & 3], f2_pack(a, b));
                    if constexpr (kFp8) {
                        // P of key j times its token's scale: the dequantized value row
                        float pa, pb2;
                        f2_unpack(f2_fma(f2_pack(a, b), f2_pack(cs[2 * j], cs[2 * j + 1]), f2_pack(0.f, 0.f)), pa,
                                  pb2);
                        pk[j] = pack_f16(pa, pb2);
                    } else {
                        pk[j] = pack_bf16(a, b);
                    }
                }
            }
            float sum_lo, sum_hi;
            f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), sum_lo, sum_hi);
            const float sum = sum_lo + sum_hi;
            l = l * fac + sum;

            // staging pb is free once the value CTA's MMA of page it - 2 is
            // done: that MMA consumed the bulk copy made from it
            if (!warp_wait<true>(c, B_PFREE + pb, ((it / kPBufs) & 1) ^ 1)) return;
            uint8_t *stage = c.base + kStageOff + pb * kPMsgBytes;
            const uint32_t stage_s = smem_u32(stage);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                sts128(stage_s + r * 128 + 16 * (j ^ (r & 7)), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            sts32(stage_s + kFacOff + 4 * r, __float_as_uint(fac));
            if (pg == s.p1 - 1) sts32(stage_s + kInvLOff + 4 * r, __float_as_uint(l > 0.f ? 1.f / l : 0.f));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // this warp's 32 rows of P and of the row factors; the bulk
                // copies' completion on the same barrier makes them visible
                const bool last = pg == s.p1 - 1;
                const uint32_t bar = peer_pfull + pb * 8;
                const uint32_t rows_off = (uint32_t)(32 * (warp & 3)) * 128, fac_off = (uint32_t)(32 * (warp & 3)) * 4;
                const uint32_t dst = peer_buf + pb * kPMsgBytes;
                mbar_arrive_expect_tx_remote_relaxed(bar, 32 * 128 + (last ? 2 : 1) * 32 * 4);
                bulk_copy_to_peer(dst + rows_off, stage + rows_off, 32 * 128, bar);
                bulk_copy_to_peer(dst + kFacOff + fac_off, stage + kFacOff + fac_off, 32 * 4, bar);
                if (last) bulk_copy_to_peer(dst + kInvLOff + fac_off, stage + kInvLOff + fac_off, 32 * 4, bar);
            }
        }
        // LSE of this row over the segment (natural log)
        if (row_ok) {
            const float lse_row = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
            if (s.n_split <= 1) {
                p.lse[(size_t)s.b * p.rows + gr] = lse_row;
            } else {
                const int slot = p.num_splits[s.b] + s.split;
                if (slot >= 0 && slot < p.max_splits) p.lse_accum[(size_t)slot * p.rows + gr] = lse_row;
                else atomicOr(p.status, MLA_DEVERR_SEQLEN);
            }
        }
    }
    // the peer's last commits arrive on our P-free barriers: let them land
    // before this CTA can leave (this also covers the last bulk copies)
    for (uint32_t k = it > (uint32_t)kPBufs ? it - kPBufs : 0; k < it; ++k)
        if (!warp_wait<true>(c, B_PFREE + (int)(k % kPBufs), (k / kPBufs) & 1)) return;
}

// Value-CTA row warps: V tail zeroing (e4m3 cache: widening of each V page),
// lazy O rescale, epilogue.
__device__ void value_rows(const DecodeParams &p, const Ctx &c, uint32_t tmem, int part, int tile) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int tid = threadIdx.x - 64;  // 0..127 among the row warps
    const uint32_t epi_s = smem_u32(c.base + kEpiOff);
    PartWalk walk;
    walk.init(p, part);
    Segment s;
    uint32_t it = 0, oseg = 0;  // oseg: segments with pages so far
    while (walk.next(p, s)) {
        float inv_l = 0.f;
        for (int pg = s.p0; pg < s.p1; ++pg, ++it) {
            const int pb = it % kPBufs, st = it % kVStages;
            if constexpr (kFp8) {
                // widen the page's V codes in place as soon as they land (rows
                // past the sequence's end become zeros); the 128 threads' reads
                // all come before any write through B_VREAD, a bounded barrier
                if (!warp_wait(c, B_VLAND + st, (it / kVStages) & 1)) return;
                const uint32_t stage = smem_u32(c.base + kVRingOff + st * kVStageBytes);
                const bool ok = widen_e4m3<16, 128>(stage, stage + kVLandOff, tid, min(s.T - pg * kPage, kPage), [&] {
                    mbar_arrive(c.bar(B_VREAD));
                    return warp_wait(c, B_VREAD, it & 1);
                });
                if (!ok) return;
                fence_proxy_async_smem();
                mbar_arrive(c.bar(B_VFULL + st));
            }
            if (!warp_wait<true>(c, B_PFULL + pb, (it / kPBufs) & 1)) return;
            const uint32_t buf_s = smem_u32(c.base + kPBufOff + pb * kPMsgBytes);
            const float fac = __uint_as_float(lds32(buf_s + kFacOff + 4 * r));
            if (pg == s.p1 - 1) inv_l = __uint_as_float(lds32(buf_s + kInvLOff + 4 * r));
            // rows past the sequence's end in its last page: zero them in V so
            // that garbage (even NaN) times a zero weight stays zero
            const int tail = s.T - pg * kPage;
            if (!kFp8 && tail < kPage) {
                if constexpr (kSparse) {
                    for (int ch = 0; ch < kVChunks; ++ch)
                        if (!warp_wait(c, B_CHUNK + st * kKChunks + ch, (it / kVStages) & 1)) return;
                } else if (!warp_wait(c, B_VFULL + st, (it / kVStages) & 1)) {
                    return;
                }
                // thread t zeroes 16-byte piece t % 8 of rows tail + t / 8,
                // + 16, ... in every chunk (whole 128-byte rows, so the swizzle
                // does not matter)
                const uint32_t vt = smem_u32(c.base + kVRingOff + st * kVStageBytes) + 16u * (uint32_t)(tid & 7);
                for (int rr = (tail > 0 ? tail : 0) + (tid >> 3); rr < kPage; rr += 16)
#pragma unroll
                    for (int ch = 0; ch < kVChunks; ++ch) sts128(vt + ch * kChunkBytes + rr * 128, 0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
            }
            // lazy rescale of this row of O before the next accumulation
            const bool need = (pg > s.p0) && (fac != 1.f);
            if (__any_sync(0xffffffffu, need)) {
                if (!warp_wait(c, B_PVDONE, (it - 1) & 1)) return;  // every earlier P V has landed
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < 16; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + ch * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * fac);
                    tmem_st32(tmem + lane_base + ch * 32, v);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(c.bar(B_PREADY + pb));
        }
        // epilogue: O / l -> bf16 output, or fp32 partial for the combine.
        // Each 64-column chunk goes TMEM -> registers -> smem (row per
        // thread), then the warp writes its 32 whole rows with coalesced stores.
        const bool has_pages = s.p1 > s.p0;
        if (has_pages) {
            // every P V of the segment has landed.  (The per-page barrier
            // cannot serve here: the row warps only know that the MMA of page
            // it - 3 is done, and a parity wait cannot tell phase it - 1 from
            // phase it - 3.)
            if (!warp_wait(c, B_ODONE, oseg & 1)) return;
            ++oseg;
            tc_fence_after();
        }
        const bool split = s.n_split > 1;
        int slot = 0;
        if (split) {
            slot = p.num_splits[s.b] + s.split;
            if (slot < 0 || slot >= p.max_splits) {
                if (tid == 0) atomicOr(p.status, MLA_DEVERR_SEQLEN);
                slot = -1;
            }
        }
        // each warp stores the 32 rows of its own TMEM lane quarter, through
        // its own slice of the staging tile: no cross-warp barrier is needed
        const int wrow0 = 32 * (warp & 3);
#pragma unroll 1
        for (int ch = 0; ch < kDv / (int)kEpiCols; ++ch) {
            uint32_t v[64];
            if (has_pages) {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                tmem_ld32(tmem + lane_base + ch * kEpiCols, lo);
                tmem_ld32(tmem + lane_base + ch * kEpiCols + 32, hi);
                tmem_wait_ld();
                if (ch == kDv / (int)kEpiCols - 1) {  // the last TMEM read: O may be overwritten now
                    tc_fence_before();
                    mbar_arrive(c.bar(B_OEMPTY));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) v[j] = 0u;
            }
            const uint32_t srow = epi_s + r * kEpiStride;
            if (split) {  // fp32 partial: 256 B of the row
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    sts128(srow + 16 * j, __float_as_uint(__uint_as_float(v[4 * j]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * j + 1]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * j + 2]) * inv_l),
                           __float_as_uint(__uint_as_float(v[4 * j + 3]) * inv_l));
            } else {  // bf16 output: 128 B of the row
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    sts128(srow + 16 * j,
                           pack_bf16(__uint_as_float(v[8 * j]) * inv_l, __uint_as_float(v[8 * j + 1]) * inv_l),
                           pack_bf16(__uint_as_float(v[8 * j + 2]) * inv_l, __uint_as_float(v[8 * j + 3]) * inv_l),
                           pack_bf16(__uint_as_float(v[8 * j + 4]) * inv_l, __uint_as_float(v[8 * j + 5]) * inv_l),
                           pack_bf16(__uint_as_float(v[8 * j + 6]) * inv_l, __uint_as_float(v[8 * j + 7]) * inv_l));
            }
            __syncwarp();
            if (slot >= 0) {
                // all of the warp's shared loads first, then its global stores
                uint4 x[16];
                if (split) {
                    // fp32: 256 B per row chunk, two rows per warp store
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        x[k] = lds128(epi_s + (wrow0 + 2 * k + (lane >> 4)) * kEpiStride + 16 * (lane & 15));
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int g = tile * kTileRows + wrow0 + 2 * k + (lane >> 4);
                        if (g < p.rows)
                            reinterpret_cast<uint4 *>(p.o_accum + ((size_t)slot * p.rows + g) * kDv + ch * kEpiCols)[lane & 15] = x[k];
                    }
                } else {
                    // bf16: 128 B per row chunk, four rows per warp store
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        x[k] = lds128(epi_s + (wrow0 + 4 * k + (lane >> 3)) * kEpiStride + 16 * (lane & 7));
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int g = tile * kTileRows + wrow0 + 4 * k + (lane >> 3);
                        if (g < p.rows)
                            reinterpret_cast<uint4 *>(p.o + ((size_t)s.b * p.rows + g) * kDv + ch * kEpiCols)[lane & 7] = x[k];
                    }
                }
            }
            __syncwarp();  // the slice is rewritten by the next chunk
        }
    }
}




// -------------------------------------------------------------- kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
split_kv_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap kv_map2,
                   const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t rank = cluster_ctarank();
    const bool is_score = rank == 0;
    const int part = blockIdx.x >> 1;
    const int tile = blockIdx.y;
    const int warp = threadIdx.x >> 5;

    Ctx c;
    c.base = base;
    c.bars = reinterpret_cast<uint64_t *>(base + kBarOff);
    c.abort_flag = reinterpret_cast<volatile int *>(base + kAbortOff);
    c.status = p.status;
    c.peer = rank ^ 1u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kTmemSlotOff);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKSlots; ++i) {
            mbar_init(c.bar(B_KFULL + i), 1);
            mbar_init(c.bar(B_KEMPTY + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(c.bar(B_VFULL + i), kFp8 ? 128 : 1);  // e4m3: the 128 row threads that widened the page
            mbar_init(c.bar(B_VEMPTY + i), 1);
        }
        if constexpr (kSparse) {
            for (int i = 0; i < kScSlots; ++i) {
                mbar_init(c.bar(B_SCFULL + i), 1);
                mbar_init(c.bar(B_SCEMPTY + i), 128);
            }
            for (int i = 0; i < kVStages * kKChunks; ++i) mbar_init(c.bar(B_CHUNK + i), 1);
        }
        if constexpr (kFp8) {
            for (int i = 0; i < kVStages; ++i) mbar_init(c.bar(B_VLAND + i), 1);
            for (int i = 0; i < kScSlots; ++i) {
                mbar_init(c.bar(B_SCFULL + i), 1);
                mbar_init(c.bar(B_SCEMPTY + i), 128);
            }
            mbar_init(c.bar(B_VREAD), 128);
        }
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(c.bar(B_SFULL + i), 1);
            mbar_init(c.bar(B_SEMPTY + i), 128);
        }
        mbar_init(c.bar(B_QFULL), 128);
        mbar_init(c.bar(B_QACK), kScoreIssuers);  // every score-MMA issuer has seen a segment's Q
        for (int i = 0; i < kPBufs; ++i) {
            mbar_init(c.bar(B_PFREE + i), 1);
            mbar_init(c.bar(B_PFULL + i), 4);  // one arrival per row warp of the score CTA
            mbar_init(c.bar(B_PREADY + i), 128);
        }
        mbar_init(c.bar(B_PVDONE), 1);
        mbar_init(c.bar(B_ODONE), 1);
        mbar_init(c.bar(B_OEMPTY), 128);
        mbar_init(c.bar(B_FINAL), is_score ? kScoreIssuers : 1);  // one commit per MMA issuer
        *c.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&kv_map);
        if constexpr (kFp8) tma_prefetch_desc(&kv_map2);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_arrive();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Everything above touches only this CTA's shared memory, TMEM and the
    // kernel parameters, so it overlaps the previous kernel's tail when the
    // launch is programmatic; no global memory is read or written before this.
    // (This kernel never triggers its own dependents early: doing so, at the
    // start or after the last page, measured 1-4 % slower on GB300; the
    // combine launch then follows this grid's completion.)
    griddep_wait();

    if (warp == 0 || warp == 7) {
        if (kFp8 && is_score) {
            if (elect_one_lane()) score_producer_e4m3(p, c, &kv_map, part, warp == 0 ? 0 : 1);
        } else if (kSparse && is_score) {
            if (warp == 0) score_producer_sparse(p, c, &kv_map, part, tile);
        } else if (kSparse) {
            if (warp == 0) value_producer_sparse(p, c, &kv_map, part, tile);
        } else if (elect_one_lane() && (warp == 0 || (is_score && kScoreIssuers > 1))) {
            if (is_score) score_producer(p, c, &kv_map, part, tile, warp == 0 ? 0 : 1);
            else value_producer(p, c, kFp8 ? &kv_map2 : &kv_map, part);
        }
    } else if (warp == 1 || warp == 6) {
        if (elect_one_lane() && (warp == 1 || (is_score && kScoreIssuers > 1))) {
            if (is_score) score_mma(p, c, tmem, part, warp == 1 ? 0 : 1);
            else value_mma(p, c, tmem, part);
            // all MMAs this thread issued must finish before TMEM is released
            mma_commit(c.bar(B_FINAL));
            mbar_wait(c.bar(B_FINAL), 0, c.status);
        }
        __syncwarp();
    } else {
        if (is_score) score_rows(p, c, tmem, part, tile);
        else value_rows(p, c, tmem, part, tile);
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA may leave while its peer can still touch its shared memory
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// -------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// kcache [num_blocks][64][D] bf16 viewed as a 3-D tensor {D, 64, num_blocks};
// one box is a 64-dim x 64-token chunk, stored with the 128-byte swizzle that
// the tcgen05 K-major (K) and MN-major (V) operand descriptors expect.
// e4m3 pages: the codes of a page viewed as {D bytes, 64, num_blocks} with the
// page stride; a box (64 codes x 64 tokens) lands unswizzled, 64 B per token.
// The tensor maps of the cache.  bf16 rows: `m` only.  e4m3 pages: `m` lands
// each 64-code box with the 64-byte swizzle of the fp8 MMA operands (score
// CTA), `m2` unswizzled, 64 B per token, for the value CTA's widening.
bool make_kv_map(CUtensorMap *m, CUtensorMap *m2, const void *kcache, int64_t num_blocks) {
    auto enc = encode_fn();
    if (!enc) return false;
    if constexpr (kSparse) {
        // gathers: the cache as a 2-D tensor of num_blocks * 64 rows of D
        // elements, one 64-element row per box (tile::gather4 takes 4 rows)
        cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)num_blocks * kPage};
        cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
        cuuint32_t box[2] = {64, 1};
        cuuint32_t es[2] = {1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(kcache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if constexpr (kFp8) {
        cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kPage, (cuuint64_t)num_blocks};
        cuuint64_t strides[2] = {(cuuint64_t)kD, (cuuint64_t)kE4PageBytes};
        cuuint32_t box[3] = {64, (cuuint32_t)kPage, 1};
        cuuint32_t es[3] = {1, 1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(kcache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
               enc(m2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(kcache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    *m2 = *m;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kPage, (cuuint64_t)num_blocks};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kPage * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kPage, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(kcache), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
bool g_attr_set[kMaxDevices] = {};
std::mutex g_attr_mutex;

cudaError_t prepare(int dev) {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (g_attr_set[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(split_kv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess) g_attr_set[dev] = true;
    return e;
}

}  // namespace

#if !MLA_SPLIT_SPARSE
template <>
cudaError_t split_kv_tc_max_pairs<kD, kFp8>(int *pairs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare(dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    cfg.numAttrs = 0;  // the cluster shape is fixed by the kernel's attribute
    e = cudaOccupancyMaxActiveClusters(&n, split_kv_tc_kernel, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, split_kv_tc_kernel, &cfg);
    }
    if (e != cudaSuccess) return e;
    *pairs = n;
    return cudaSuccess;
}

#endif

#if MLA_SPLIT_SPARSE && MLA_SPARSE_MULTICAST
cudaError_t launch_split_kv_tc_sparse(const DecodeParams &p, cudaStream_t stream) {
#elif MLA_SPLIT_SPARSE
cudaError_t launch_split_kv_tc_sparse_local(const DecodeParams &p, cudaStream_t stream) {
#else
template <>
cudaError_t launch_split_kv_tc<kD, kFp8>(const DecodeParams &p, cudaStream_t stream) {
#endif
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare(dev)) != cudaSuccess) return e;
    CUtensorMap map;
    CUtensorMap map2;
    if (!make_kv_map(&map, &map2, p.kcache, p.num_blocks)) return cudaErrorInvalidValue;
    const int tiles = (p.rows + kTileRows - 1) / kTileRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * p.num_parts, tiles, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // prologue overlaps the previous kernel
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_tc_kernel, map, map2, p);
}

}  // namespace mla
