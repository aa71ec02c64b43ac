// Split-KV kernel for the 576-wide latent cache stored as packed e4m3 pages
// with per-token fp32 scales.
#define MLA_SPLIT_D 576
#define MLA_SPLIT_FP8 1
#include "mla_split_tc_impl.cuh"
