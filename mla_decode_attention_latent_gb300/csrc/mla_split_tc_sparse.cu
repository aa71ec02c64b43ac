// Split-KV kernel for the sparse top-k decode: 576-wide bf16 cache rows
// gathered row by row from per-query-token index lists.
#define MLA_SPLIT_D 576
#define MLA_SPLIT_SPARSE 1
#include "mla_split_tc_impl.cuh"
