// Split-KV kernel for the sparse top-k decode in which each CTA of a pair
// gathers every row chunk it uses itself (no cluster multicast).
#define MLA_SPLIT_D 576
#define MLA_SPLIT_SPARSE 1
#define MLA_SPARSE_MULTICAST 0
#include "mla_split_tc_impl.cuh"
