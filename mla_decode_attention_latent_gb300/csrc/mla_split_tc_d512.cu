// Split-KV kernel for a 512-wide cached row (the d_qk = 512 variant: the row is
// both key and value, no separate RoPE part).
#define MLA_SPLIT_D 512
#include "mla_split_tc_impl.cuh"
