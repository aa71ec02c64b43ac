// Split-KV kernel for the 576-wide latent cache (512 latent + 64 RoPE dims).
#define MLA_SPLIT_D 576
#include "mla_split_tc_impl.cuh"

namespace mla {
int split_kv_tc_tile_rows() { return kTileRows; }  // the same for every row width
}  // namespace mla
