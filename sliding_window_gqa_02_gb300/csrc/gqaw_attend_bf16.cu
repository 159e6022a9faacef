// gqaw_attend_bf16.cu -- instantiations and launch of the persistent attention kernel
// for bfloat16 caches (head sizes 8..256, query-head blocks of 1, 2, 4 or 8).
#include "gqaw_attend_launch.cuh"

namespace gqaw {

cudaError_t launch_attend_bf16(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  return attend_launch::by_size<__nv_bfloat16>(p, gb, max_ctas, stream);
}

int attend_tile_bf16(int D) { return attend_launch::tile<__nv_bfloat16>(D); }

}  // namespace gqaw
