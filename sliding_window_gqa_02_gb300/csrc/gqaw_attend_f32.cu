// gqaw_attend_f32.cu -- instantiations and launch of the persistent attention kernel
// for float caches (head sizes 8..256, query-head blocks of 1, 2, 4 or 8).
#include "gqaw_attend_launch.cuh"

namespace gqaw {

cudaError_t launch_attend_f32(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  return attend_launch::by_size<float>(p, gb, max_ctas, stream);
}

int attend_tile_f32(int D) { return attend_launch::tile<float>(D); }

}  // namespace gqaw
