// gqaw_mmad.cu -- the small-step tensor-core kernel (gqaw_mmad.cuh) for bf16 caches,
// and the dispatch to the quantized-cache instantiations.
#include "gqaw_mmad.cuh"

namespace gqaw {

cudaError_t launch_mmad_q8(const Params &p, const TdArgs &ta, const TdMaps &maps, int max_ctas, cudaStream_t stream);

cudaError_t launch_mmad(const Params &p, const TdArgs &ta, const TdMaps &maps, int max_ctas, cudaStream_t stream) {
  if (p.quant) return launch_mmad_q8(p, ta, maps, max_ctas, stream);
  return launch_mmad_t<0>(p, ta, maps, max_ctas, stream);
}

}  // namespace gqaw
