// gqaw_mmad_q8.cu -- the small-step tensor-core kernel (gqaw_mmad.cuh) for quantized
// caches: int8 and fp8 e4m3 code tiles widened to fp16 operands in shared memory.
#include "gqaw_mmad.cuh"

namespace gqaw {

cudaError_t launch_mmad_q8(const Params &p, const TdArgs &ta, const TdMaps &maps, int max_ctas, cudaStream_t stream) {
  if (p.quant == GQAW_I8) return launch_mmad_t<GQAW_I8>(p, ta, maps, max_ctas, stream);
  if (p.quant == GQAW_E4M3) return launch_mmad_t<GQAW_E4M3>(p, ta, maps, max_ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gqaw
