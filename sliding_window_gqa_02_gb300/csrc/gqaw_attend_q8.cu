// gqaw_attend_q8.cu -- instantiations and launch of the persistent attention kernel
// for quantized caches: 1-byte int8 or fp8 e4m3 codes with per-tensor scales (mobius
// issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1, inputs k_scale and
// v_scale), bfloat16 queries and outputs, head sizes 64, 128 and 256.
#include "gqaw_attend_launch.cuh"

namespace gqaw {
namespace {

template <typename TC>
cudaError_t by_code_size(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (p.D) {
    case 64: return attend_launch::by_block<__nv_bfloat16, TC, 64>(p, gb, max_ctas, stream);
    case 128: return attend_launch::by_block<__nv_bfloat16, TC, 128>(p, gb, max_ctas, stream);
    case 256: return attend_launch::by_block<__nv_bfloat16, TC, 256>(p, gb, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attend_q8(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  if (p.quant == GQAW_I8) return by_code_size<CodeI8>(p, gb, max_ctas, stream);
  if (p.quant == GQAW_E4M3) return by_code_size<CodeE4M3>(p, gb, max_ctas, stream);
  return cudaErrorInvalidValue;
}

// Key rows per staged tile (the same for both code types; independent of the head block).
int attend_tile_q8(int D) {
  switch (D) {
    case 64: return AttendCfg<CodeI8, 64, 1>::kTile;
    case 128: return AttendCfg<CodeI8, 128, 1>::kTile;
    case 256: return AttendCfg<CodeI8, 256, 1>::kTile;
  }
  return 0;
}

}  // namespace gqaw
