// gqaw_attend_q8.cu -- instantiations and launch of the persistent attention kernel
// for quantized caches: 1-byte int8 or fp8 e4m3 codes with per-tensor scales (mobius
// issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1, inputs k_scale and
// v_scale), bfloat16 queries and outputs, head sizes 64, 128 and 256.
#include <atomic>

#include "gqaw_attend.cuh"

namespace gqaw {
namespace {

constexpr int kMaxDevices = 64;

template <typename TC, int D, int GB>
cudaError_t launch_one(const Params &p, int max_ctas, cudaStream_t stream) {
  using Cfg = AttendCfg<TC, D, GB>;
  auto kernel = attend_kernel<__nv_bfloat16, TC, D, GB>;
  // Per device, once: the dynamic shared-memory limit and carveout, and how many CTAs
  // of this kernel are resident at once.
  static std::atomic<int> resident[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int slots = dev < kMaxDevices ? resident[dev].load(std::memory_order_relaxed) : 0;
  if (slots <= 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, Cfg::kThreads, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    slots = per_sm * sms > 0 ? per_sm * sms : 1;
    if (dev < kMaxDevices) resident[dev].store(slots, std::memory_order_relaxed);
  }
  // A persistent grid: never more CTAs than can be resident together.
  const int grid = max_ctas < slots ? max_ctas : slots;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename TC, int D>
cudaError_t by_block(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (gb) {
    case 1: return launch_one<TC, D, 1>(p, max_ctas, stream);
    case 2: return launch_one<TC, D, 2>(p, max_ctas, stream);
    case 4: return launch_one<TC, D, 4>(p, max_ctas, stream);
    case 8: return launch_one<TC, D, 8>(p, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TC>
cudaError_t by_size(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (p.D) {
    case 64: return by_block<TC, 64>(p, gb, max_ctas, stream);
    case 128: return by_block<TC, 128>(p, gb, max_ctas, stream);
    case 256: return by_block<TC, 256>(p, gb, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attend_q8(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  if (p.quant == GQAW_I8) return by_size<CodeI8>(p, gb, max_ctas, stream);
  if (p.quant == GQAW_E4M3) return by_size<CodeE4M3>(p, gb, max_ctas, stream);
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
