// gqaw_attend_f32.cu -- instantiations and launch of the persistent attention kernel
// for float caches (head sizes 8..256, query-head blocks of 1, 2, 4 or 8).
#include <atomic>

#include "gqaw_attend.cuh"

namespace gqaw {
namespace {

constexpr int kMaxDevices = 64;

template <int D, int GB>
cudaError_t launch_one(const Params &p, int max_ctas, cudaStream_t stream) {
  using Cfg = AttendCfg<float, D, GB>;
  // Per device, once: the dynamic shared-memory limit and carveout (function
  // attributes), and how many CTAs of this kernel are resident at once.
  static std::atomic<int> resident[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int slots = dev < kMaxDevices ? resident[dev].load(std::memory_order_relaxed) : 0;
  if (slots <= 0) {
    e = cudaFuncSetAttribute(attend_kernel<float, float, D, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attend_kernel<float, float, D, GB>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<float, float, D, GB>, Cfg::kThreads, Cfg::kSmem);
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
  e = cudaLaunchKernelEx(&cfg, attend_kernel<float, float, D, GB>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t by_block(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (gb) {
    case 1: return launch_one<D, 1>(p, max_ctas, stream);
    case 2: return launch_one<D, 2>(p, max_ctas, stream);
    case 4: return launch_one<D, 4>(p, max_ctas, stream);
    case 8: return launch_one<D, 8>(p, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attend_f32(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (p.D) {
    case 8: return by_block<8>(p, gb, max_ctas, stream);
    case 16: return by_block<16>(p, gb, max_ctas, stream);
    case 32: return by_block<32>(p, gb, max_ctas, stream);
    case 64: return by_block<64>(p, gb, max_ctas, stream);
    case 128: return by_block<128>(p, gb, max_ctas, stream);
    case 256: return by_block<256>(p, gb, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

// Key rows per staged tile (independent of the head block).
int attend_tile_f32(int D) {
  switch (D) {
    case 8: return AttendCfg<float, 8, 1>::kTile;
    case 16: return AttendCfg<float, 16, 1>::kTile;
    case 32: return AttendCfg<float, 32, 1>::kTile;
    case 64: return AttendCfg<float, 64, 1>::kTile;
    case 128: return AttendCfg<float, 128, 1>::kTile;
    case 256: return AttendCfg<float, 256, 1>::kTile;
  }
  return 0;
}

}  // namespace gqaw
