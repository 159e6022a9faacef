// gqaw_attend_launch.cuh -- launch of the persistent attention kernel (attend_kernel of
// gqaw_attend.cuh), shared by the translation units that instantiate it: one per cache
// type (float, bfloat16, 1-byte codes), so that the instantiations compile in parallel.
#pragma once

#include <atomic>

#include "gqaw_attend.cuh"

namespace gqaw {
namespace attend_launch {

constexpr int kMaxDevices = 64;

// One instantiation: T is the query/output type, TC the cache element type, D the head
// size, GB the query heads per CTA.
template <typename T, typename TC, int D, int GB>
cudaError_t one(const Params &p, int max_ctas, cudaStream_t stream) {
  using Cfg = AttendCfg<TC, D, GB>;
  auto kernel = attend_kernel<T, TC, D, GB>;
  // Per device, once: the dynamic shared-memory limit and carveout (function
  // attributes), and how many CTAs of this kernel are resident at once.
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

// The query-head block (1, 2, 4 or 8 heads per CTA) of one head size.
template <typename T, typename TC, int D>
cudaError_t by_block(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (gb) {
    case 1: return one<T, TC, D, 1>(p, max_ctas, stream);
    case 2: return one<T, TC, D, 2>(p, max_ctas, stream);
    case 4: return one<T, TC, D, 4>(p, max_ctas, stream);
    case 8: return one<T, TC, D, 8>(p, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

// Every head size of a cache type whose caches hold the query's own type (8..256).
template <typename T>
cudaError_t by_size(const Params &p, int gb, int max_ctas, cudaStream_t stream) {
  switch (p.D) {
    case 8: return by_block<T, T, 8>(p, gb, max_ctas, stream);
    case 16: return by_block<T, T, 16>(p, gb, max_ctas, stream);
    case 32: return by_block<T, T, 32>(p, gb, max_ctas, stream);
    case 64: return by_block<T, T, 64>(p, gb, max_ctas, stream);
    case 128: return by_block<T, T, 128>(p, gb, max_ctas, stream);
    case 256: return by_block<T, T, 256>(p, gb, max_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

// Key rows per staged tile of a cache type (independent of the head block).
template <typename TC>
int tile(int D) {
  switch (D) {
    case 8: return AttendCfg<TC, 8, 1>::kTile;
    case 16: return AttendCfg<TC, 16, 1>::kTile;
    case 32: return AttendCfg<TC, 32, 1>::kTile;
    case 64: return AttendCfg<TC, 64, 1>::kTile;
    case 128: return AttendCfg<TC, 128, 1>::kTile;
    case 256: return AttendCfg<TC, 256, 1>::kTile;
  }
  return 0;
}

}  // namespace attend_launch
}  // namespace gqaw
