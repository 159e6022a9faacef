// gqaw_attend_f32.cu -- instantiations and launch dispatch of the split-K attention
// kernel for float caches (head sizes 8..256, query-head blocks of 1, 2, 4 or 8).
#include <atomic>

#include "gqaw_attend.cuh"

namespace gqaw {
namespace {

template <int D, int GB>
cudaError_t launch_one(const Params &p, int blocks, cudaStream_t stream) {
  using Cfg = AttendCfg<float, D, GB>;
  // The dynamic shared-memory limit is a per-device function attribute: set it once
  // per device (bit d of the mask).
  static std::atomic<unsigned long long> done{0ull};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(done.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(attend_kernel<float, D, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  attend_kernel<float, D, GB><<<blocks, Cfg::kThreads, Cfg::kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t by_block(const Params &p, int gb, int blocks, cudaStream_t stream) {
  switch (gb) {
    case 1: return launch_one<D, 1>(p, blocks, stream);
    case 2: return launch_one<D, 2>(p, blocks, stream);
    case 4: return launch_one<D, 4>(p, blocks, stream);
    case 8: return launch_one<D, 8>(p, blocks, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attend_f32(const Params &p, int gb, int blocks, cudaStream_t stream) {
  switch (p.D) {
    case 8: return by_block<8>(p, gb, blocks, stream);
    case 16: return by_block<16>(p, gb, blocks, stream);
    case 32: return by_block<32>(p, gb, blocks, stream);
    case 64: return by_block<64>(p, gb, blocks, stream);
    case 128: return by_block<128>(p, gb, blocks, stream);
    case 256: return by_block<256>(p, gb, blocks, stream);
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
