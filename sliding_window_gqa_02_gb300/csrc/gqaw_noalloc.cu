// gqaw_noalloc.cu -- a step entry point for callers that cannot allocate device memory.
//
// gqa_windowed_step() asks the caller for a workspace: the split-K attention kernel
// writes its per-chunk partial results there and the finish kernel merges them.  Some
// hosts cannot provide one: a plugin inside an inference runtime that owns all device
// memory and hands the plugin no allocator, or a serving loop that forbids any
// allocation once it has started.  gqa_windowed_step_noalloc() runs the same kernels
// with that scratch taken from a fixed array compiled into this library instead.
//
// The array below is a file-scope __device__ variable: every GPU on which the library is
// loaded holds its GQAW_NOALLOC_SCRATCH_BYTES until the process exits.  In host code the
// name g_scratch is only a host-side stand-in, never a device address; the device
// address is looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached.
//
// Every call shares the array and finds there what the previous call left.  Where a
// step keeps its counters and tickets depends on its shape, and a step that stopped on
// a device error may leave them non-zero; so each call first clears the part of the
// array that a step needs at zero (status word, counters, list, tickets: a few KB, one
// cudaMemsetAsync on the call's stream).  The partial results that follow are always
// written before they are read.
#include <cstdio>
#include <mutex>

#include "gqaw_internal.cuh"

namespace gqaw {
void set_error(const char *msg);
size_t workspace_counter_bytes(const gqaw_step_args *args);
void workspace_zeroed(const void *ws, size_t bytes);
}

namespace {

static __device__ __align__(256) unsigned char g_scratch[GQAW_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_dev[kMaxDevices] = {nullptr};

// Device address of g_scratch on the current device; the first call for a device
// looks it up (with that device current) and zeroes the whole array on `stream`.
gqaw_status scratch_for_current_device(void **out, cudaStream_t stream) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    gqaw::set_error(cudaGetErrorString(e));
    return GQAW_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    gqaw::set_error("gqa_windowed_step_noalloc: device ordinal out of range");
    return GQAW_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_dev[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      gqaw::set_error(e != cudaSuccess ? cudaGetErrorString(e) : "cudaGetSymbolAddress returned NULL");
      return GQAW_ECUDA;
    }
    e = cudaMemsetAsync(p, 0, GQAW_NOALLOC_SCRATCH_BYTES, stream);
    if (e != cudaSuccess) {
      gqaw::set_error(cudaGetErrorString(e));
      return GQAW_ECUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return GQAW_OK;
}

}  // namespace

extern "C" gqaw_status gqa_windowed_step_noalloc(const gqaw_step_args *args, void *stream) {
  if (!args) {
    gqaw::set_error("args is NULL");
    return GQAW_EINVAL;
  }
  const size_t need = gqaw_workspace_bytes(args);  // also validates the sizes
  if (need == 0) return GQAW_EINVAL;                // message already set
  if (need > (size_t)GQAW_NOALLOC_SCRATCH_BYTES) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "gqa_windowed_step_noalloc: this step needs %zu bytes of scratch but the static scratch holds %zu; "
             "use gqa_windowed_step with a caller workspace",
             need, (size_t)GQAW_NOALLOC_SCRATCH_BYTES);
    gqaw::set_error(buf);
    return GQAW_EWORKSPACE;
  }
  if (args->batch_size == 0) return GQAW_OK;
  void *scratch = nullptr;
  const gqaw_status s = scratch_for_current_device(&scratch, static_cast<cudaStream_t>(stream));
  if (s != GQAW_OK) return s;
  // status word, counters, list and tickets of this step's layout start at zero
  const size_t counters = gqaw::workspace_counter_bytes(args);
  const cudaError_t e = cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    gqaw::set_error(cudaGetErrorString(e));
    return GQAW_ECUDA;
  }
  gqaw::workspace_zeroed(scratch, counters);
  gqaw_step_args a = *args;  // the caller's workspace fields are ignored
  a.workspace = scratch;
  a.workspace_bytes = GQAW_NOALLOC_SCRATCH_BYTES;
  return gqa_windowed_step(&a, stream);
}
