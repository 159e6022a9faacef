// gqaw_quant.cu -- the step's new key and value rows as a quantized cache holds them.
//
// mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1: k_scale and
// v_scale are the scales of a quantized KV cache.  A code is x / scale computed in float
// (one IEEE division), rounded to nearest even and saturated: int8 to [-128, 127], fp8
// e4m3 to the largest finite value 448 (NaN stays NaN).  The codes go to the workspace;
// the attention kernel reads the new keys and values from there (as the cache will hold
// them) and the appends copy them into the cache.  Element-wise, HBM bound: one thread per
// eight elements (a 16-byte vector of bfloat16 in, eight bytes out).
#include "gqaw_internal.cuh"

namespace gqaw {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t code_i8(float q) {
  int c = __float2int_rn(q);  // ties to even; NaN gives 0; out of range saturates
  c = c < -128 ? -128 : (c > 127 ? 127 : c);
  return (uint32_t)(c & 0xff);
}

// Two e4m3 codes of a and b, packed as (a in bits 0-7, b in bits 8-15).
__device__ __forceinline__ uint32_t codes_e4m3(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

template <int QT>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const Params p) {
  pdl_wait();  // the rows to quantize (maybe turned by the rotary kernel) are written
  const long long n8 = (long long)p.B * p.S * p.Nkv * p.D / 8;  // 8-element groups per tensor
  const long long nq8 = p.q16 ? (long long)p.B * p.S * p.Nq * p.D / 8 : 0;
  const float sk = *p.ks, sv = *p.vs;
  // the fp16 copy of the query (the tensor-core kernel's operand), when asked for.  A
  // finite bfloat16 element at or beyond 65520 in magnitude has no finite fp16 value:
  // flagged (GQAW_DEV_QUERY_RANGE), the item's output is then unspecified.
  bool out_of_range = false;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < nq8;
       idx += (long long)gridDim.x * blockDim.x) {
    float f[8];
    Elem<__nv_bfloat16>::unpack(static_cast<const uint4 *>(p.q)[idx], f);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      const float2 back = __half22float2(h);
      out_of_range |= (isinf(back.x) && !isinf(f[2 * i])) || (isinf(back.y) && !isinf(f[2 * i + 1]));
      w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    static_cast<uint4 *>(p.q16)[idx] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (out_of_range) flag(p, GQAW_DEV_QUERY_RANGE);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < 2 * n8;
       idx += (long long)gridDim.x * blockDim.x) {
    const bool val = idx >= n8;
    const long long e = val ? idx - n8 : idx;
    const uint4 u = static_cast<const uint4 *>(val ? p.vq_in : p.kq_in)[e];
    float f[8];
    Elem<__nv_bfloat16>::unpack(u, f);
    const float s = val ? sv : sk;
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __fdiv_rn(f[4 * h + i], s);
      if (QT == GQAW_I8)
        w[h] = code_i8(q[0]) | (code_i8(q[1]) << 8) | (code_i8(q[2]) << 16) | (code_i8(q[3]) << 24);
      else
        w[h] = codes_e4m3(q[0], q[1]) | (codes_e4m3(q[2], q[3]) << 16);
    }
    static_cast<uint2 *>(const_cast<void *>(val ? p.v : p.k))[e] = make_uint2(w[0], w[1]);
  }
  pdl_launch_dependents();  // done: the attention kernel may be scheduled
}

cudaError_t launch_quantize(const Params &p, int max_blocks, cudaStream_t stream) {
  const long long n = 2LL * p.B * p.S * p.Nkv * p.D / 8 + (p.q16 ? (long long)p.B * p.S * p.Nq * p.D / 8 : 0);
  long long blocks = (n + kQuantThreads - 1) / kQuantThreads;
  if (blocks > max_blocks) blocks = max_blocks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks > 0 ? blocks : 1));
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = p.quant == GQAW_I8 ? cudaLaunchKernelEx(&cfg, quantize_kernel<GQAW_I8>, p)
                                           : cudaLaunchKernelEx(&cfg, quantize_kernel<GQAW_E4M3>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqaw
