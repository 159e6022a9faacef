// gqaw_rotary.cu -- first kernel of a step with the rotary embedding turned on.
//
// mobius issue #111 "GQA In-Place KV Cache: Investigation Report", Part 1.1 (inputs
// cos_cache, sin_cache, position_ids) and Part 1.3 (attributes do_rotary,
// rotary_interleaved): the new query and key rows are turned before attention reads
// them and before the keys enter the cache.  Each pair of dimensions (x1, x2) of a row
// turns by the angle of the token's position (the rotary position embedding of
// RoFormer): y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin, with cos and sin taken from
// row `pos` of the caches at the pair's index.  Pairs are (i, i + rd/2), or (2i, 2i+1)
// when interleaved; dimensions from rd on are copied.  pos = position_ids[b, s] when
// given, else the token's absolute position P_b + s = seqlens_k[b] + 1 - S + s.
//
// The turned rows go to the workspace in the input layouts, rounded once to the
// step's dtype; the attention kernels and the cache update read them there.  The
// work is HBM bound (each new row is read once and written once, plus a cos/sin row
// that L2 serves to all heads of a token), so the kernel is element-wise with 16-byte
// accesses: a work item is one 16-byte vector of a row (interleaved pairs, and the
// dimensions past rd), or, with split pairs, the two vectors at c and c + rd/2 whose
// elements pair up.  A grid of resident blocks strides over all items.  Shapes whose
// rotary width or cache rows do not split into 16-byte vectors take the scalar
// kernel, one thread per pair.
#include <atomic>

#include "gqaw_internal.cuh"

namespace gqaw {

constexpr int kRotaryThreads = 256;
constexpr int kMaxRotaryDevices = 64;

template <typename T>
__global__ void __launch_bounds__(kRotaryThreads) rotary_kernel(const Params p) {
  pdl_wait();               // the previous step's cache update has read these buffers
  const int D = p.D, half = p.rot_dim / 2, slots = D / 2;
  const long long qrows = (long long)p.B * p.S * p.Nq;
  const long long rows = qrows + (long long)p.B * p.S * p.Nkv;
  const long long n = rows * slots;
  const T *qin = static_cast<const T *>(p.q_in), *kin = static_cast<const T *>(p.k_in);
  T *qout = static_cast<T *>(const_cast<void *>(p.q)), *kout = static_cast<T *>(p.krot);
  const T *rc = static_cast<const T *>(p.rcos), *rs = static_cast<const T *>(p.rsin);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / slots;
    const int slot = (int)(idx - row * slots);
    const bool isq = row < qrows;
    const long long token = isq ? row / p.Nq : (row - qrows) / p.Nkv;  // b * S + s
    const long long off = isq ? row * D : (row - qrows) * D;
    const T *x = (isq ? qin : kin) + off;
    T *y = (isq ? qout : kout) + off;
    const int b = (int)(token / p.S), s = (int)(token - (long long)b * p.S);
    const long long pos = p.pos_ids ? p.pos_ids[token] : (long long)p.seqlens[b] + 1 - p.S + s;
    int i1, i2;  // the two dimensions this thread writes
    if (slot < half) {
      i1 = p.rot_inter ? 2 * slot : slot;
      i2 = p.rot_inter ? 2 * slot + 1 : slot + half;
    } else {  // beyond the rotary dimensions: copy two elements
      i1 = p.rot_dim + 2 * (slot - half);
      i2 = i1 + 1;
    }
    const float x1 = Elem<T>::load(x[i1]), x2 = Elem<T>::load(x[i2]);
    float y1 = x1, y2 = x2;
    if (slot < half) {
      if (pos >= 0 && pos < p.rot_len) {
        const float c = Elem<T>::load(rc[pos * half + slot]), sn = Elem<T>::load(rs[pos * half + slot]);
        y1 = fmaf(x1, c, -x2 * sn);
        y2 = fmaf(x2, c, x1 * sn);
      } else if (slot == 0) {
        flag(p, GQAW_DEV_BAD_POSITION);  // the row is copied unturned
      }
    }
    y[i1] = Elem<T>::store(y1);
    y[i2] = Elem<T>::store(y2);
  }
  pdl_launch_dependents();  // done: the attention kernel may be scheduled
}

// 16-byte vectors of T: unpack to floats (Elem<T>::unpack) and pack back, rounding once.
__device__ __forceinline__ uint4 pack_vec(const float *f, float) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
__device__ __forceinline__ uint4 pack_vec(const float *f, __nv_bfloat16) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// Half a vector of T (8 bytes) as floats: the cos or sin of VEC/2 interleaved pairs.
__device__ __forceinline__ void unpack_half(const void *src, float *f, float) {
  const uint2 u = *static_cast<const uint2 *>(src);
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
}
__device__ __forceinline__ void unpack_half(const void *src, float *f, __nv_bfloat16) {
  const uint2 u = *static_cast<const uint2 *>(src);
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}

// Vector kernel.  Items per row: `pitems` rotation items (split pairs: half / VEC
// vector pairs; interleaved: rd / VEC vectors) then (D - rd) / VEC copied vectors.
// The host takes this kernel only when every count and offset is whole in vectors,
// cos/sin are 16-byte aligned and the item count fits in 31 bits.
template <typename T>
__global__ void __launch_bounds__(kRotaryThreads) rotary_vec_kernel(const Params p) {
  constexpr int VEC = Elem<T>::kPerVec;
  pdl_wait();               // the previous step's cache update has read these buffers
  const unsigned D = p.D, half = p.rot_dim / 2;
  const unsigned pitems = p.rot_inter ? p.rot_dim / VEC : half / VEC;
  const unsigned ipr = pitems + (D - p.rot_dim) / VEC;
  const unsigned S = p.S, Nq = p.Nq, Nkv = p.Nkv;
  const unsigned qrows = p.B * S * Nq;
  const unsigned n = (qrows + p.B * S * Nkv) * ipr;
  for (unsigned idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
    const unsigned row = idx / ipr, item = idx - row * ipr;
    const bool isq = row < qrows;
    const unsigned r = isq ? row : row - qrows;
    const unsigned token = isq ? r / Nq : r / Nkv;  // b * S + s
    const T *x = static_cast<const T *>(isq ? p.q_in : p.k_in) + (size_t)r * D;
    T *y = static_cast<T *>(isq ? const_cast<void *>(p.q) : p.krot) + (size_t)r * D;
    if (item >= pitems) {  // past the rotary width: copy
      const unsigned c = p.rot_dim + (item - pitems) * VEC;
      *reinterpret_cast<uint4 *>(y + c) = *reinterpret_cast<const uint4 *>(x + c);
      continue;
    }
    const unsigned b = token / S, s = token - b * S;
    const long long pos = p.pos_ids ? p.pos_ids[token] : (long long)p.seqlens[b] + 1 - (long long)S + s;
    const bool ok = pos >= 0 && pos < p.rot_len;
    if (!ok && item == 0) flag(p, GQAW_DEV_BAD_POSITION);  // the row is copied unturned
    const T *cs = static_cast<const T *>(p.rcos) + (ok ? pos : 0) * half;
    const T *sn = static_cast<const T *>(p.rsin) + (ok ? pos : 0) * half;
    float a[VEC], o[VEC];
    if (p.rot_inter) {  // pairs (2i, 2i+1) inside one vector
      const unsigned c = item * VEC;
      Elem<T>::unpack(*reinterpret_cast<const uint4 *>(x + c), a);
      float cv[VEC / 2], sv[VEC / 2];
      unpack_half(cs + c / 2, cv, T());
      unpack_half(sn + c / 2, sv, T());
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) {
        const float x1 = a[2 * i], x2 = a[2 * i + 1];
        o[2 * i] = ok ? fmaf(x1, cv[i], -x2 * sv[i]) : x1;
        o[2 * i + 1] = ok ? fmaf(x2, cv[i], x1 * sv[i]) : x2;
      }
      *reinterpret_cast<uint4 *>(y + c) = pack_vec(o, T());
    } else {  // pairs (i, i + half): vectors at c and c + half
      const unsigned c = item * VEC;
      float bv[VEC], cv[VEC], sv[VEC], o2[VEC];
      Elem<T>::unpack(*reinterpret_cast<const uint4 *>(x + c), a);
      Elem<T>::unpack(*reinterpret_cast<const uint4 *>(x + c + half), bv);
      Elem<T>::unpack(*reinterpret_cast<const uint4 *>(cs + c), cv);
      Elem<T>::unpack(*reinterpret_cast<const uint4 *>(sn + c), sv);
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        o[i] = ok ? fmaf(a[i], cv[i], -bv[i] * sv[i]) : a[i];
        o2[i] = ok ? fmaf(bv[i], cv[i], a[i] * sv[i]) : bv[i];
      }
      *reinterpret_cast<uint4 *>(y + c) = pack_vec(o, T());
      *reinterpret_cast<uint4 *>(y + c + half) = pack_vec(o2, T());
    }
  }
  pdl_launch_dependents();  // done: the attention kernel may be scheduled
}

template <typename K>
int resident_blocks(K kernel, int dev, cudaError_t *err) {
  int sms = 0, per_sm = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (*err != cudaSuccess) return 0;
  *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kRotaryThreads, 0);
  if (*err != cudaSuccess) return 0;
  return sms * (per_sm > 0 ? per_sm : 1);
}

cudaError_t launch_rotary(const Params &p, cudaStream_t stream) {
  const bool bf16 = p.qbytes == 2;
  const int vec = bf16 ? 8 : 4;  // elements per 16-byte vector
  const int half = p.rot_dim / 2;
  const long long rows = (long long)p.B * p.S * (p.Nq + p.Nkv);
  const int pitems = p.rot_inter ? p.rot_dim / vec : half / vec;
  const long long vitems = rows * (pitems + (p.D - p.rot_dim) / vec);
  const bool use_vec = (p.rot_inter ? p.rot_dim % vec == 0 : half % vec == 0) && (p.D - p.rot_dim) % vec == 0 &&
                       reinterpret_cast<uintptr_t>(p.rcos) % 16 == 0 && reinterpret_cast<uintptr_t>(p.rsin) % 16 == 0 &&
                       rows < 0x7fffffffLL && vitems < 0x7fffffffLL;
  // resident blocks per device and kernel (index: vector kernel, then bf16), found on first use
  static std::atomic<int> resident[kMaxRotaryDevices][4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int ki = (use_vec ? 2 : 0) + (bf16 ? 1 : 0);
  int slots = dev < kMaxRotaryDevices ? resident[dev][ki].load(std::memory_order_relaxed) : 0;
  if (slots <= 0) {
    switch (ki) {
      case 0: slots = resident_blocks(rotary_kernel<float>, dev, &e); break;
      case 1: slots = resident_blocks(rotary_kernel<__nv_bfloat16>, dev, &e); break;
      case 2: slots = resident_blocks(rotary_vec_kernel<float>, dev, &e); break;
      default: slots = resident_blocks(rotary_vec_kernel<__nv_bfloat16>, dev, &e); break;
    }
    if (e != cudaSuccess) return e;
    if (dev < kMaxRotaryDevices) resident[dev][ki].store(slots, std::memory_order_relaxed);
  }
  const long long n = use_vec ? vitems : rows * (p.D / 2);
  const long long need = (n + kRotaryThreads - 1) / kRotaryThreads;
  const int blocks = (int)(need < slots ? need : slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks > 0 ? blocks : 1);
  cfg.blockDim = dim3(kRotaryThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (ki) {
    case 0: e = cudaLaunchKernelEx(&cfg, rotary_kernel<float>, p); break;
    case 1: e = cudaLaunchKernelEx(&cfg, rotary_kernel<__nv_bfloat16>, p); break;
    case 2: e = cudaLaunchKernelEx(&cfg, rotary_vec_kernel<float>, p); break;
    default: e = cudaLaunchKernelEx(&cfg, rotary_vec_kernel<__nv_bfloat16>, p); break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqaw
