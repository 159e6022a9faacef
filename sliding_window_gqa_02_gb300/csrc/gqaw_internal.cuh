// gqaw_internal.cuh -- device-side building blocks shared by the step's kernels.
//
// The per-item plan follows onnxruntime PR #32419 "Specify GroupQueryAttention
// windowed KV cache layout contract" (Description: L(T), row layout) and PR #31142
// "[CPU] Add windowed kv cache for GQA" (review thread: 64-bit planner arithmetic,
// past length P = seqlens_k[b] + 1 - S).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gqaw.h"

namespace gqaw {

// Everything a kernel needs, passed by value.
struct Params {
  const void *q, *k, *v;     // (B,S,Nq*D), (B,S,Nkv*D), (B,S,Nkv*D)
  const void *pk, *pv;       // past (B,Nkv,C,D)
  void *prk, *prv;           // present (B,Nkv,C,D)
  const int32_t *seqlens;    // (B,)
  const float *bias;         // NULL or [b*bsb + h*bsh + s*bss + j]
  long long bsb, bsh, bss;
  void *out;                 // (B,S,Nq*D)
  float *partials;           // per attention CTA, 2 slots of GB x (D accumulators, max, sum)
  uint32_t *status;          // device status word
  uint32_t *move_count;      // items registered for the cache-update kernel this step
  uint32_t *done_count;      // cache-update blocks finished this step
  uint32_t *job_count;       // cache-update jobs taken this step (separate present buffers)
  int32_t *move_list;        // (B,) the registered items
  uint32_t *tickets;         // per attention unit: contributors finished
  int32_t *resident_out;     // NULL or (B,)
  int B, S, Nq, Nkv, D, C, W, total, group;
  int headblocks;            // query-head blocks per kv head
  long long nunits;          // attention units: B * S * Nkv * headblocks
  int tpu;                   // key tiles per unit: ceil(min(W, total) / tile)
  float qscale;              // q multiplier: scale*log2(e), or scale/softcap with softcap
  float capmul;              // softcap*log2(e), or 0 without softcap
  float biasmul;             // log2(e)
  int ncg;                   // most column groups per cache row in the copy jobs
  int rowbytes;              // D * cache element size
  int qbytes;                // query/key/value/output element size (4 or 2)
  const float *sink;         // NULL or (Nq,): sink logit per query head (natural-log units)
  int sink_mode;             // 0: no sink; 1: sink[h]; 2: a sink of 0 for every head
  // rotary embedding (rot_dim > 0): q is the turned query in the workspace and krot the
  // turned keys, written by the rotary kernel from the step's inputs q_in and k_in (k is
  // krot, or the codes of krot with a quantized cache)
  const void *q_in, *k_in;
  void *krot;
  const void *rcos, *rsin;   // (rot_len, rot_dim / 2) in the step's dtype
  const long long *pos_ids;  // NULL (positions P_b + s) or (B, S)
  int rot_dim, rot_inter, rot_len;
  // quantized cache (quant > 0: GQAW_I8 or GQAW_E4M3): k and v above are the code rows of
  // the step's new keys and values in the workspace, written by the quantize kernel from
  // kq_in and vq_in (the step's rows of dtype T); ks, vs: device scales
  int quant;
  const void *kq_in, *vq_in;
  const float *ks, *vs;
  void *q16;                 // NULL, or an fp16 copy of the query rows for the tensor-core kernel
  // small-step kernel, bf16 caches: the rows a CTA moves whose destination another CTA
  // may still read, written later by the unit's last contributor (kMoveStashBytes per CTA)
  unsigned char *stash;
  int no_finish;             // the host launches no cache-update kernel for this step
};

constexpr float kLog2e = 1.4426950408889634f;

// The sink logit of query head h in log2 units, -inf when there is none (mobius
// issue #111, Part 1.1 input head_sink and Part 1.3 smooth_softmax).
__device__ __forceinline__ float sink_log2(const Params &p, int h) {
  if (p.sink_mode == 1) return p.sink[h] * kLog2e;
  return p.sink_mode == 2 ? 0.f : -INFINITY;
}

// Output of a softmax row from its accumulator A and denominator l, both taken
// against the reference maximum m (log2 units), with the sink logit s2 joining the
// denominator: A / (l + 2^(s2 - m)), scaled by 2^(m - s2) when the sink is the larger
// so that nothing overflows.  Without a sink (s2 = -inf) this is A / l exactly.
__device__ __forceinline__ float sink_divide(float A, float l, float m, float s2) {
  if (s2 <= m) return A / (l + exp2f(s2 - m));
  const float f = exp2f(m - s2);
  return (A * f) / fmaf(l, f, 1.f);
}

// The factor 1 / (l + 2^(s2 - m)) that turns accumulators into outputs, in the same
// overflow-safe form; 1 / l exactly without a sink.
__device__ __forceinline__ float sink_reciprocal(float l, float m, float s2) {
  if (s2 <= m) return 1.f / (l + exp2f(s2 - m));
  const float f = exp2f(m - s2);
  return f / fmaf(l, f, 1.f);
}

// L(T) in 64-bit integers.
__device__ __forceinline__ long long resident_len(long long T, long long C, long long W) {
  if (T <= C) return T;
  const long long G = C - W + 1;
  return T - G * ((T - C + G - 1) / G);
}

struct Plan {
  long long T, P, Lp, Lt;
};

// Per-item plan from seqlens_k[b] (plan_from: from that value, already loaded).  Returns
// false (and the caller flags the item) when the item's seqlens_k is out of range.
__device__ __forceinline__ bool plan_from(const Params &p, int seqlen, Plan &pl) {
  const long long T = (long long)seqlen + 1;
  const long long P = T - p.S;
  if (P < 0 || T > (long long)p.total) return false;
  pl.T = T;
  pl.P = P;
  pl.Lp = resident_len(P, p.C, p.W);
  pl.Lt = resident_len(T, p.C, p.W);
  return true;
}
__device__ __forceinline__ bool plan_item(const Params &p, int b, Plan &pl) { return plan_from(p, p.seqlens[b], pl); }

__device__ __forceinline__ void flag(const Params &p, uint32_t bits) { atomicOr(p.status, bits); }

// Flag of a cache-update list entry (item index | flag): present is a separate buffer and
// the attention kernel has written the surviving rows of the window and the new rows;
// only the surviving rows below the window (which the step does not read) are left.
constexpr int kListBelowOnly = 1 << 30;

// Does item b need the cache-update kernel?  Yes when a block of rows is reclaimed
// (seed = L(P) + S - L(T) > 0: rows move, and the new rows land on rows the attention
// may still read) or when present is a separate buffer (every surviving row is
// copied).  Otherwise the new rows go to rows [L(P), L(P) + S), which no query of the
// step reads, and the attention kernel appends them itself.
__device__ __forceinline__ bool item_moves(const Params &p, const Plan &pl) {
  return pl.Lp + p.S - pl.Lt > 0 || p.pk != p.prk || p.pv != p.prv;
}

// ---------------------------------------------------------------- conversions

// 1-byte codes of a quantized cache (int8, fp8 e4m3); only their size and bits matter here.
struct CodeI8 {
  uint8_t bits;
};
struct CodeE4M3 {
  uint8_t bits;
};

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static void unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static float store(float x) { return x; }
  __device__ __forceinline__ static float load(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  // A bfloat16 is the high half of a float32: widening is a shift (exact).
  __device__ __forceinline__ static void unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = __uint_as_float(u.z << 16);
    f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = __uint_as_float(u.w << 16);
    f[7] = __uint_as_float(u.w & 0xffff0000u);
  }
  __device__ __forceinline__ static __nv_bfloat16 store(float x) { return __float2bfloat16_rn(x); }
  __device__ __forceinline__ static float load(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Float pairs out of a 16-byte vector of elements: pair j covers elements 2j and 2j+1.
template <typename T> struct Pairs;
template <> struct Pairs<float> {
  // pair j (0..1) of a 16-byte vector of 4 floats
  __device__ __forceinline__ static float2 get(const uint4 &u, int j) {
    return j == 0 ? make_float2(__uint_as_float(u.x), __uint_as_float(u.y))
                  : make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
};
template <> struct Pairs<__nv_bfloat16> {
  // pair j (0..3) of a 16-byte vector of 8 bfloat16: widening is a shift (exact)
  __device__ __forceinline__ static float2 get(const uint4 &u, int j) {
    const uint32_t w = j == 0 ? u.x : (j == 1 ? u.y : (j == 2 ? u.z : u.w));
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};
template <> struct Pairs<CodeI8> {
  // pair j (0..7) of a 16-byte vector of 16 int8 codes, as floats (exact): the byte,
  // biased by 128, is placed in the low mantissa bits of 2^23, which is then subtracted
  // with the bias
  __device__ __forceinline__ static float2 get(const uint4 &u, int j) {
    const uint32_t w = (j < 2 ? u.x : (j < 4 ? u.y : (j < 6 ? u.z : u.w))) ^ 0x80808080u;
    const uint32_t b = (j & 1) * 2;  // first byte of the pair in the word
    const float lo = __uint_as_float(__byte_perm(w, 0x4B000000u, b | 0x7540u)) - 8388736.f;
    const float hi = __uint_as_float(__byte_perm(w, 0x4B000000u, (b + 1) | 0x7540u)) - 8388736.f;
    return make_float2(lo, hi);
  }
};
template <> struct Pairs<CodeE4M3> {
  // pair j (0..7) of a 16-byte vector of 16 fp8 e4m3 codes, as floats (exact): the
  // hardware pair conversion to half precision, then widening
  __device__ __forceinline__ static float2 get(const uint4 &u, int j) {
    const uint32_t w = j < 2 ? u.x : (j < 4 ? u.y : (j < 6 ? u.z : u.w));
    const uint16_t pair = (uint16_t)(w >> ((j & 1) * 16));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
  }
};


// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete; give up after about
// two seconds of SM clock (4e9 cycles) (returns false: the caller flags GQAW_DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > 4000000000ll) return false;
  }
  return true;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on `bar` with tx bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read once (K/V rows of the window).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Programmatic dependent launch: the kernels of a step are launched with
// programmatic stream serialisation, so a kernel may start while the previous one in
// the stream drains.  pdl_wait() blocks until that previous kernel has completed and
// its memory is visible; nothing produced upstream may be read before it.
// pdl_launch_dependents() lets the next kernel in the stream be launched early (its
// CTAs then wait in their own pdl_wait()).  A kernel signals only when its CTA's main
// work is done: signalled at the start, the next grid's CTAs become resident as SMs
// free up, ahead of this grid's CTAs that are not resident yet, and hold those SMs
// while they wait -- a persistent grid with one CTA per SM then runs partly serialised.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns whether `pred` held for any participating thread.
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

}  // namespace gqaw
