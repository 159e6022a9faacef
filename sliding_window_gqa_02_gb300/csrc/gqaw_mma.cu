// gqaw_mma.cu -- multi-token windowed GQA attention on the 5th-generation tensor cores.
//
// For steps with S > 1 new tokens (speculative verify, chunked prefill) the logits of
// all query heads of a kv group and of many tokens share the same K/V rows, so
// Q.K^T and P.V are genuine dense contractions: they run as tcgen05.mma (bf16
// operands, fp32 accumulators in tensor memory).
//
// What it computes is the same as the decode kernel (gqaw_attend.cuh): query of token
// s at absolute position i = P + s attends keys i - W < j <= i (onnxruntime PR #34226
// "Fix CPU Attention causal mask for q_len=1 with past_key and kv_len > 1",
// Description), logit softcap * tanh(scale q.k / softcap) + bias[b, h, s, j] with j the
// absolute key position (PR #32419 "Specify GroupQueryAttention windowed KV cache
// layout contract", Description), keys before P read from the pre-step cache rows,
// keys from P on from the new input rows -- no staging copy (PR #31142 "[CPU] Add
// windowed kv cache for GQA", "Staging for hazardous steps"), since this kernel runs
// before any cache row moves.
//
// Tiling: units of (item, kv head, 128-row query tile, key split), walked grid-strided
// by a persistent grid of one CTA per SM.  Query rows are (token, head) pairs
// r = t * g + head, so a tile holds 128/g tokens x g heads.  Keys come in tiles of 128:
// cache tiles ending exactly at the item's last past row (the rows below the window in
// the first one are older resident rows, or zeros where the tensor map runs below row
// 0: always finite), then tiles of the new rows.  Key tiles are numbered across the
// units of a CTA, so the rings and barrier phases run on from one unit to the next: the
// next unit's query tile loads once the last S product of the previous one is done, its
// first S product runs while the softmax warps finish the previous unit, and its first
// O += P V waits until they have read O out of tensor memory.
//
// Warp roles (12 warps):
//   warps 0-7   softmax: two threads per query row (TMEM lane), warps w and w + 4
//               taking the row's key columns 0-63 and 64-127; per key tile each reads
//               its 64 logits twice from tensor memory (the maximum, exchanged with
//               the partner through shared memory; then P = 2^(z - m) as bf16 into
//               tensor memory) and keeps a partial running sum
//   warp 8      MMA issue (one thread): S(k) = Q K(k)^T into one of two tensor-memory
//               buffers (both operands in shared memory), O += P V(k) (P from tensor
//               memory, V from shared memory)
//   warp 9      TMA loads of the query tile and of K tiles into a 3-stage ring
//   warp 10     TMA loads of V tiles into a 2-stage ring
//   warp 11     bookkeeping of the item (resident length, cache-update list) and the
//               appends of the tile's new rows, off the softmax's path
// Tensor memory (512 columns): S buffers [0, 128) and [128, 256), O [256, 384), P
// buffers [384, 448) and [448, 512); nothing aliases.  Per key tile k the MMA thread
// issues S(k+1) as soon as K(k+1) has landed and the softmax is done with S(k-1), so it
// runs while the softmax works on S(k); then O += P(k) V(k) once P(k) is written.  The
// completion of S(k) also covers O += P(k-2) V(k-2), issued before it, so P buffer
// k % 2 is free when S(k) is; O += P(k-1) V(k-1) is waited for only when the softmax has
// to rescale O.  Likewise S buffer (k+1) % 2 is free once P(k-1) is written.
#include <cuda.h>

#include "gqaw_tc.cuh"

namespace gqaw {

namespace {

constexpr int kRows = 128;       // query rows per CTA (M)
constexpr int kKeys = 128;       // keys per tile (N of Q.K^T, K of P.V)
constexpr int kHalfKeys = 64;    // columns of a tile row per softmax thread
constexpr int kD = 128;          // head size
constexpr int kHalf = 16384;     // bytes of a [128 rows][64 bf16] swizzled block
constexpr int kTile = 2 * kHalf; // one 128 x 128 bf16 operand
constexpr int kKStages = 3, kVStages = 2;
constexpr int kMmaWarp = 8, kLoadWarp = 9, kVLoadWarp = 10, kAppendWarp = 11;
constexpr int kThreads = 384;
// shared memory: Q, the K ring, the V ring (each operand two 64-column halves)
constexpr int kSmemQ = 0;
constexpr int kSmemK = kSmemQ + kTile;
constexpr int kSmemV = kSmemK + kKStages * kTile;
constexpr int kSmemBars = kSmemV + kVStages * kTile;
constexpr int kSmemTotal = kSmemBars + 256;
constexpr int kSmemAlloc = kSmemTotal + 1024;  // room to align the base to 1024 bytes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 2 * kKeys, kTmemP = kTmemO + kD;  // P: two buffers of 64 columns
constexpr float kRescaleLog2 = 8.0f;           // lazy rescale threshold (log2 units)
constexpr float kDangerLog2 = 16.0f;           // most a fast-path P may exceed 1 (log2 units)
constexpr int kSoftmaxBar = 5;                 // named barrier of the 8 softmax warps (1-4: warp pairs)

constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(kRows, kKeys, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kRows, kD, 0, 1);

// 2^x, approximate (ex2.approx, relative error ~2^-22; -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh from its exponential form, tanh(x) = 1 - 2 / (e^(2x) + 1): absolute error about
// 1e-7 (it saturates to +-1 correctly), which is what a logit cap multiplies.
__device__ __forceinline__ float fast_tanh(float x) {
  const float e = fast_exp2(2.8853900817779268f * fminf(fmaxf(x, -15.f), 15.f));  // 2 log2(e) x
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return fmaf(-2.f, r, 1.f);
}

// Packed pairs of fp32 (sm_100 family): one instruction computes both lanes.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ bool abort_set(const int *f) { return *reinterpret_cast<const volatile int *>(f) != 0; }

// Bit c set when column 32 * c32 + c of a key tile lies in [c_lo, c_hi).
__device__ __forceinline__ uint32_t chunk_mask(int c32, int c_lo, int c_hi) {
  const int lo = min(max(c_lo - c32 * 32, 0), 32), hi = min(max(c_hi - c32 * 32, 0), 32);
  const uint32_t below_hi = hi >= 32 ? 0xffffffffu : (1u << hi) - 1u;
  const uint32_t below_lo = lo >= 32 ? 0xffffffffu : (1u << lo) - 1u;
  return below_hi & ~below_lo;
}

// The largest logit of this thread's row among its 64 columns of the tile, read from
// tensor memory 32 at a time (kMasked: only columns in [c_lo, c_hi), relative to the
// first of the 64, count).
template <bool kMasked>
__device__ __forceinline__ float tile_max(uint32_t ts, int c_lo, int c_hi) {
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c32 = 0; c32 < kHalfKeys / 32; ++c32) {
    float v[32];
    tc::tmem_ld32(ts + c32 * 32, v);
    if (kMasked) {
      const uint32_t m = chunk_mask(c32, c_lo, c_hi);
#pragma unroll
      for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], (m >> c) & 1u ? v[c] : -INFINITY);
    } else {
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        mx[(c / 8) & 3] = max3(mx[(c / 8) & 3], v[c], v[c + 1]);
        mx[(c / 8) & 3] = max3(mx[(c / 8) & 3], v[c + 2], v[c + 3]);
        mx[(c / 8) & 3] = max3(mx[(c / 8) & 3], v[c + 4], v[c + 5]);
        mx[(c / 8) & 3] = max3(mx[(c / 8) & 3], v[c + 6], v[c + 7]);
      }
    }
  }
  return max3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
}

// P = 2^(z * zs - base) of this thread's 64 logits of the row (tensor memory at ts), as
// bf16 pairs into 32 columns at tp; returns the sum of the fp32 values.  The stores are
// waited for by the caller.  A fully visible tile works on packed pairs; with kMax it
// also leaves the largest raw logit of the 64 in *mx.
template <bool kMasked, bool kMax = false>
__device__ __forceinline__ float tile_p(uint32_t ts, uint32_t tp, int c_lo, int c_hi, float zs, float base,
                                        float *mx = nullptr) {
  if (kMasked) {
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c32 = 0; c32 < kHalfKeys / 32; ++c32) {
      float v[32];
      tc::tmem_ld32(ts + c32 * 32, v);
      const uint32_t m = chunk_mask(c32, c_lo, c_hi);
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float a0 = (m >> (2 * c)) & 1u ? fast_exp2(fmaf(v[2 * c], zs, -base)) : 0.f;
        const float a1 = (m >> (2 * c + 1)) & 1u ? fast_exp2(fmaf(v[2 * c + 1], zs, -base)) : 0.f;
        ls[c & 3] += a0 + a1;
        pk[c] = tc::pack_bf16x2(a0, a1);
      }
      tc::tmem_st16_async(tp + c32 * 16, pk);
    }
    return (ls[0] + ls[1]) + (ls[2] + ls[3]);
  }
  const uint64_t zs2 = pack2(zs, zs), nb2 = pack2(-base, -base);
  uint64_t acc[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c32 = 0; c32 < kHalfKeys / 32; ++c32) {
    float v[32];
    tc::tmem_ld32(ts + c32 * 32, v);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if (kMax) m4[c & 3] = max3(m4[c & 3], v[2 * c], v[2 * c + 1]);
      float x0, x1;
      unpack2(fma2(pack2(v[2 * c], v[2 * c + 1]), zs2, nb2), x0, x1);
      const float a0 = fast_exp2(x0), a1 = fast_exp2(x1);
      acc[c & 1] = add2(acc[c & 1], pack2(a0, a1));
      pk[c] = tc::pack_bf16x2(a0, a1);
    }
    tc::tmem_st16_async(tp + c32 * 16, pk);
  }
  if (kMax) *mx = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
  float l0, l1, l2, l3;
  unpack2(acc[0], l0, l1);
  unpack2(acc[1], l2, l3);
  return (l0 + l1) + (l2 + l3);
}

// One unit of work of a CTA: (item, kv head, 128-row query tile, key split), and the
// key tiles it covers.  Every warp role decodes the same sequence of units.
struct Unit {
  Plan pl;
  long long P, id;  // id: (item, kv head, query tile), the index of the split tickets
  int b, kvh, rt, sp, s0, s_end, tpq, nc, t_begin, ntl;
  bool ok, moves;
};

// seqlens_k of unit u's item: loaded one unit ahead, so the load's latency is not paid
// at the unit boundary.
__device__ __forceinline__ int unit_seqlen(const Params &p, const TcArgs &ta, long long u) {
  return u < ta.units ? p.seqlens[(unsigned)u / (unsigned)ta.nsplit / (unsigned)ta.rowtiles / (unsigned)p.Nkv] : 0;
}

__device__ __forceinline__ Unit unit_at(const Params &p, const TcArgs &ta, long long u, int seqlen) {
  Unit x;
  const unsigned uu = (unsigned)u, id = uu / (unsigned)ta.nsplit;  // units < 2^31 (host check)
  const unsigned slice = id / (unsigned)ta.rowtiles;
  x.sp = (int)(uu - id * (unsigned)ta.nsplit);
  x.id = id;
  x.rt = (int)(id - slice * (unsigned)ta.rowtiles);
  x.kvh = (int)(slice % (unsigned)p.Nkv);
  x.b = (int)(slice / (unsigned)p.Nkv);
  x.ok = plan_from(p, seqlen, x.pl);
  x.s0 = x.rt * ta.tokens_per_tile;
  x.s_end = x.s0 + ta.tokens_per_tile < p.S ? x.s0 + ta.tokens_per_tile : p.S;
  x.tpq = (x.s_end - x.s0 + 3) / 4;  // tokens per TMEM lane quarter
  x.P = 0;
  x.nc = x.t_begin = x.ntl = 0;
  x.moves = false;
  if (x.ok) {
    // nc cache tiles ending at P, then tiles of new rows
    x.P = x.pl.P;
    const long long klo = x.P + x.s0 - p.W + 1 > 0 ? x.P + x.s0 - p.W + 1 : 0;
    x.nc = (int)((x.P - klo + kKeys - 1) / kKeys);
    const int nt = x.nc + (x.s_end + kKeys - 1) / kKeys;
    x.t_begin = (int)((unsigned)(x.sp * nt) / (unsigned)ta.nsplit);
    x.ntl = (int)((unsigned)((x.sp + 1) * nt) / (unsigned)ta.nsplit) - x.t_begin;
    x.moves = item_moves(p, x.pl);
  }
  return x;
}

// Absolute position of key tile t's first column.
__device__ __forceinline__ long long key0(const Unit &x, int t) {
  return t < x.nc ? x.P - (long long)(x.nc - t) * kKeys : x.P + (long long)(t - x.nc) * kKeys;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    mma_attend_kernel(const Params p, const TcArgs ta, const __grid_constant__ TcMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmemBars);
  uint64_t *q_full = bars;                   // the unit's query tile landed
  uint64_t *k_full = bars + 1;               // [3] K stage landed
  uint64_t *k_free = bars + 4;               // [3] K stage read by its S product
  uint64_t *v_full = bars + 7;               // [2] V stage landed
  uint64_t *s_full = bars + 9;               // [2] S buffer written
  // p_full and pv_done are per P buffer: the softmax may finish P(k+1) before the MMA
  // thread has looked for P(k), and a parity wait cannot tell two phases apart.
  uint64_t *p_full = bars + 11;              // [2] P buffer written (and O rescaled) by the softmax warps
  uint64_t *pv_done = bars + 13;             // [2] O += P V(k) done: P buffer and V stage k % 2 free
  uint64_t *mma_done = bars + 15;            // every MMA of the CTA done
  uint64_t *q_free = bars + 16;              // the unit's last S product done: the query tile may be replaced
  uint64_t *o_free = bars + 17;              // the softmax warps have read the unit's O
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 18);
  __shared__ int s_last, s_abort;
  __shared__ float xch[3][2][kRows];  // [tile & 1 | 2 for the sums][column half][row]
  __shared__ int xok[2][2][4];        // [tile & 1][column half][lane quarter]: the wait held

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    mbar_init(o_free, 8);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(mma_done, 1);
    mbar_fence_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  const int g = p.group;
  // Units u = blockIdx.x + i * gridDim.x; key tiles and query tiles are numbered across
  // them (gk, qi), so every ring and barrier phase simply continues from unit to unit.

  if (warp == kLoadWarp || warp == kVLoadWarp) {
    // ------------------------------------------------------------ TMA loads (K and Q | V)
    if (lane == 0) {
      const bool value = warp == kVLoadWarp;
      const uint64_t pol = tc::policy_evict_normal(), qpol = policy_evict_first();
      const int nst = value ? kVStages : kKStages;
      uint64_t *full = value ? v_full : k_full, *empty = value ? pv_done : k_free;
      unsigned char *ring = smem + (value ? kSmemV : kSmemK);
      long long gk = 0;
      int qi = 0, st = 0, ph = 0;  // tile j sits in stage j % nst, phase (j / nst) & 1
      bool fine = true;
      Unit x = unit_at(p, ta, blockIdx.x, unit_seqlen(p, ta, blockIdx.x));
      for (long long u = blockIdx.x; u < ta.units && fine && !abort_set(&s_abort); u += gridDim.x) {
        // the next unit is decoded while this one's loads wait for ring stages
        const int sq_next = unit_seqlen(p, ta, u + gridDim.x);
        Unit nx;
        bool have_nx = false;
        auto decode_next = [&]() {
          if (!have_nx) nx = unit_at(p, ta, u + gridDim.x, sq_next);
          have_nx = true;
        };
        const int slice = x.b * p.Nkv + x.kvh;
        for (int k = 0; k < x.ntl; ++k) {
          if (gk >= nst && !mbar_wait(&empty[st], ph ^ 1)) {  // the tile nst back has been read
            fine = false;
            break;
          }
          const int t = x.t_begin + k;
          unsigned char *dst = ring + st * kTile;
          mbar_arrive_expect_tx(&full[st], kTile);
          if (t < x.nc) {
            const CUtensorMap *m = value ? &maps.vc : &maps.kc;
            const int row = (int)(x.pl.Lp - (long long)(x.nc - t) * kKeys);  // may be < 0: zeros
            tc::tma_load_3d(dst, m, 0, row, slice, &full[st], pol);
            tc::tma_load_3d(dst + kHalf, m, 64, row, slice, &full[st], pol);
          } else {
            const CUtensorMap *m = value ? &maps.vn : &maps.kn;
            const int tokrow = x.b * p.S + (t - x.nc) * kKeys;
            tc::tma_load_3d(dst, m, 0, x.kvh, tokrow, &full[st], pol);
            tc::tma_load_3d(dst + kHalf, m, 64, x.kvh, tokrow, &full[st], pol);
          }
          ++gk;
          if (++st == nst) st = 0, ph ^= 1;
          // the query tile after the unit's first K tile (which only needs a free ring
          // stage), once the previous unit's S products are done with the last one
          if (k == 0 && !value) {
            if (qi > 0 && !mbar_wait(q_free, (qi - 1) & 1)) {
              fine = false;
              break;
            }
            mbar_arrive_expect_tx(q_full, kTile);
            for (int q = 0; q < 4; ++q) {  // quarter q: tokens s0 + q * tpq ..., rows [32q, 32q + 32)
              const int qtok = x.b * p.S + x.s0 + q * x.tpq;
              tc::tma_load_3d(smem + kSmemQ + q * 4096, &maps.q, 0, x.kvh * g, qtok, q_full, qpol);
              tc::tma_load_3d(smem + kSmemQ + kHalf + q * 4096, &maps.q, 64, x.kvh * g, qtok, q_full, qpol);
            }
            ++qi;
            if (u + gridDim.x < ta.units) {  // the next unit's query tile into L2
              decode_next();
              for (int q = 0; q < 4; ++q)
                for (int c0 = 0; c0 < 128; c0 += 64)
                  tc::tma_prefetch_3d(&maps.q, c0, nx.kvh * g, nx.b * p.S + nx.s0 + q * nx.tpq);
            }
          }
          if (k == 0) decode_next();
        }
        decode_next();
        x = nx;
      }
      if (!fine) {
        flag(p, GQAW_DEV_TIMEOUT);
        s_abort = 1;
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (long long j = gk - nst > 0 ? gk - nst : 0; j < gk; ++j)
        if (!mbar_wait(&full[j % nst], (j / nst) & 1)) flag(p, GQAW_DEV_TIMEOUT);
      if (!value && qi > 0 && !mbar_wait(q_full, (qi - 1) & 1)) flag(p, GQAW_DEV_TIMEOUT);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      // Shared-memory descriptors are built once; an operand at byte offset x from a base
      // is the base descriptor plus x / 16 (the start-address field, bits 0-13, cannot
      // carry: every address is below 256 KB).
      const uint64_t dq = tc::smem_desc_sw128(smem + kSmemQ, 16, 1024);
      const uint64_t dk = tc::smem_desc_sw128(smem + kSmemK, 16, 1024);
      const uint64_t dv = tc::smem_desc_sw128(smem + kSmemV, kHalf, 1024);
      auto issue_s = [&](int kst, int buf) {  // S(buf) = Q K^T, K in stage kst
        const uint64_t b0 = dk + (uint64_t)((kst * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk / 4) * kHalf + (kk % 4) * 32) >> 4);
          tc::mma_bf16_ss(tmem + buf * kKeys, dq + off, b0 + off, kIdescQK, kk > 0);
        }
      };
      auto issue_o = [&](int buf, bool acc) {  // O += P V, P buffer and V stage buf
        // V: rows = keys (K), 64-dim halves (MN) 16 KB apart, 8-key groups 1 KB apart
        const uint64_t b0 = dv + (uint64_t)((buf * kTile) >> 4);
        const uint32_t pa = tmem + kTmemP + buf * (kKeys / 2);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc::mma_bf16_ts(tmem + kTmemO, pa + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, acc || kk > 0);
      };
      // K(j) sits in stage j % 3 with phase (j / 3) & 1; (kst, kph) track the next K to
      // read.  K(k + 1) is waited for one tile ahead, off the path from O += P(k-1) V(k-1)
      // to S(k+1).  An abort elsewhere shows up here as an expired wait.
      long long gk = 0;
      int qi = 0, kst = 0, kph = 0;
      auto next_k = [&]() {
        kst = kst == kKStages - 1 ? 0 : kst + 1;
        if (kst == 0) kph ^= 1;
      };
      bool fine = true;
      Unit x = unit_at(p, ta, blockIdx.x, unit_seqlen(p, ta, blockIdx.x));
      for (long long u = blockIdx.x; u < ta.units && fine; u += gridDim.x) {
        // the next unit is decoded right after this one's first S product is issued
        const int sq_next = unit_seqlen(p, ta, u + gridDim.x);
        if (x.ntl <= 0) {
          x = unit_at(p, ta, u + gridDim.x, sq_next);
          continue;
        }
        fine = mbar_wait(q_full, qi & 1) && mbar_wait(&k_full[kst], kph);
        if (!fine) break;
        tc::fence_after_sync();
        issue_s(kst, (int)(gk & 1));
        tc::mma_commit(&s_full[gk & 1]);
        tc::mma_commit(&k_free[kst]);
        next_k();
        const Unit nx = unit_at(p, ta, u + gridDim.x, sq_next);
        if (x.ntl == 1) tc::mma_commit(q_free);
        if (x.ntl > 1 && !(fine = mbar_wait(&k_full[kst], kph))) break;
        for (int k = 0; k < x.ntl && fine; ++k) {
          const long long gt = gk + k;
          if (k + 1 < x.ntl) {  // S(k + 1) while the softmax works on S(k); P(k - 1) freed its buffer
            const int buf = (int)((gt + 1) & 1);
            tc::fence_after_sync();
            issue_s(kst, buf);
            tc::mma_commit(&s_full[buf]);
            tc::mma_commit(&k_free[kst]);
            next_k();
            if (k + 2 == x.ntl) tc::mma_commit(q_free);  // the unit's last S product
            if (k + 2 < x.ntl && !(fine = mbar_wait(&k_full[kst], kph))) break;
          }
          // the first O += P V of a unit overwrites O: the softmax has read the last unit's
          fine = mbar_wait(&v_full[gt & 1], (gt >> 1) & 1) && mbar_wait(&p_full[gt & 1], (gt >> 1) & 1) &&
                 (k > 0 || qi == 0 || mbar_wait(o_free, (qi - 1) & 1));
          if (!fine) break;
          tc::fence_after_sync();
          issue_o((int)(gt & 1), k > 0);
          tc::mma_commit(&pv_done[gt & 1]);
        }
        gk += x.ntl;
        ++qi;
        x = nx;
      }
      if (!fine) {
        flag(p, GQAW_DEV_TIMEOUT);
        s_abort = 1;
      }
      tc::mma_commit(mma_done);  // every MMA issued has completed before TMEM is released
      if (!mbar_wait(mma_done, 0)) flag(p, GQAW_DEV_TIMEOUT);
    }
  } else if (warp == kAppendWarp) {
    // ------------------------------------------------------------ bookkeeping, appends
    for (long long u = blockIdx.x; u < ta.units; u += gridDim.x) {
      const Unit x = unit_at(p, ta, u, unit_seqlen(p, ta, u));
      if (!x.ok) {
        if (x.kvh == 0 && x.rt == 0 && x.sp == 0 && lane == 0) flag(p, GQAW_DEV_BAD_SEQLEN);
        continue;
      }
      if (x.kvh == 0 && x.rt == 0 && x.sp == 0 && lane == 0) {
        if (p.resident_out) p.resident_out[x.b] = (int32_t)x.pl.Lt;
        if (x.moves) p.move_list[atomicAdd(p.move_count, 1u)] = x.b;
      }
      if (!x.moves && x.sp == 0) {  // append the new rows of this tile's tokens at L(P) + s
        constexpr int kPerRow = kD * 2 / 16, kBatch = 8;
        const int nrow = x.s_end - x.s0;
        const int n = 2 * nrow * kPerRow;
        for (int e0 = 0; e0 < n; e0 += 32 * kBatch) {
          uint4 v[kBatch];
          size_t dst[kBatch];
#pragma unroll
          for (int uu = 0; uu < kBatch; ++uu) {
            const int e = e0 + uu * 32 + lane;
            if (e < n) {
              const int tensor = e / (nrow * kPerRow);
              const int rem = e % (nrow * kPerRow);
              const int s = x.s0 + rem / kPerRow, vec = rem % kPerRow;
              const size_t in_row = ((size_t)x.b * p.S + s) * p.Nkv + x.kvh;
              const size_t out_row = ((size_t)x.b * p.Nkv + x.kvh) * (size_t)p.C + (size_t)(x.pl.Lp + s);
              v[uu] = reinterpret_cast<const uint4 *>(static_cast<const char *>(tensor ? p.v : p.k) + in_row * kD * 2)[vec];
              dst[uu] = (out_row * kD * 2 + (size_t)vec * 16) | (size_t)tensor;  // 16-byte aligned: bit 0 free
            }
          }
#pragma unroll
          for (int uu = 0; uu < kBatch; ++uu) {
            if (e0 + uu * 32 + lane < n) {
              char *base = static_cast<char *>(dst[uu] & 1 ? p.prv : p.prk);
              *reinterpret_cast<uint4 *>(base + (dst[uu] & ~(size_t)1)) = v[uu];
            }
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- softmax (warps 0-7)
  if (warp < 8) {
    const int wq = warp & 3;                       // TMEM lane quarter
    const int hf = (warp >> 2) & 1;                // column half of the row
    const int r = wq * 32 + lane;                  // query row = TMEM lane
    const int bar_pair = 1 + wq;                   // named barrier of warps wq and wq + 4
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    // this thread's O columns [64 hf, 64 hf + 64) and P columns [32 hf, 32 hf + 32)
    const uint32_t to = tmem + kTmemO + hf * kHalfKeys + lane_off, tp = tmem + kTmemP + hf * 32 + lane_off;
    const bool plain = p.capmul == 0.f && p.bias == nullptr;  // logits need only the scale
    long long gk = 0;  // key tiles of earlier units
    Unit x = unit_at(p, ta, blockIdx.x, unit_seqlen(p, ta, blockIdx.x));
    for (long long u = blockIdx.x; u < ta.units; u += gridDim.x) {
      // the next unit is decoded while the first S product of this one is computed
      const int sq_next = unit_seqlen(p, ta, u + gridDim.x);
      Unit nx;
      bool have_nx = false;
      auto decode_next = [&]() {
        if (!have_nx) nx = unit_at(p, ta, u + gridDim.x, sq_next);
        have_nx = true;
      };
      // The tile's tokens are spread evenly over the four lane quarters, tpq tokens
      // each, so a short step (S x g < 128 rows) still gives every warp real rows.
      const int tl = lane / g;                     // token within the quarter
      const int tok = x.s0 + wq * x.tpq + tl;
      const int hh = lane % g;
      const bool row_ok = x.ok && tl < x.tpq && tok < x.s_end;
      const long long qpos = x.P + tok;            // absolute position of the row's token
      const long long rlo = qpos - p.W + 1 > 0 ? qpos - p.W + 1 : 0;
      const int h = x.kvh * g + hh;
      float m_run = -INFINITY, l_run = 0.f, o_owed = 1.f;
      int done = 0;
      if (x.ntl > 0) {
        const float *bias_row = (row_ok && p.bias) ? p.bias + (long long)x.b * p.bsb + (long long)h * p.bsh +
                                                         (long long)tok * p.bss
                                                   : nullptr;
        // Visible columns of this row's half in tile k: [lo - 128 k, hi - 128 k) relative
        // to the half's first column, clamped (consecutive key tiles start 128 positions
        // apart, across the cache/new boundary too).  Both bounds only decrease, so they
        // are kept at -128 once below it.
        int lo = 0, hi = 0;
        if (row_ok) {
          const long long j0 = key0(x, x.t_begin) + hf * kHalfKeys;
          lo = (int)min(max(rlo - j0, -128LL), 1LL << 30);
          hi = (int)min(max(qpos - j0 + 1, -128LL), 1LL << 30);
        }
        // pend: the factor O in tensor memory still owes once O += P(k-1) V(k-1) has
        // landed (a reference raised after P(k-1) was computed against the old one)
        float pend = 1.f;
          for (int k = 0; k < x.ntl; ++k) {
            const long long gt = gk + k;  // tile number across units
            const uint32_t ts = tmem + (uint32_t)(gt & 1) * kKeys + hf * kHalfKeys + lane_off;  // this half of S(k)
            const uint32_t tpk = tp + (uint32_t)(gt & 1) * (kKeys / 2);
            const int c_lo = min(max(lo, 0), kHalfKeys), c_hi = min(max(hi, 0), kHalfKeys);
            lo = max(lo - kKeys, -kKeys);
            hi = max(hi - kKeys, -kKeys);
            if (k == 0) decode_next();
        const bool okw = __all_sync(0xffffffffu, mbar_wait(&s_full[gt & 1], (gt >> 1) & 1));
            tc::fence_after_sync();
            const bool whole = __all_sync(0xffffffffu, c_lo == 0 && c_hi == kHalfKeys);

            // Fast path (a plain, fully visible tile of rows that have a reference already):
            // P against the running reference m_run in the same pass as the tile maximum.
            // Otherwise pass 1 finds the maximum first (capped or biased logits are written
            // back transformed, invisible columns as -inf).
            const bool fast = okw && plain && whole && __all_sync(0xffffffffu, m_run > -INFINITY);
            float mt = -INFINITY, lt = 0.f;
            if (fast) {
              lt = tile_p<false, true>(ts, tpk, 0, kHalfKeys, p.qscale, m_run, &mt);
              mt *= p.qscale;  // qscale > 0: max commutes with the scale
            } else if (okw && plain) {
              mt = (whole ? tile_max<false>(ts, c_lo, c_hi) : tile_max<true>(ts, c_lo, c_hi)) * p.qscale;
            } else if (okw) {
              float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      #pragma unroll
              for (int c32 = 0; c32 < kHalfKeys / 32; ++c32) {
                float v[32];
                tc::tmem_ld32(ts + c32 * 32, v);
                const float *brow = bias_row ? bias_row + key0(x, x.t_begin + k) + hf * kHalfKeys + c32 * 32 : nullptr;
      #pragma unroll
                for (int c = 0; c < 32; ++c) {
                  const int col = c32 * 32 + c;
                  const bool vis = col >= c_lo && col < c_hi;
                  float xv = v[c] * p.qscale;
                  if (p.capmul != 0.f) xv = p.capmul * fast_tanh(xv);
                  if (vis && brow) xv = fmaf(p.biasmul, brow[c], xv);
                  v[c] = vis ? xv : -INFINITY;
                  mx[c & 3] = fmaxf(mx[c & 3], v[c]);
                }
                tc::tmem_st32(ts + c32 * 32, v);
              }
              mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            }

            // Exchange with the partner half (slot k & 1: the partner has read slot k & 1 of
            // tile k - 2 before it reached the barrier of tile k - 1).  The pair takes the
            // careful path when either half did not take the fast one or saw a logit more than
            // 2^16 above the reference; an expired wait on either side ends both loops.
            xch[gt & 1][hf][r] = mt;
            if (lane == 0) xok[gt & 1][hf][wq] = okw;
            const bool careful = named_barrier_or(bar_pair, 64, !fast || mt > m_run + kDangerLog2);
            if (!okw || !xok[gt & 1][hf ^ 1][wq]) {
              flag(p, GQAW_DEV_TIMEOUT);
              s_abort = 1;
              break;
            }
            mt = fmaxf(mt, xch[gt & 1][hf ^ 1][r]);

            // lazy rescale: the reference moves only when exceeded by more than 2^8 (both halves
            // decide alike).  Careful path: O is rescaled now (with what it owes) and P is
            // computed against the new reference.  Fast path: P(k) already used the old one, so
            // the sum is rescaled after adding it and O owes the factor after O += P(k) V(k).
            const bool need = mt > m_run + kRescaleLog2;
            float alpha = 1.f;
            if (need) {
              alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mt);
              m_run = mt;
            }
            const float oscale = careful ? pend * alpha : pend;
            if (k > 0 && __any_sync(0xffffffffu, oscale != 1.f)) {
              const bool okp = __all_sync(0xffffffffu, mbar_wait(&pv_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1));
              if (named_barrier_or(bar_pair, 64, !okp)) {
                flag(p, GQAW_DEV_TIMEOUT);
                s_abort = 1;
                break;
              }
              tc::fence_after_sync();
      #pragma unroll
              for (int c32 = 0; c32 < kHalfKeys / 32; ++c32) {
                float v[32];
                tc::tmem_ld32(to + c32 * 32, v);
      #pragma unroll
                for (int c = 0; c < 32; ++c) v[c] *= oscale;
                tc::tmem_st32(to + c32 * 32, v);
              }
            }
            if (careful) {
              // ---- pass 2: P = 2^(z - m) (plain logits are still unscaled)
              const float base = m_run == -INFINITY ? 0.f : m_run;
              const float zs = plain ? p.qscale : 1.f;
              l_run = l_run * alpha + (plain && !whole ? tile_p<true>(ts, tpk, c_lo, c_hi, zs, base)
                                                       : tile_p<false>(ts, tpk, c_lo, c_hi, zs, base));
              pend = 1.f;
            } else {
              l_run = (l_run + lt) * alpha;
              pend = alpha;
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[gt & 1]);
            ++done;
          }
          // the last O += P V; the row sum from both halves; what O still owes joins the
          // final scale (the epilogue multiplies O by pend)
          const bool okf = done == x.ntl && __all_sync(0xffffffffu, mbar_wait(&pv_done[(gk + x.ntl - 1) & 1], ((gk + x.ntl - 1) >> 1) & 1));
          xch[2][hf][r] = l_run;
          if (named_barrier_or(bar_pair, 64, !okf)) {
            flag(p, GQAW_DEV_TIMEOUT);
            done = 0;
          }
          l_run += xch[2][hf ^ 1][r];
          o_owed = pend;
          tc::fence_after_sync();
      }

      // ---- epilogue of the unit: O leaves tensor memory first (then the next unit's
      // first O += P V may overwrite it), then this half's 64 columns of (O, m, l) go out
      const bool have_o = x.ntl > 0 && done == x.ntl;
      float o0[32], o1[32];
      if (have_o) {
        tc::tmem_ld32(to, o0);
        tc::tmem_ld32(to + 32, o1);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o0[c] = o1[c] = 0.f;
      }
      if (x.ntl > 0) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
      }
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
      const long long orow = ((long long)x.b * p.S + tok) * p.Nq + h;
      if (ta.nsplit == 1) {
        if (row_ok) {
          const float inv = sink_reciprocal(l_run, m_run, sink_log2(p, h)) * o_owed;
#pragma unroll
          for (int c32 = 0; c32 < 2; ++c32) {
            const float *v = c32 ? o1 : o0;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 w;
              w.x = tc::pack_bf16x2(v[c] * inv, v[c + 1] * inv);
              w.y = tc::pack_bf16x2(v[c + 2] * inv, v[c + 3] * inv);
              w.z = tc::pack_bf16x2(v[c + 4] * inv, v[c + 5] * inv);
              w.w = tc::pack_bf16x2(v[c + 6] * inv, v[c + 7] * inv);
              *reinterpret_cast<uint4 *>(out + orow * kD + hf * kHalfKeys + c32 * 32 + c) = w;
            }
          }
        }
      } else {
        // Partial block of a unit: 33 float4 columns x 128 rows, column-major so that a
        // warp's 32 rows are contiguous; columns 0-31 hold O, column 32 holds (m, l).
        float4 *const part = reinterpret_cast<float4 *>(p.partials);
        auto part_at = [&](long long unit, int c4) { return part + (unit * (kTcPartialStride / 4) + c4) * kRows + r; };
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          const float *v = c32 ? o1 : o0;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *part_at(u, hf * 16 + c32 * 8 + j) =
                make_float4(v[4 * j] * o_owed, v[4 * j + 1] * o_owed, v[4 * j + 2] * o_owed, v[4 * j + 3] * o_owed);
        }
        if (hf == 0) *part_at(u, kD / 4) = make_float4(m_run, l_run, 0.f, 0.f);
        // the last split of the query tile to finish merges them (a barrier of the
        // softmax warps: the other roles run ahead on their own units)
        named_barrier(kSoftmaxBar, 256);
        if (tid == 0) {
          __threadfence();
          s_last = x.ok && atomicAdd(&p.tickets[x.id], 1u) == (unsigned)ta.nsplit - 1u;
        }
        named_barrier(kSoftmaxBar, 256);
        if (s_last) {
          __threadfence();
          if (row_ok) {
            const long long first = u - x.sp;  // split 0 of this query tile
            const int ns = ta.nsplit < 16 ? ta.nsplit : 16;
            float mq[16], f[16];
            float M = -INFINITY, L = 0.f;
            for (int q = 0; q < ns; ++q) {
              const float4 ml = __ldcg(part_at(first + q, kD / 4));
              mq[q] = ml.x;
              f[q] = ml.y;  // l for now
              M = fmaxf(M, ml.x);
            }
            const float mb = M == -INFINITY ? 0.f : M;
            for (int q = 0; q < ns; ++q) {
              const float w = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - mb);
              L += w * f[q];
              f[q] = w;
            }
            const float inv = sink_reciprocal(L, mb, sink_log2(p, h));
#pragma unroll 1
            for (int c32 = 2 * hf; c32 < 2 * hf + 2; ++c32) {  // this half's output columns
              float acc[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) acc[c] = 0.f;
              for (int q = 0; q < ns; ++q) {
                if (f[q] == 0.f) continue;
                float4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = __ldcg(part_at(first + q, c32 * 8 + j));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  acc[4 * j] = fmaf(f[q], v[j].x, acc[4 * j]);
                  acc[4 * j + 1] = fmaf(f[q], v[j].y, acc[4 * j + 1]);
                  acc[4 * j + 2] = fmaf(f[q], v[j].z, acc[4 * j + 2]);
                  acc[4 * j + 3] = fmaf(f[q], v[j].w, acc[4 * j + 3]);
                }
              }
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint4 w;
                w.x = tc::pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
                w.y = tc::pack_bf16x2(acc[c + 2] * inv, acc[c + 3] * inv);
                w.z = tc::pack_bf16x2(acc[c + 4] * inv, acc[c + 5] * inv);
                w.w = tc::pack_bf16x2(acc[c + 6] * inv, acc[c + 7] * inv);
                *reinterpret_cast<uint4 *>(out + orow * kD + c32 * 32 + c) = w;
              }
            }
          }
          if (tid == 0) p.tickets[x.id] = 0u;
        }
      }
      gk += x.ntl;
      decode_next();
      x = nx;
    }
  }

  // release tensor memory (all tcgen05 work of this CTA is complete)
  tc::fence_before_sync();
  __syncthreads();
  pdl_launch_dependents();  // this CTA's work is done: the cache-update kernel may be launched
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

int mma_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_mma(const Params &p, const TcArgs &ta, const TcMaps &maps, int grid, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  static int sms_cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(mma_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) {
      sms_cache[dev] = sms;
      attr_done[dev] = true;
    } else if (grid > sms) {
      grid = sms;
    }
  }
  // persistent: at most one CTA per SM, each walking the units grid-strided
  if (dev < 64 && grid > sms_cache[dev]) grid = sms_cache[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mma_attend_kernel, p, ta, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqaw
