// gqaw_attend.cuh -- split-K windowed GQA attention over the pre-step cache.
//
// What it computes: for one batch item b, one new token s (absolute position
// i = P + s) and a block of query heads of one kv head, the softmax attention over the
// visible keys i - W < j <= i (onnxruntime PR #34226 "Fix CPU Attention causal mask
// for q_len=1 with past_key and kv_len > 1", Description: j <= i + past_len; local
// window of W keys), restricted to one chunk of those keys.  Keys older than P are
// past cache rows (row j - P + L(P), PR #32419 row layout); keys from P on are the new
// input rows, read in place: no staging copy is needed because this kernel runs before
// any row of the cache moves (the cache update is a separate, later kernel).
//
// Design (GB300):
//  * One CTA per (item, token, kv head, head block, key chunk).  All query heads of
//    the block share every K/V tile the CTA stages (GQA sharing inside the CTA).
//  * A producer warp streams K and V tiles into shared memory with bulk TMA copies
//    (cp.async.bulk, L2 evict-first) through an NST-stage mbarrier ring; the cache
//    rows of a tile are contiguous in the BNSH layout, so a tile is one copy per
//    tensor, plus one copy per new row.
//  * Four consumer warps: a "row group" of LPR lanes owns one key row at a time, each
//    lane a slice of DPL head dimensions (16-byte vectors interleaved so every
//    quarter-warp reads 128 contiguous bytes: no shared-memory bank conflicts).
//    Logits are reduced across the group with xor shuffles; every group keeps its own
//    online-softmax state (running max in log2 units, sum, accumulator).
//  * The end of the chunk merges group states with shuffles, warp states through
//    shared memory, then writes either the final output (one chunk) or a partial
//    (max, sum, accumulator) for the split combine.
#pragma once

#include "gqaw_internal.cuh"

namespace gqaw {

template <typename T, int D, int GB>
struct AttendCfg {
  static constexpr int kElem = (int)sizeof(T);
  static constexpr int kEPV = 16 / kElem;          // elements per 16-byte vector
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kNV = kRowBytes / 16;         // vectors per row
  static constexpr int kVPL0 = (64 / (GB * kEPV)) > 0 ? (64 / (GB * kEPV)) : 1;
  static constexpr int kVPL1 = kVPL0 < kNV ? kVPL0 : kNV;
  static constexpr int kVPL = (kNV / kVPL1 > 32) ? kNV / 32 : kVPL1;  // vectors per lane
  static constexpr int kLPR = kNV / kVPL;            // lanes per key row
  static constexpr int kDPL = kVPL * kEPV;           // dims per lane
  static constexpr int kRPW = 32 / kLPR;             // rows per warp pass
  static constexpr int kWarps = 4;                   // consumer warps
  static constexpr int kThreads = (kWarps + 1) * 32; // + producer warp
  static constexpr int kTile0 = 8192 / kRowBytes;
  static constexpr int kTile = kTile0 < 8 ? 8 : (kTile0 > 64 ? 64 : kTile0);
  static constexpr int kPasses = (kTile + kWarps * kRPW - 1) / (kWarps * kRPW);
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = 2 * kTile * kRowBytes;
  static constexpr int kMergeBytes = kWarps * GB * (D + 2) * 4;
  static constexpr int kSmem = kStages * kStageBytes + kMergeBytes + 2 * kStages * 8;
  static_assert(kNV * 16 == kRowBytes, "row must be whole 16-byte vectors");
  static_assert((kLPR & (kLPR - 1)) == 0 && kLPR <= 32, "lanes per row: power of two <= 32");
};

template <typename T, int D, int GB>
__global__ void __launch_bounds__(AttendCfg<T, D, GB>::kThreads)
    attend_kernel(const Params p) {
  using Cfg = AttendCfg<T, D, GB>;
  constexpr int EPV = Cfg::kEPV, VPL = Cfg::kVPL, LPR = Cfg::kLPR, DPL = Cfg::kDPL;
  constexpr int RPW = Cfg::kRPW, NW = Cfg::kWarps, TILE = Cfg::kTile, NST = Cfg::kStages;
  constexpr int ROWB = Cfg::kRowBytes, PASSES = Cfg::kPasses;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stage_base = smem;
  float *merge = reinterpret_cast<float *>(smem + NST * Cfg::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NST * Cfg::kStageBytes + Cfg::kMergeBytes);
  uint64_t *empty = full + NST;

  // ---- which work unit
  const int split = blockIdx.x % p.nsplit;
  int unit = blockIdx.x / p.nsplit;
  const int hb = unit % p.headblocks;
  unit /= p.headblocks;
  const int kvh = unit % p.Nkv;
  unit /= p.Nkv;
  const int s = unit % p.S;
  const int b = unit / p.S;

  Plan pl;
  if (!plan_item(p, b, pl)) {
    if (threadIdx.x == 0) flag(p, GQAW_DEV_BAD_SEQLEN);
    return;
  }
  const long long i = pl.P + s;                       // absolute query position
  const long long lo = i - p.W + 1 > 0 ? i - p.W + 1 : 0;
  const long long c0 = lo + (long long)split * p.chunk;
  const long long c1 = c0 + p.chunk < i + 1 ? c0 + p.chunk : i + 1;
  const int head_in_group0 = hb * GB;
  const long long row0 = ((long long)b * p.S + s) * p.Nq;  // first output row of (b, s)

  if (c0 >= c1) {  // empty chunk (short item): an empty partial
    if (threadIdx.x < GB && head_in_group0 + (int)threadIdx.x < p.group) {
      const long long r = row0 + (long long)kvh * p.group + head_in_group0 + threadIdx.x;
      p.ws_m[r * p.nsplit + split] = -INFINITY;
      p.ws_l[r * p.nsplit + split] = 0.f;
    }
    return;
  }
  const int ntiles = (int)((c1 - c0 + TILE - 1) / TILE);

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], NW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T *kin = static_cast<const T *>(p.k);
  const T *vin = static_cast<const T *>(p.v);
  const size_t slice = ((size_t)b * p.Nkv + kvh) * (size_t)p.C;

  if (warp == NW) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const T *pk = static_cast<const T *>(p.pk) + slice * D;
      const T *pv = static_cast<const T *>(p.pv) + slice * D;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % NST;
        if (t >= NST && !mbar_wait(&empty[st], ((t / NST) - 1) & 1)) {
          flag(p, GQAW_DEV_TIMEOUT);
          break;
        }
        const long long j0 = c0 + (long long)t * TILE;
        const long long j1 = j0 + TILE < c1 ? j0 + TILE : c1;
        unsigned char *ks = stage_base + st * Cfg::kStageBytes;
        unsigned char *vs = ks + TILE * ROWB;
        mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * (j1 - j0) * ROWB));
        const long long jc1 = j1 < pl.P ? j1 : pl.P;  // cache rows: keys before P
        if (j0 < jc1) {
          const long long r = j0 - pl.P + pl.Lp;
          const uint32_t bytes = (uint32_t)((jc1 - j0) * ROWB);
          bulk_g2s(ks, pk + r * D, bytes, &full[st], pol);
          bulk_g2s(vs, pv + r * D, bytes, &full[st], pol);
        }
        for (long long j = (j0 > pl.P ? j0 : pl.P); j < j1; ++j) {  // new rows: keys from P
          const size_t off = (((size_t)b * p.S + (size_t)(j - pl.P)) * p.Nkv + kvh) * D;
          bulk_g2s(ks + (j - j0) * ROWB, kin + off, ROWB, &full[st], pol);
          bulk_g2s(vs + (j - j0) * ROWB, vin + off, ROWB, &full[st], pol);
        }
        issued = t + 1;
      }
      // Drain: no copy may still be landing in shared memory when the CTA exits.
      for (int t = issued - NST > 0 ? issued - NST : 0; t < issued; ++t)
        if (!mbar_wait(&full[t % NST], (t / NST) & 1)) flag(p, GQAW_DEV_TIMEOUT);
    }
    return;
  }

  // ================================================================== consumers
  const int gi = lane / LPR, li = lane % LPR;
  float qf[GB][DPL];
  {
    const T *qin = static_cast<const T *>(p.q);
#pragma unroll
    for (int r = 0; r < GB; ++r) {
      const int hg = head_in_group0 + r;
      const bool ok = hg < p.group;
      const T *qrow = qin + (row0 + (long long)kvh * p.group + (ok ? hg : 0)) * D;
#pragma unroll
      for (int m = 0; m < VPL; ++m) {
        const uint4 u = *reinterpret_cast<const uint4 *>(qrow + (li + LPR * m) * EPV);
        float f[EPV];
        Elem<T>::unpack(u, f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) qf[r][m * EPV + e] = ok ? f[e] * p.qscale : 0.f;
      }
    }
  }
  float mrun[GB], lrun[GB], acc[GB][DPL];
#pragma unroll
  for (int r = 0; r < GB; ++r) {
    mrun[r] = -INFINITY;
    lrun[r] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[r][d] = 0.f;
  }
  const float *bias_bs = p.bias ? p.bias + b * p.bsb + s * p.bss : nullptr;
  const int hq0 = kvh * p.group + head_in_group0;  // first query head of this block

  bool alive = true;
  for (int t = 0; t < ntiles && alive; ++t) {
    const int st = t % NST;
    if (!mbar_wait(&full[st], (t / NST) & 1)) {
      if (lane == 0) flag(p, GQAW_DEV_TIMEOUT);
      alive = false;
      break;
    }
    const long long j0 = c0 + (long long)t * TILE;
    const long long j1 = j0 + TILE < c1 ? j0 + TILE : c1;
    const int n = (int)(j1 - j0);
    const unsigned char *ks = stage_base + st * Cfg::kStageBytes;
    const unsigned char *vs = ks + TILE * ROWB;

    float sc[PASSES][GB];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = ps * NW * RPW + warp * RPW + gi;
      const bool valid = r < n;
      float part[GB];
#pragma unroll
      for (int h = 0; h < GB; ++h) part[h] = 0.f;
      if (valid) {
#pragma unroll
        for (int m = 0; m < VPL; ++m) {
          const uint4 u = *reinterpret_cast<const uint4 *>(ks + r * ROWB + (li + LPR * m) * 16);
          float f[EPV];
          Elem<T>::unpack(u, f);
#pragma unroll
          for (int e = 0; e < EPV; ++e)
#pragma unroll
            for (int h = 0; h < GB; ++h) part[h] = fmaf(qf[h][m * EPV + e], f[e], part[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < GB; ++h) {
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
        float z = part[h];
        if (p.capmul != 0.f) z = p.capmul * tanhf(z);
        if (valid && bias_bs && head_in_group0 + h < p.group)
          z += p.biasmul * bias_bs[(long long)(hq0 + h) * p.bsh + j0 + r];
        sc[ps][h] = valid ? z : -INFINITY;
      }
    }
    // online softmax update, once per tile per row group
    float pw[PASSES][GB];
#pragma unroll
    for (int h = 0; h < GB; ++h) {
      float mt = sc[0][h];
#pragma unroll
      for (int ps = 1; ps < PASSES; ++ps) mt = fmaxf(mt, sc[ps][h]);
      const float mnew = fmaxf(mrun[h], mt);
      const float base = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = exp2f(mrun[h] - base);
      lrun[h] *= alpha;
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[h][d] *= alpha;
      mrun[h] = mnew;
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        pw[ps][h] = exp2f(sc[ps][h] - base);
        lrun[h] += pw[ps][h];
      }
    }
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = ps * NW * RPW + warp * RPW + gi;
      if (r < n) {
#pragma unroll
        for (int m = 0; m < VPL; ++m) {
          const uint4 u = *reinterpret_cast<const uint4 *>(vs + r * ROWB + (li + LPR * m) * 16);
          float f[EPV];
          Elem<T>::unpack(u, f);
#pragma unroll
          for (int e = 0; e < EPV; ++e)
#pragma unroll
            for (int h = 0; h < GB; ++h) acc[h][m * EPV + e] = fmaf(pw[ps][h], f[e], acc[h][m * EPV + e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- merge the row groups of this warp (lanes with equal li hold equal dims)
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < GB; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, mrun[h], off);
      const float lo2 = __shfl_xor_sync(0xffffffffu, lrun[h], off);
      const float mn = fmaxf(mrun[h], mo);
      const float base = mn == -INFINITY ? 0.f : mn;
      const float fa = exp2f(mrun[h] - base), fb = exp2f(mo - base);
      lrun[h] = lrun[h] * fa + lo2 * fb;
#pragma unroll
      for (int d = 0; d < DPL; ++d) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[h][d], off);
        acc[h][d] = acc[h][d] * fa + ao * fb;
      }
      mrun[h] = mn;
    }
  }
  // ---- warp states to shared memory: merge[warp][h][0..D) acc, [D] max, [D+1] sum
  if (gi == 0) {
#pragma unroll
    for (int h = 0; h < GB; ++h) {
      float *row = merge + (warp * GB + h) * (D + 2);
#pragma unroll
      for (int m = 0; m < VPL; ++m)
#pragma unroll
        for (int e = 0; e < EPV; ++e) row[(li + LPR * m) * EPV + e] = acc[h][m * EPV + e];
      if (li == 0) {
        row[D] = mrun[h];
        row[D + 1] = lrun[h];
      }
    }
  }
  named_barrier(1, NW * 32);
  T *out = static_cast<T *>(p.out);
  for (int idx = threadIdx.x; idx < GB * D; idx += NW * 32) {
    const int h = idx / D, d = idx % D;
    if (head_in_group0 + h >= p.group) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, merge[(w * GB + h) * (D + 2) + D]);
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float *row = merge + (w * GB + h) * (D + 2);
      const float f = exp2f(row[D] - base);
      L = fmaf(f, row[D + 1], L);
      A = fmaf(f, row[d], A);
    }
    const long long orow = row0 + hq0 + h;
    if (p.nsplit == 1) {
      out[orow * D + d] = Elem<T>::store(A / L);
    } else {
      const long long pr = orow * p.nsplit + split;
      p.ws_acc[pr * D + d] = A;
      if (d == 0) {
        p.ws_m[pr] = M;
        p.ws_l[pr] = L;
      }
    }
  }
}

}  // namespace gqaw
