// gqaw_attend.cuh -- windowed GQA attention over the pre-step cache (persistent, stream-K).
//
// What it computes: for one batch item b, one new token s (absolute position
// i = P + s) and a block of query heads of one kv head (a "unit"), the softmax attention
// over the visible keys i - W < j <= i (onnxruntime PR #34226 "Fix CPU Attention causal
// mask for q_len=1 with past_key and kv_len > 1", Description: j <= i + past_len; local
// window of W keys).  Keys older than P are past cache rows (row j - P + L(P), PR
// #32419 row layout); keys from P on are the new input rows, read in place: no staging
// copy is needed because this kernel runs before any row of the cache moves.
//
// Design (GB300; decode is HBM bound: the K/V window is read once):
//  * Persistent stream-K: the step's work is the sequence of (unit, key tile) pairs,
//    TPU tiles per unit; each of the G resident CTAs (2 per SM) takes one contiguous
//    range of it, so every CTA streams the same number of tiles and the TMA pipeline
//    runs on across unit boundaries.  A unit cut by a range boundary is finished by
//    its last contributor (ticket), which merges the contributors' partial softmax
//    states with log-sum-exp weights; every other unit is written directly.
//  * All query heads of a unit share every K/V tile the CTA stages (GQA sharing).
//  * Thread 0 streams K and V tiles into shared memory with bulk TMA copies
//    (cp.async.bulk, L2 evict-first) through an NST-stage mbarrier ring; the cache
//    rows of a tile are contiguous in the BNSH layout, so a tile is one copy per
//    tensor, plus one copy per new row.
//  * A "row group" of LPR lanes owns one key row at a time, each lane a slice of DPL
//    head dimensions (16-byte vectors interleaved so every quarter-warp reads 128
//    contiguous bytes: no shared-memory bank conflicts).  Dot products use packed
//    fp32 FMA (two lanes of math per instruction); 64-row tiles give every warp four
//    independent rows per tile to interleave.
//  * The partial dot products of the GB heads are reduce-scattered across the group
//    with xor shuffles: after log2 steps every lane owns the complete logit of OWN
//    heads, so softcap, bias, the running max and exp2 are evaluated once per head,
//    not once per lane; the probabilities are then broadcast back for P.V.
//  * Online softmax in log2 units with lazy rescaling: the reference max only moves
//    when a logit exceeds it by more than 8 (a factor 256).
//  * Step bookkeeping folded in: the CTA holding a unit's first tile records L(T) and
//    registers items that need the cache-update kernel; the CTA holding a unit's last
//    tile appends the new row of items that reclaim nothing (row L(P) + s, never read
//    by this step).
#pragma once

#include "gqaw_internal.cuh"

namespace gqaw {

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

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
  static constexpr int kPairs = kDPL / 2;            // float2 pairs per lane
  static constexpr int kRPW = 32 / kLPR;             // rows per warp pass
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTile0 = 16384 / kRowBytes;
  static constexpr int kTile = kTile0 < 8 ? 8 : (kTile0 > 64 ? 64 : kTile0);
  static constexpr int kPasses = (kTile + kWarps * kRPW - 1) / (kWarps * kRPW);
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = 2 * kTile * kRowBytes;
  static constexpr int kMergeBytes = kWarps * GB * (D + 2) * 4;
  static constexpr int kSmem = kStages * kStageBytes + kMergeBytes + 2 * kStages * 8;
  // reduce-scatter of GB logits over LPR lanes
  static constexpr int kHalvings = ilog2(GB) < ilog2(kLPR) ? ilog2(GB) : ilog2(kLPR);
  static constexpr int kOwn = GB >> kHalvings;       // heads whose logit a lane owns
  static_assert(kNV * 16 == kRowBytes, "row must be whole 16-byte vectors");
  static_assert((kLPR & (kLPR - 1)) == 0 && kLPR <= 32, "lanes per row: power of two <= 32");
};

// Lazy rescale threshold (log2 units): probabilities stay below 2^8 between rescales.
constexpr float kRescaleThreshold = 8.0f;

// A unit: (item, new token, kv head, query-head block) and its visible key range.
struct Unit {
  int b, s, kvh, hb;
  bool ok;          // the item's seqlens_k is valid
  Plan pl;
  long long lo, hi;  // visible keys [lo, hi), hi = i + 1
  int ntiles;        // tiles holding visible keys
};

__device__ __forceinline__ Unit unit_at(const Params &p, long long u, int tile) {
  Unit x;
  long long r = u;
  x.hb = (int)(r % p.headblocks);
  r /= p.headblocks;
  x.kvh = (int)(r % p.Nkv);
  r /= p.Nkv;
  x.s = (int)(r % p.S);
  x.b = (int)(r / p.S);
  x.ok = plan_item(p, x.b, x.pl);
  x.lo = x.hi = 0;
  x.ntiles = 0;
  if (x.ok) {
    const long long i = x.pl.P + x.s;
    x.lo = i - p.W + 1 > 0 ? i - p.W + 1 : 0;
    x.hi = i + 1;
    x.ntiles = (int)((x.hi - x.lo + tile - 1) / tile);
  }
  return x;
}

// The CTA whose tile range holds virtual tile x: CTA c covers [c*V/G, (c+1)*V/G).
__device__ __forceinline__ long long cta_of_tile(long long x, long long V, long long G) {
  return ((x + 1) * G - 1) / V;
}

// T: query and output elements; TC: cache elements (T itself, or 1-byte codes of a
// quantized cache, scaled by *p.ks and *p.vs).
template <typename T, typename TC, int D, int GB>
__global__ void __launch_bounds__(AttendCfg<TC, D, GB>::kThreads, 2)
    attend_kernel(const Params p) {
  using Cfg = AttendCfg<TC, D, GB>;
  constexpr int EPV = Cfg::kEPV, VPL = Cfg::kVPL, LPR = Cfg::kLPR;
  constexpr int PAIRS = Cfg::kPairs, PPV = EPV / 2;  // pairs per vector
  constexpr int RPW = Cfg::kRPW, NW = Cfg::kWarps, TILE = Cfg::kTile, NST = Cfg::kStages;
  constexpr int ROWB = Cfg::kRowBytes, PASSES = Cfg::kPasses;
  constexpr int HALV = Cfg::kHalvings, OWN = Cfg::kOwn;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stage_base = smem;
  float *merge = reinterpret_cast<float *>(smem + NST * Cfg::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NST * Cfg::kStageBytes + Cfg::kMergeBytes);
  uint64_t *empty = full + NST;
  __shared__ int s_last;

  const long long TPU = p.tpu;
  const long long V = p.nunits * TPU;
  const long long G = gridDim.x;
  const long long cta = blockIdx.x;
  const long long tb = cta * V / G, te = (cta + 1) * V / G;  // this CTA's virtual tiles
  if (tb >= te) {
    pdl_wait();
    pdl_launch_dependents();
    return;
  }
  const long long ufirst = tb / TPU, ulast = (te - 1) / TPU;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], NW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();                // the previous kernel (a cache update) has finished

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // quantized cache: codes times the per-tensor scales (key scale folded into q)
  const float qscale = p.ks ? p.qscale * *p.ks : p.qscale;
  const float vscale = p.vs ? *p.vs : 1.f;

  // ---------------------------------------------------------------- producer state
  // Thread 0 walks the same (unit, tile) sequence as the consumers, NST - 1 tiles
  // ahead, skipping tiles past a unit's visible keys.
  Unit pu_x;
  long long pu = ufirst;
  int plt = 0, preal = 0;
  int issued = 0;
  bool pdone = false, alive = true;
  uint64_t pol = 0;
  if (threadIdx.x == 0) {
    pol = policy_evict_first();
    pu_x = unit_at(p, pu, TILE);
    plt = (int)(tb - pu * TPU);
    const long long e = te - pu * TPU < TPU ? te - pu * TPU : TPU;
    preal = (int)(e < pu_x.ntiles ? e : pu_x.ntiles);
  }
  // Issue the next tile of the sequence; false when the CTA's range is exhausted.
  auto issue_next = [&]() -> bool {
    while (plt >= preal) {
      ++pu;
      if (pu > ulast) {
        pdone = true;
        return false;
      }
      pu_x = unit_at(p, pu, TILE);
      plt = 0;
      const long long e = te - pu * TPU < TPU ? te - pu * TPU : TPU;
      preal = (int)(e < pu_x.ntiles ? e : pu_x.ntiles);
    }
    const int st = issued % NST;
    if (issued >= NST && !mbar_wait(&empty[st], ((issued / NST) - 1) & 1)) {
      flag(p, GQAW_DEV_TIMEOUT);
      alive = false;
      return false;
    }
    const long long j0 = pu_x.lo + (long long)plt * TILE;
    const long long j1 = j0 + TILE < pu_x.hi ? j0 + TILE : pu_x.hi;
    const size_t slice = ((size_t)pu_x.b * p.Nkv + pu_x.kvh) * (size_t)p.C;
    const TC *pk = static_cast<const TC *>(p.pk) + slice * D;
    const TC *pv = static_cast<const TC *>(p.pv) + slice * D;
    unsigned char *ks = stage_base + st * Cfg::kStageBytes;
    unsigned char *vs = ks + TILE * ROWB;
    mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * (j1 - j0) * ROWB));
    const long long jc1 = j1 < pu_x.pl.P ? j1 : pu_x.pl.P;  // cache rows: keys before P
    if (j0 < jc1) {
      const long long r = j0 - pu_x.pl.P + pu_x.pl.Lp;
      const uint32_t bytes = (uint32_t)((jc1 - j0) * ROWB);
      bulk_g2s(ks, pk + r * D, bytes, &full[st], pol);
      bulk_g2s(vs, pv + r * D, bytes, &full[st], pol);
    }
    for (long long j = (j0 > pu_x.pl.P ? j0 : pu_x.pl.P); j < j1; ++j) {  // new rows: keys from P
      const size_t off = (((size_t)pu_x.b * p.S + (size_t)(j - pu_x.pl.P)) * p.Nkv + pu_x.kvh) * D;
      bulk_g2s(ks + (j - j0) * ROWB, static_cast<const TC *>(p.k) + off, ROWB, &full[st], pol);
      bulk_g2s(vs + (j - j0) * ROWB, static_cast<const TC *>(p.v) + off, ROWB, &full[st], pol);
    }
    ++plt;
    ++issued;
    return true;
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < NST - 1 && !pdone && alive; ++k) issue_next();

  // ---------------------------------------------------------------- consumer lanes
  const int gi = lane / LPR, li = lane % LPR;
  const int gbase = gi * LPR;  // first lane of this row group
  // heads whose logits this lane owns after the reduce-scatter: [own0, own0 + OWN)
  int own0 = 0;
#pragma unroll
  for (int k = 0; k < HALV; ++k)
    if (li & (LPR >> (k + 1))) own0 += GB >> (k + 1);
  // lane owning head h's logit
  auto owner = [&](int h) {
    int src = 0;
    const int hq = h / OWN;
#pragma unroll
    for (int k = 0; k < HALV; ++k)
      if (hq & (1 << (HALV - 1 - k))) src += LPR >> (k + 1);
    return gbase + src;
  };

  int k = 0;  // tiles consumed by this CTA
  for (long long u = ufirst; u <= ulast; ++u) {
    const Unit x = unit_at(p, u, TILE);
    const int lt0 = u == ufirst ? (int)(tb - u * TPU) : 0;
    const int lt1 = (int)(te - u * TPU < TPU ? te - u * TPU : TPU);
    const int real1 = lt1 < x.ntiles ? lt1 : x.ntiles;
    if (!x.ok) {  // every CTA touching the unit skips it: no ticket, no output
      if (lt0 == 0 && x.s == 0 && x.kvh == 0 && x.hb == 0 && threadIdx.x == 0) flag(p, GQAW_DEV_BAD_SEQLEN);
      continue;
    }
    const int head_in_group0 = x.hb * GB;
    const int nheads = p.group - head_in_group0 < GB ? p.group - head_in_group0 : GB;
    const int hq0 = x.kvh * p.group + head_in_group0;                      // first query head
    const long long orow0 = ((long long)x.b * p.S + x.s) * p.Nq + hq0;     // its output row
    const bool moves = item_moves(p, x.pl);

    if (lt0 == 0 && x.s == 0 && x.kvh == 0 && x.hb == 0 && threadIdx.x == 0) {
      if (p.resident_out) p.resident_out[x.b] = (int32_t)x.pl.Lt;
      if (moves) p.move_list[atomicAdd(p.move_count, 1u)] = x.b;
    }
    if (!moves && x.hb == 0 && x.ntiles - 1 >= lt0 && x.ntiles - 1 < lt1) {
      // append new row s at row L(P) + s: no query of this step reads it
      const size_t slice_row = ((size_t)x.b * p.Nkv + x.kvh) * (size_t)p.C + (size_t)(x.pl.Lp + x.s);
      const size_t in_row = ((size_t)x.b * p.S + x.s) * p.Nkv + x.kvh;
      for (int e = threadIdx.x; e < 2 * (ROWB / 16); e += blockDim.x) {
        const int tensor = e / (ROWB / 16), vec = e % (ROWB / 16);
        const uint4 *srcv =
            reinterpret_cast<const uint4 *>(static_cast<const char *>(tensor ? p.v : p.k) + in_row * ROWB);
        uint4 *dstv = reinterpret_cast<uint4 *>(static_cast<char *>(tensor ? p.prv : p.prk) + slice_row * ROWB);
        dstv[vec] = srcv[vec];
      }
    }

    float2 q2[GB][PAIRS];
    {
      // the lane's EPV query dims per cache vector take QV 16-byte vectors of T (one
      // when T is the cache type); a quantized cache's key scale is folded in here
      constexpr int PPT = 8 / (int)sizeof(T), QV = PPV / PPT;
      const T *qin = static_cast<const T *>(p.q);
#pragma unroll
      for (int r = 0; r < GB; ++r) {
        const bool ok = r < nheads;
        const T *qrow = qin + (orow0 + (ok ? r : 0)) * D;
#pragma unroll
        for (int m = 0; m < VPL; ++m) {
#pragma unroll
          for (int qv = 0; qv < QV; ++qv) {
            const uint4 uq = *reinterpret_cast<const uint4 *>(qrow + (li + LPR * m) * EPV + qv * 2 * PPT);
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
              const float2 f = Pairs<T>::get(uq, j);
              q2[r][m * PPV + qv * PPT + j] = ok ? make_float2(f.x * qscale, f.y * qscale) : make_float2(0.f, 0.f);
            }
          }
        }
      }
    }
    float2 acc2[GB][PAIRS];
#pragma unroll
    for (int r = 0; r < GB; ++r)
#pragma unroll
      for (int d = 0; d < PAIRS; ++d) acc2[r][d] = make_float2(0.f, 0.f);
    float m_own[OWN], l_own[OWN];
#pragma unroll
    for (int o = 0; o < OWN; ++o) {
      m_own[o] = -INFINITY;
      l_own[o] = 0.f;
    }
    const float *bias_bs = p.bias ? p.bias + x.b * p.bsb + x.s * p.bss : nullptr;

    for (int lt = lt0; lt < real1; ++lt, ++k) {
      if (threadIdx.x == 0 && !pdone && alive) issue_next();
      const int st = k % NST;
      if (!mbar_wait(&full[st], (k / NST) & 1)) {
        if (lane == 0) flag(p, GQAW_DEV_TIMEOUT);
        break;
      }
      const long long j0 = x.lo + (long long)lt * TILE;
      const long long j1 = j0 + TILE < x.hi ? j0 + TILE : x.hi;
      const int n = (int)(j1 - j0);
      const unsigned char *ks = stage_base + st * Cfg::kStageBytes;
      const unsigned char *vs = ks + TILE * ROWB;

      // ---- logits: packed FMA over the lane's dims, reduce-scatter over the group
      float so[PASSES][OWN];
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = ps * NW * RPW + warp * RPW + gi;
        const bool valid = r < n;
        float2 part2[GB];
#pragma unroll
        for (int h = 0; h < GB; ++h) part2[h] = make_float2(0.f, 0.f);
        if (valid) {
#pragma unroll
          for (int m = 0; m < VPL; ++m) {
            const uint4 uk = *reinterpret_cast<const uint4 *>(ks + r * ROWB + (li + LPR * m) * 16);
#pragma unroll
            for (int j = 0; j < PPV; ++j) {
              const float2 k2 = Pairs<TC>::get(uk, j);
#pragma unroll
              for (int h = 0; h < GB; ++h) part2[h] = __ffma2_rn(q2[h][m * PPV + j], k2, part2[h]);
            }
          }
        }
        float v[GB];
#pragma unroll
        for (int h = 0; h < GB; ++h) v[h] = part2[h].x + part2[h].y;
        // halving steps: keep one half of the values, send the other half
#pragma unroll
        for (int hs = 0, nv = GB; hs < HALV; ++hs) {
          const int off = LPR >> (hs + 1);
          const bool upper = (li & off) != 0;
          nv >>= 1;
#pragma unroll
          for (int xx = 0; xx < GB / 2; ++xx) {
            if (xx < nv) {
              const float send = upper ? v[xx] : v[nv + xx];
              const float keep = upper ? v[nv + xx] : v[xx];
              v[xx] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
          }
        }
        // remaining lanes of the group: plain xor sums
#pragma unroll
        for (int off = (LPR >> (HALV + 1)); off >= 1; off >>= 1)
#pragma unroll
          for (int o = 0; o < OWN; ++o) v[o] += __shfl_xor_sync(0xffffffffu, v[o], off);
#pragma unroll
        for (int o = 0; o < OWN; ++o) {
          float z = v[o];
          if (p.capmul != 0.f) z = p.capmul * tanhf(z);
          if (valid && bias_bs && own0 + o < nheads)
            z += p.biasmul * bias_bs[(long long)(hq0 + own0 + o) * p.bsh + j0 + r];
          so[ps][o] = valid ? z : -INFINITY;
        }
      }

      // ---- online softmax of the owned heads, lazy rescaling
      bool need = false;
      float mt[OWN];
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        mt[o] = so[0][o];
#pragma unroll
        for (int ps = 1; ps < PASSES; ++ps) mt[o] = fmaxf(mt[o], so[ps][o]);
        need |= mt[o] > m_own[o] + kRescaleThreshold;
      }
      if (__any_sync(0xffffffffu, need)) {
        float a_own[OWN];
#pragma unroll
        for (int o = 0; o < OWN; ++o) {
          const float mn = mt[o] > m_own[o] + kRescaleThreshold ? mt[o] : m_own[o];
          a_own[o] = mn == -INFINITY ? 1.f : exp2f(m_own[o] - mn);
          l_own[o] *= a_own[o];
          m_own[o] = mn;
        }
#pragma unroll
        for (int h = 0; h < GB; ++h) {
          const float a = __shfl_sync(0xffffffffu, a_own[h % OWN], owner(h));
          const float2 a2 = make_float2(a, a);
#pragma unroll
          for (int d = 0; d < PAIRS; ++d) acc2[h][d] = __fmul2_rn(acc2[h][d], a2);
        }
      }
      float pw[PASSES][GB];
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        float po[OWN];
#pragma unroll
        for (int o = 0; o < OWN; ++o) {
          const float base = m_own[o] == -INFINITY ? 0.f : m_own[o];
          po[o] = exp2f(so[ps][o] - base);
          l_own[o] += po[o];
        }
#pragma unroll
        for (int h = 0; h < GB; ++h) pw[ps][h] = __shfl_sync(0xffffffffu, po[h % OWN], owner(h));
      }

      // ---- P.V with packed FMA
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const int r = ps * NW * RPW + warp * RPW + gi;
        if (r < n) {
#pragma unroll
          for (int m = 0; m < VPL; ++m) {
            const uint4 uv = *reinterpret_cast<const uint4 *>(vs + r * ROWB + (li + LPR * m) * 16);
#pragma unroll
            for (int j = 0; j < PPV; ++j) {
              const float2 v2 = Pairs<TC>::get(uv, j);
#pragma unroll
              for (int h = 0; h < GB; ++h)
                acc2[h][m * PPV + j] = __ffma2_rn(make_float2(pw[ps][h], pw[ps][h]), v2, acc2[h][m * PPV + j]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- every lane gets (max, sum) of every head of the block
    float mrun[GB], lrun[GB];
#pragma unroll
    for (int h = 0; h < GB; ++h) {
      mrun[h] = __shfl_sync(0xffffffffu, m_own[h % OWN], owner(h));
      lrun[h] = __shfl_sync(0xffffffffu, l_own[h % OWN], owner(h));
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
        for (int d = 0; d < PAIRS; ++d) {
          const float ax = __shfl_xor_sync(0xffffffffu, acc2[h][d].x, off);
          const float ay = __shfl_xor_sync(0xffffffffu, acc2[h][d].y, off);
          acc2[h][d] = make_float2(acc2[h][d].x * fa + ax * fb, acc2[h][d].y * fa + ay * fb);
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
          for (int j = 0; j < PPV; ++j) {
            row[(li + LPR * m) * EPV + 2 * j] = acc2[h][m * PPV + j].x;
            row[(li + LPR * m) * EPV + 2 * j + 1] = acc2[h][m * PPV + j].y;
          }
        if (li == 0) {
          row[D] = mrun[h];
          row[D + 1] = lrun[h];
        }
      }
    }
    __syncthreads();

    // ---- this CTA's state of the unit; written out, or published as a partial
    const long long cf = cta_of_tile(u * TPU, V, G), cl = cta_of_tile((u + 1) * TPU - 1, V, G);
    const int slot = u == ufirst ? 0 : 1;  // only a CTA's first and last unit can be shared
    T *out = static_cast<T *>(p.out);
    for (int idx = threadIdx.x; idx < nheads * D; idx += NW * 32) {
      const int h = idx / D, d = idx % D;
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
      if (cf == cl) {
        out[(orow0 + h) * D + d] = Elem<T>::store(sink_divide(A, L, base, sink_log2(p, hq0 + h)) * vscale);
      } else {
        float *part = p.partials + ((cta * 2 + slot) * GB + h) * (D + 2);
        part[d] = A;
        if (d == 0) {
          part[D] = M;
          part[D + 1] = L;
        }
      }
    }
    if (cf != cl) {
      // last contributor merges the partials of CTAs cf..cl
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&p.tickets[u], 1u) == (unsigned)(cl - cf);
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int idx = threadIdx.x; idx < nheads * D; idx += NW * 32) {
          const int h = idx / D, d = idx % D;
          float M = -INFINITY;
          for (long long c = cf; c <= cl; ++c) {
            const int sl = u == c * V / G / TPU ? 0 : 1;
            M = fmaxf(M, __ldcg(p.partials + ((c * 2 + sl) * GB + h) * (D + 2) + D));
          }
          const float base = M == -INFINITY ? 0.f : M;
          float L = 0.f, A = 0.f;
          for (long long c = cf; c <= cl; ++c) {
            const int sl = u == c * V / G / TPU ? 0 : 1;
            const float *part = p.partials + ((c * 2 + sl) * GB + h) * (D + 2);
            const float mc = __ldcg(part + D);
            if (mc == -INFINITY) continue;  // contributor held no visible key
            const float f = exp2f(mc - base);
            L = fmaf(f, __ldcg(part + D + 1), L);
            A = fmaf(f, __ldcg(part + d), A);
          }
          out[(orow0 + h) * D + d] = Elem<T>::store(sink_divide(A, L, base, sink_log2(p, hq0 + h)) * vscale);
        }
        if (threadIdx.x == 0) p.tickets[u] = 0u;  // ready for the next step
      }
    }
    __syncthreads();  // the merge area is reused by the next unit
  }

  pdl_launch_dependents();  // this CTA's work is done: the cache-update kernel may be launched
  // Drain: no copy may still be landing in shared memory when the CTA exits.
  if (threadIdx.x == 0)
    for (int u2 = issued - NST > 0 ? issued - NST : 0; u2 < issued; ++u2)
      if (!mbar_wait(&full[u2 % NST], (u2 / NST) & 1)) flag(p, GQAW_DEV_TIMEOUT);
}

}  // namespace gqaw
