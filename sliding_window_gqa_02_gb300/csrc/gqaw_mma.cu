// gqaw_mma.cu -- multi-token windowed GQA attention on the 5th-generation tensor cores.
//
// For steps with S > 1 new tokens (speculative verify, chunked prefill) the logits of
// all query heads of a kv group and of many tokens share the same K/V rows, so
// Q.K^T and P.V are genuine dense contractions: they run as tcgen05.mma (bf16
// operands from shared memory, fp32 accumulators in tensor memory).
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
// Tiling: one CTA per (item, kv head, 128-row query tile, key split).  Query rows are
// (token, head) pairs r = t * g + head, so one TMA box brings 128/g tokens x g heads.
// Keys come in tiles of 128: first the cache rows [klo, P), then the new rows
// [P, P + s_end).  Per key tile:
//   S = Q K^T      tcgen05.mma M=128 N=128, K=128 in 8 steps (both operands K-major)
//   softmax        one thread per query row reads its 128 logits from tensor memory
//                  (no shuffles), masks, online max/sum, writes P (bf16) to shared
//                  memory in the 128-byte-swizzled K-major layout
//   O += P V       tcgen05.mma M=128 N=128 (V is the MN-major B operand)
// K/V tiles arrive by TMA (128-byte swizzle) into a two-stage ring; the load of tile
// t + 1 overlaps the softmax and P.V of tile t.
#include <cuda.h>

#include "gqaw_tc.cuh"

namespace gqaw {

namespace {

constexpr int kRows = 128;       // query rows per CTA (M)
constexpr int kKeys = 128;       // keys per tile (N of Q.K^T, K of P.V)
constexpr int kD = 128;          // head size
constexpr int kHalf = 16384;     // bytes of a [128 rows][64 bf16] swizzled block
constexpr int kThreads = 128;
// shared memory: Q, two K buffers, two V buffers, P -- each two 64-column halves
constexpr int kSmemQ = 0;
constexpr int kSmemK = 2 * kHalf;
constexpr int kSmemV = kSmemK + 4 * kHalf;
constexpr int kSmemP = kSmemV + 4 * kHalf;
constexpr int kSmemBars = kSmemP + 2 * kHalf;
constexpr int kSmemTotal = kSmemBars + 256;
constexpr int kSmemAlloc = kSmemTotal + 1024;  // room to align the base to 1024 bytes
constexpr uint32_t kTmemCols = 512;            // S: two buffers, columns [0,256); O: [256,384)
constexpr float kRescaleLog2 = 8.0f;           // lazy rescale threshold (log2 units)

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

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    mma_attend_kernel(const Params p, const TcArgs ta, const __grid_constant__ TcMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + kSmemBars);  // [2]: K tile landed
  uint64_t *vfull = kfull + 2;                                        // [2]: V tile landed
  uint64_t *bar_q = vfull + 2;
  uint64_t *bar_s = bar_q + 1;  // [2]: S = Q K^T done, per tensor-memory buffer
  uint64_t *bar_o = bar_s + 2;  // O += P V done
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_o + 1);
  __shared__ int s_last, s_abort;

  const int tid = threadIdx.x, warp = tid >> 5;
  int x = blockIdx.x;
  const int sp = x % ta.nsplit;
  x /= ta.nsplit;
  const int rt = x % ta.rowtiles;
  x /= ta.rowtiles;
  const int kvh = x % p.Nkv;
  const int b = x / p.Nkv;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&bar_s[i], 1);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_o, 1);
    mbar_fence_init();
    s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 2 * kKeys;
  pdl_wait();

  Plan pl;
  const bool ok = plan_item(p, b, pl);
  const int g = p.group;
  const int s0 = rt * ta.tokens_per_tile;
  const int s_end = s0 + ta.tokens_per_tile < p.S ? s0 + ta.tokens_per_tile : p.S;
  const long long unit_tile = ((long long)b * p.Nkv + kvh) * ta.rowtiles + rt;

  // key tiles of this query tile: cache rows [klo, P), then new rows [P, P + s_end)
  long long klo = 0, P = 0;
  int nc = 0, ni = 0, t_begin = 0, t_end = 0;
  bool moves = false;
  if (ok) {
    P = pl.P;
    klo = P + s0 - p.W + 1 > 0 ? P + s0 - p.W + 1 : 0;
    nc = (int)((P - klo + kKeys - 1) / kKeys);
    ni = (int)((s_end + kKeys - 1) / kKeys);
    const int nt = nc + ni;
    t_begin = (int)((long long)sp * nt / ta.nsplit);
    t_end = (int)((long long)(sp + 1) * nt / ta.nsplit);
    moves = item_moves(p, pl);
    if (kvh == 0 && rt == 0 && sp == 0 && tid == 0) {
      if (p.resident_out) p.resident_out[b] = (int32_t)pl.Lt;
      if (moves) p.move_list[atomicAdd(p.move_count, 1u)] = b;
    }
    if (!moves && sp == 0) {  // append the new rows of this query tile's tokens at L(P) + s
      const int per_row = kD * 2 / 16;
      const int n = 2 * (s_end - s0) * per_row;
      for (int e = tid; e < n; e += kThreads) {
        const int tensor = e / ((s_end - s0) * per_row);
        const int rem = e % ((s_end - s0) * per_row);
        const int s = s0 + rem / per_row, vec = rem % per_row;
        const size_t in_row = ((size_t)b * p.S + s) * p.Nkv + kvh;
        const size_t out_row = ((size_t)b * p.Nkv + kvh) * (size_t)p.C + (size_t)(pl.Lp + s);
        reinterpret_cast<uint4 *>(static_cast<char *>(tensor ? p.prv : p.prk) + out_row * kD * 2)[vec] =
            reinterpret_cast<const uint4 *>(static_cast<const char *>(tensor ? p.v : p.k) + in_row * kD * 2)[vec];
      }
    }
  } else if (kvh == 0 && rt == 0 && sp == 0 && tid == 0) {
    flag(p, GQAW_DEV_BAD_SEQLEN);
  }

  // This thread's query row.  The tile's tokens are spread evenly over the four TMEM
  // lane quarters (one warp each), tpq tokens per quarter, so a short step (S x g < 128
  // rows) still gives every warp real rows.
  const int r = tid;
  const int tpq = (s_end - s0 + 3) / 4;
  const int tl = (r % 32) / g;  // token within the quarter
  const int tok = s0 + (r / 32) * tpq + tl;
  const int hh = r % g;
  const bool row_ok = ok && tl < tpq && tok < s_end;
  const long long qi = P + tok;  // absolute position of the row's token
  const long long rlo = qi - p.W + 1 > 0 ? qi - p.W + 1 : 0;
  const int h = kvh * g + hh;
  const float *bias_row = (row_ok && p.bias) ? p.bias + (long long)b * p.bsb + (long long)h * p.bsh +
                                                   (long long)tok * p.bss
                                             : nullptr;

  uint64_t pol = 0;
  const int row0_cache = (int)(((long long)b * p.Nkv + kvh) * p.C);
  // Thread 0: load the K (or V) half-tiles of key tile t into buffer `dst`.
  auto load_kv = [&](int t, unsigned char *dst, uint64_t *bar, bool value) {
    mbar_arrive_expect_tx(bar, 2 * kHalf);
    if (t < nc) {
      const CUtensorMap *m = value ? &maps.vc : &maps.kc;
      const int row = row0_cache + (int)(klo + (long long)t * kKeys - P + pl.Lp);
      tc::tma_load_2d(dst, m, 0, row, bar, pol);
      tc::tma_load_2d(dst + kHalf, m, 64, row, bar, pol);
    } else {
      const CUtensorMap *m = value ? &maps.vn : &maps.kn;
      const int tokrow = b * p.S + (t - nc) * kKeys;
      tc::tma_load_3d(dst, m, 0, kvh, tokrow, bar, pol);
      tc::tma_load_3d(dst + kHalf, m, 64, kvh, tokrow, bar, pol);
    }
  };
  auto kbuf = [&](int k) { return smem + kSmemK + (k % 2) * 2 * kHalf; };
  auto vbuf = [&](int k) { return smem + kSmemV + (k % 2) * 2 * kHalf; };
  const int ntl = t_end - t_begin;  // key tiles of this CTA
  // S = Q K^T of local tile k into tensor-memory buffer k % 2 (thread 0).
  auto issue_qk = [&](int k) {
    if (!mbar_wait(&kfull[k % 2], (k / 2) & 1)) flag(p, GQAW_DEV_TIMEOUT);
    tc::fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const int half = kk / 4, off = (kk % 4) * 32;
      const uint64_t a = tc::smem_desc_sw128(smem + kSmemQ + half * kHalf + off, 16, 1024);
      const uint64_t bd = tc::smem_desc_sw128(kbuf(k) + half * kHalf + off, 16, 1024);
      tc::mma_bf16_ss(tmem_s + (k % 2) * kKeys, a, bd, kIdescQK, kk > 0);
    }
    tc::mma_commit(&bar_s[k % 2]);
  };
  if (tid == 0 && ntl > 0) {
    pol = policy_evict_first();
    mbar_arrive_expect_tx(bar_q, 2 * kHalf);
    for (int q = 0; q < 4; ++q) {  // quarter q: tokens s0 + q * tpq ..., rows [32q, 32q + 32)
      const int qtok = b * p.S + s0 + q * tpq;
      tc::tma_load_3d(smem + kSmemQ + q * 4096, &maps.q, 0, kvh * g, qtok, bar_q, tc::policy_evict_last());
      tc::tma_load_3d(smem + kSmemQ + kHalf + q * 4096, &maps.q, 64, kvh * g, qtok, bar_q,
                      tc::policy_evict_last());
    }
    for (int k = 0; k < 2 && k < ntl; ++k) {
      load_kv(t_begin + k, kbuf(k), &kfull[k % 2], false);
      load_kv(t_begin + k, vbuf(k), &vfull[k % 2], true);
    }
    if (!mbar_wait(bar_q, 0)) flag(p, GQAW_DEV_TIMEOUT);
    issue_qk(0);
  }

  float m_run = -INFINITY, l_run = 0.f;
  const bool plain = p.capmul == 0.f && p.bias == nullptr;  // logits need only the scale
  // A bounded wait that expires sets s_abort; every thread reads it after the tile's
  // barrier, so the whole CTA leaves the loop together.
  auto bail = [&]() {
    flag(p, GQAW_DEV_TIMEOUT);
    s_abort = 1;
  };
  int done_tiles = 0;
  for (int k = 0; k < ntl; ++k) {
    const int t = t_begin + k;
    const long long j0 = t < nc ? klo + (long long)t * kKeys : P + (long long)(t - nc) * kKeys;
    const long long jhi_src = t < nc ? P : P + s_end;  // keys of this source
    const int nvalid = (int)(jhi_src - j0 < kKeys ? jhi_src - j0 : kKeys);
    // visible columns of this row in this tile: [c_lo, c_hi)
    int c_lo = 0, c_hi = 0;
    if (row_ok) {
      const long long lo = rlo - j0, hi = qi - j0 + 1;
      c_lo = (int)(lo < 0 ? 0 : (lo > kKeys ? kKeys : lo));
      c_hi = (int)(hi < 0 ? 0 : (hi > nvalid ? nvalid : hi));
    }

    // ---- tensor core: S of the next tile while this one is in softmax
    if (tid == 0 && k + 1 < ntl) issue_qk(k + 1);
    if (!mbar_wait(&bar_s[k % 2], (k / 2) & 1)) bail();
    tc::fence_after_sync();
    // K buffer k % 2 is free again (Q.K^T of tile k is done): fetch K of tile k + 2
    if (tid == 0 && k + 2 < ntl) load_kv(t + 2, kbuf(k), &kfull[k % 2], false);

    // ---- logits of this row (log2 units), row maximum
    float z[kKeys];
    const uint32_t ts = tmem_s + (k % 2) * kKeys + ((uint32_t)(warp * 32) << 16);
    float mt = -INFINITY;
    if (plain) {
#pragma unroll
      for (int c32 = 0; c32 < kKeys / 32; ++c32) {
        float v[32];
        tc::tmem_ld32(ts + c32 * 32, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = c32 * 32 + c;
          z[col] = (col >= c_lo && col < c_hi) ? v[c] : -INFINITY;
          mt = fmaxf(mt, z[col]);
        }
      }
      mt *= p.qscale;  // qscale > 0: max commutes with the scale
    } else {
      const float *brow = bias_row ? bias_row + j0 : nullptr;  // this tile's bias columns
#pragma unroll
      for (int c32 = 0; c32 < kKeys / 32; ++c32) {
        float v[32];
        tc::tmem_ld32(ts + c32 * 32, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = c32 * 32 + c;
          const bool vis = col >= c_lo && col < c_hi;
          float x = v[c] * p.qscale;
          if (p.capmul != 0.f) x = p.capmul * fast_tanh(x);
          if (vis && brow) x = fmaf(p.biasmul, brow[col], x);
          z[col] = vis ? x : -INFINITY;
          mt = fmaxf(mt, z[col]);
        }
      }
    }

    // ---- the previous P.V has finished: P buffer, V buffer (k-1) % 2 and O are free
    if (k > 0 && !mbar_wait(bar_o, (k - 1) & 1)) bail();
    if (tid == 0 && k >= 1 && k + 1 < ntl) load_kv(t + 1, vbuf(k + 1), &vfull[(k + 1) % 2], true);
    tc::fence_after_sync();

    // lazy rescale: the reference max moves only when exceeded by more than 2^8
    const bool need = mt > m_run + kRescaleLog2;
    float alpha = 1.f;
    if (need) {
      alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mt);
      m_run = mt;
      l_run *= alpha;
    }
    if (k > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int c32 = 0; c32 < kD / 32; ++c32) {
        float v[32];
        const uint32_t ta_o = tmem_o + ((uint32_t)(warp * 32) << 16) + c32 * 32;
        tc::tmem_ld32(ta_o, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] *= alpha;
        tc::tmem_st32(ta_o, v);
      }
    }
    // ---- P (bf16) into shared memory, K-major with 128-byte swizzle
    const float base = m_run == -INFINITY ? 0.f : m_run;
    const float zs = plain ? p.qscale : 1.f;  // plain logits are still unscaled
#pragma unroll
    for (int q = 0; q < kKeys / 8; ++q) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pv[e] = fast_exp2(fmaf(z[q * 8 + e], zs, -base));
        l_run += pv[e];
      }
      uint4 w;
      w.x = tc::pack_bf16x2(pv[0], pv[1]);
      w.y = tc::pack_bf16x2(pv[2], pv[3]);
      w.z = tc::pack_bf16x2(pv[4], pv[5]);
      w.w = tc::pack_bf16x2(pv[6], pv[7]);
      const int half = q / 8, chunk = q % 8;
      *reinterpret_cast<uint4 *>(smem + kSmemP + half * kHalf + r * 128 + ((chunk ^ (r & 7)) * 16)) = w;
    }
    // keys past this source's range: their V rows must be finite (0 * NaN is NaN)
    unsigned char *vb = vbuf(k);
    if (nvalid < kKeys) {
      if (!mbar_wait(&vfull[k % 2], (k / 2) & 1)) bail();
      for (int e = tid; e < (kKeys - nvalid) * 16; e += kThreads) {
        const int row = nvalid + e / 16, part = e % 16;  // 16 chunks of 16 B per key (two halves)
        *reinterpret_cast<uint4 *>(vb + (part / 8) * kHalf + row * 128 + (part % 8) * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- O += P V
    if (tid == 0) {
      if (!mbar_wait(&vfull[k % 2], (k / 2) & 1)) bail();
      tc::fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const int half = kk / 4, off = (kk % 4) * 32;
        const uint64_t a = tc::smem_desc_sw128(smem + kSmemP + half * kHalf + off, 16, 1024);
        // V: rows = keys (K), 64-dim halves (MN) 16 KB apart, 8-key groups 1 KB apart
        const uint64_t bd = tc::smem_desc_sw128(vb + kk * 16 * 128, kHalf, 1024);
        tc::mma_bf16_ss(tmem_o, a, bd, kIdescPV, k > 0 || kk > 0);
      }
      tc::mma_commit(bar_o);
    }
    ++done_tiles;
    if (s_abort) break;  // uniform: read by all threads after the barrier above
  }
  if (done_tiles > 0 && !mbar_wait(bar_o, (done_tiles - 1) & 1)) flag(p, GQAW_DEV_TIMEOUT);
  // an S = Q K^T issued ahead for a tile the loop did not reach must land before exit
  if (tid == 0 && done_tiles < ntl && done_tiles + 1 <= ntl)
    mbar_wait(&bar_s[done_tiles % 2], (done_tiles / 2) & 1);
  tc::fence_after_sync();

  // ---- epilogue: this CTA's (O, m, l) for its row
  float o[kD];
  if (ntl > 0) {
#pragma unroll
    for (int c32 = 0; c32 < kD / 32; ++c32) {
      float v[32];
      tc::tmem_ld32(tmem_o + ((uint32_t)(warp * 32) << 16) + c32 * 32, v);
#pragma unroll
      for (int c = 0; c < 32; ++c) o[c32 * 32 + c] = v[c];
    }
  } else {
#pragma unroll
    for (int c = 0; c < kD; ++c) o[c] = 0.f;
  }
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
  const long long orow = ((long long)b * p.S + tok) * p.Nq + h;
  if (ok) {
    if (ta.nsplit == 1) {
      if (row_ok) {
        const float inv = sink_reciprocal(l_run, m_run, sink_log2(p, h));
#pragma unroll
        for (int c = 0; c < kD; c += 8) {
          uint4 w;
          w.x = tc::pack_bf16x2(o[c] * inv, o[c + 1] * inv);
          w.y = tc::pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
          w.z = tc::pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
          w.w = tc::pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
          *reinterpret_cast<uint4 *>(out + orow * kD + c) = w;
        }
      }
    } else {
      float *part = p.partials + ((long long)blockIdx.x * kRows + r) * kTcPartialStride;
#pragma unroll
      for (int c = 0; c < kD; c += 4)
        *reinterpret_cast<float4 *>(part + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
      part[kD] = m_run;
      part[kD + 1] = l_run;
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&p.tickets[unit_tile], 1u) == (unsigned)ta.nsplit - 1u;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        if (row_ok) {
          const long long first = (long long)blockIdx.x - sp;  // split 0 of this query tile
          float M = -INFINITY;
          for (int q = 0; q < ta.nsplit; ++q)
            M = fmaxf(M, __ldcg(p.partials + ((first + q) * kRows + r) * kTcPartialStride + kD));
          const float mb = M == -INFINITY ? 0.f : M;
          float L = 0.f;
          float f[16];
          for (int q = 0; q < ta.nsplit && q < 16; ++q) {
            const float mq = __ldcg(p.partials + ((first + q) * kRows + r) * kTcPartialStride + kD);
            f[q] = mq == -INFINITY ? 0.f : exp2f(mq - mb);
            L += f[q] * __ldcg(p.partials + ((first + q) * kRows + r) * kTcPartialStride + kD + 1);
          }
          const float inv = sink_reciprocal(L, mb, sink_log2(p, h));
          for (int c = 0; c < kD; c += 2) {
            float a0 = 0.f, a1 = 0.f;
            for (int q = 0; q < ta.nsplit && q < 16; ++q) {
              if (f[q] == 0.f) continue;
              const float *pq = p.partials + ((first + q) * kRows + r) * kTcPartialStride;
              a0 = fmaf(f[q], __ldcg(pq + c), a0);
              a1 = fmaf(f[q], __ldcg(pq + c + 1), a1);
            }
            *reinterpret_cast<uint32_t *>(out + orow * kD + c) = tc::pack_bf16x2(a0 * inv, a1 * inv);
          }
        }
        if (tid == 0) p.tickets[unit_tile] = 0u;
      }
    }
  }

  // release tensor memory (all tcgen05.ld of this CTA are complete)
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
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(mma_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done[dev] = true;
  }
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
