// gqaw_finish.cu -- second kernel of a step: split combine + cache update.
//
// Blocks [0, ncombine) merge the per-chunk partial results of the attention kernel
// (log-sum-exp in log2 units) into the output.  The remaining blocks update the cache
// of one (item, kv head, K or V, column group) each:
//
//  * block compaction (onnxruntime PR #31142 "[CPU] Add windowed kv cache for GQA",
//    Key design decisions: "Drifting layout", "Skip compaction on drifting steps"):
//    with kept = L(T) - S surviving rows and seed = L(P) + S - L(T) (a whole number of
//    G-row blocks), present row r <- past row r + seed for r in [0, kept).  Nothing
//    moves when seed == 0 and the cache is updated in place.
//  * append (PR #32419 "Specify GroupQueryAttention windowed KV cache layout
//    contract", Description: row i holds absolute position T - L + i): present rows
//    [max(kept, 0), L(T)) <- the last new rows.  When S > L(T) only the tail survives.
//
// In place, the move reads rows [seed, seed + kept) and writes rows [0, kept): an
// overlapping forward move.  It runs in ascending batches; each batch loads all its
// source vectors into registers, synchronises the block, then stores.  A batch's
// sources lie at or above its first destination row plus seed, and every earlier
// store went below that row, so every source is read before anything overwrites it.
// The column groups of a row are independent chains (a row only moves within its own
// columns), so several blocks share a slice without any ordering between them.
#include "gqaw_internal.cuh"

namespace gqaw {

constexpr int kFinishThreads = 256;
constexpr int kCopyVecs = 8;  // 16-byte vectors per thread per batch (32 KB per block)

template <typename T>
__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const Params p) {
  if ((int)blockIdx.x < p.ncombine) {
    // ------------------------------------------------------------- split combine
    const long long nrows = (long long)p.B * p.S * p.Nq;
    const long long e = (long long)blockIdx.x * kFinishThreads + threadIdx.x;
    if (e >= nrows * p.D) return;
    const long long row = e / p.D;
    const int d = (int)(e % p.D);
    const int b = (int)(row / ((long long)p.S * p.Nq));
    Plan pl;
    if (!plan_item(p, b, pl)) return;  // flagged by the attention kernel
    const float *m = p.ws_m + row * p.nsplit;
    const float *l = p.ws_l + row * p.nsplit;
    float M = -INFINITY;
    for (int sp = 0; sp < p.nsplit; ++sp) M = fmaxf(M, m[sp]);
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, A = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) {
      if (m[sp] == -INFINITY) continue;  // empty chunk: its accumulator is not written
      const float f = exp2f(m[sp] - base);
      L = fmaf(f, l[sp], L);
      A = fmaf(f, p.ws_acc[(row * p.nsplit + sp) * p.D + d], A);
    }
    static_cast<T *>(p.out)[row * p.D + d] = Elem<T>::store(A / L);
    return;
  }

  // --------------------------------------------------------------- cache update
  int job = (int)blockIdx.x - p.ncombine;
  const int cg = job % p.ncg;
  job /= p.ncg;
  const int tensor = job & 1;  // 0: key, 1: value
  const int sl = job >> 1;     // b * Nkv + kvh
  const int b = sl / p.Nkv, kvh = sl % p.Nkv;
  Plan pl;
  if (!plan_item(p, b, pl)) {
    if (threadIdx.x == 0) flag(p, GQAW_DEV_BAD_SEQLEN);
    return;
  }
  const long long kept = pl.Lt - p.S;
  const long long seed = pl.Lp + p.S - pl.Lt;
  const int rowb = p.rowbytes;
  const char *src = static_cast<const char *>(tensor ? p.pv : p.pk) + (size_t)sl * p.C * rowb;
  char *dst = static_cast<char *>(tensor ? p.prv : p.prk) + (size_t)sl * p.C * rowb;
  const bool inplace = src == dst;
  const int cvec = rowb / 16 / p.ncg;  // vectors per row in this column group
  const int col0 = cg * cvec * 16;

  if (kept > 0 && (seed > 0 || !inplace)) {
    const int rows_per_batch = kFinishThreads * kCopyVecs / cvec;
    for (long long r0 = 0; r0 < kept; r0 += rows_per_batch) {
      const int nrow = (int)(kept - r0 < rows_per_batch ? kept - r0 : rows_per_batch);
      const int nvec = nrow * cvec;
      uint4 buf[kCopyVecs];
#pragma unroll
      for (int u = 0; u < kCopyVecs; ++u) {
        const int e = threadIdx.x + u * kFinishThreads;
        if (e < nvec) {
          const long long r = r0 + e / cvec;
          buf[u] = *reinterpret_cast<const uint4 *>(src + (r + seed) * rowb + col0 + (e % cvec) * 16);
        }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kCopyVecs; ++u) {
        const int e = threadIdx.x + u * kFinishThreads;
        if (e < nvec) {
          const long long r = r0 + e / cvec;
          *reinterpret_cast<uint4 *>(dst + r * rowb + col0 + (e % cvec) * 16) = buf[u];
        }
      }
    }
  }

  // Append: present row r (r >= max(kept, 0)) holds new token seed + r - Lp.
  const long long a0 = kept > 0 ? kept : 0;
  const long long napp = pl.Lt - a0;
  const char *newrows = static_cast<const char *>(tensor ? p.v : p.k);
  for (long long e = threadIdx.x; e < napp * cvec; e += kFinishThreads) {
    const long long r = a0 + e / cvec;
    const long long sj = seed + r - pl.Lp;
    const size_t off = (((size_t)b * p.S + (size_t)sj) * p.Nkv + kvh) * (size_t)rowb;
    *reinterpret_cast<uint4 *>(dst + r * rowb + col0 + (e % cvec) * 16) =
        *reinterpret_cast<const uint4 *>(newrows + off + col0 + (e % cvec) * 16);
  }
  if (p.resident_out && kvh == 0 && tensor == 0 && cg == 0 && threadIdx.x == 0)
    p.resident_out[b] = (int32_t)pl.Lt;
}

cudaError_t launch_finish(const Params &p, int dtype, int blocks, cudaStream_t stream) {
  if (dtype == GQAW_F32)
    finish_kernel<float><<<blocks, kFinishThreads, 0, stream>>>(p);
  else
    finish_kernel<__nv_bfloat16><<<blocks, kFinishThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gqaw
