// gqaw_finish.cu -- second kernel of a step: the cache update of registered items.
//
// The attention kernel already appended the new rows of every item that reclaims no
// block (in place) and registered the others in a list in the workspace.  This kernel
// updates the cache of the registered items, one job per (item, kv head, K or V,
// column group), grid-strided over its blocks:
//
//  * block compaction (onnxruntime PR #31142 "[CPU] Add windowed kv cache for GQA",
//    Key design decisions: "Drifting layout", "Skip compaction on drifting steps"):
//    with kept = L(T) - S surviving rows and seed = L(P) + S - L(T) (a whole number of
//    G-row blocks), present row r <- past row r + seed for r in [0, kept).  With a
//    separate present buffer every surviving row is copied (seed may be 0).
//  * append (PR #32419 "Specify GroupQueryAttention windowed KV cache layout
//    contract", Description: row i holds absolute position T - L + i): present rows
//    [max(kept, 0), L(T)) <- the last new rows.  When S > L(T) only the tail survives.
//  * for an entry flagged kListBelowOnly (a separate present buffer whose window rows and
//    new rows the small-step attention kernel has written from its staged tiles), only
//    the surviving rows below the window: present row r <- past row r + seed for
//    r in [0, lo_row - seed), lo_row = L(P) - min(P, W - 1) the window's first row.
//
// In place, the move reads rows [seed, seed + kept) and writes rows [0, kept): an
// overlapping forward move.  It runs in ascending batches; each batch loads all its
// source vectors into registers, synchronises the block, then stores.  A batch's
// sources lie at or above its first destination row plus seed, and every earlier
// store went below that row, so every source is read before anything overwrites it.
// The column groups of a row are independent chains (a row only moves within its own
// columns), so several blocks share a slice without any ordering between them.
//
// The last block to finish empties the list for the next step.
//
// With separate present buffers nothing a block stores is read by another, and
// finish_copy_kernel replaces the chains by independent jobs: one per 32 KB segment of
// whole rows of a slice, taken one at a time from a counter in the workspace, so that
// every block keeps a batch in flight (a chain's batches are round trips one after the
// other, and there are fewer chains than blocks).
#include "gqaw_internal.cuh"

namespace gqaw {

constexpr int kFinishThreads = 256;
constexpr int kCopyVecs = 8;  // 16-byte vectors per thread per batch (32 KB per block)

__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const Params p) {
  pdl_wait();                // the attention kernel has finished reading the cache
  const unsigned nmove = *reinterpret_cast<volatile unsigned *>(p.move_count);
  if (nmove == 0) {          // nothing registered: nothing to reset either
    pdl_launch_dependents(); // the next step's kernels may be launched now
    return;
  }
  // With rows to move, the next step's kernels are let in only when this block is done:
  // launched early, their CTAs would hold whole SMs (waiting for this grid) that the
  // copies need.
  // Whole rows (one contiguous chain per slice) unless that leaves fewer chains than
  // blocks; then rows split into column groups, up to p.ncg of them.  nmove is the same
  // for every block, so they all agree on the job numbering.
  int ncg = 1;
  while (ncg < p.ncg && (long long)nmove * p.Nkv * 2 * ncg < gridDim.x) ncg *= 2;
  const int per_item = p.Nkv * 2 * ncg;
  const long long njobs = (long long)nmove * per_item;
  const int rowb = p.rowbytes;
  const int cvec = rowb / 16 / ncg;  // vectors per row in one column group

  for (long long job0 = blockIdx.x; job0 < njobs; job0 += gridDim.x) {
    const int entry = p.move_list[job0 / per_item];
    const int b = entry & (kListBelowOnly - 1);
    const bool below_only = (entry & kListBelowOnly) != 0;
    int job = (int)(job0 % per_item);
    const int cg = job % ncg;
    job /= ncg;
    const int tensor = job & 1;  // 0: key, 1: value
    const int kvh = job >> 1;
    Plan pl;
    if (!plan_item(p, b, pl)) continue;  // registered items were valid; defensive
    const long long kept = pl.Lt - p.S;
    const long long seed = pl.Lp + p.S - pl.Lt;
    const long long nwin = pl.P < p.W - 1 ? pl.P : p.W - 1;
    // rows to move: all surviving ones, or those below the window
    const long long nmove = below_only ? pl.Lp - nwin - seed : kept;
    const size_t sl = (size_t)b * p.Nkv + kvh;
    const char *src = static_cast<const char *>(tensor ? p.pv : p.pk) + sl * p.C * rowb;
    char *dst = static_cast<char *>(tensor ? p.prv : p.prk) + sl * p.C * rowb;
    const bool inplace = src == dst;
    const int col0 = cg * cvec * 16;

    if (nmove > 0 && (seed > 0 || !inplace)) {
      const int rows_per_batch = kFinishThreads * kCopyVecs / cvec;
      for (long long r0 = 0; r0 < nmove; r0 += rows_per_batch) {
        const int nrow = (int)(nmove - r0 < rows_per_batch ? nmove - r0 : rows_per_batch);
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

    if (below_only) continue;  // the new rows are in place already
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
  }

  pdl_launch_dependents();

  // Completion ticket: every block has read move_count above; the last one resets the
  // list so the next step's attention kernel starts from an empty list.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.done_count, 1u) == gridDim.x - 1) {
      *p.move_count = 0u;
      *p.done_count = 0u;
      __threadfence();
    }
  }
}

namespace {

constexpr int kPlanCache = 512;  // registered items whose plans a copy block keeps in shared memory

// A registered item as the copy jobs need it (b < 0: its seqlens_k is out of range).
struct CopyPlan {
  long long Lp, Lt, nrows;  // nrows: the rows to move (0 or less: none)
  int b, below_only;
};

__device__ __forceinline__ CopyPlan copy_plan(const Params &p, int entry) {
  CopyPlan cp;
  cp.b = entry & (kListBelowOnly - 1);
  cp.below_only = (entry & kListBelowOnly) != 0;
  Plan pl;
  if (!plan_item(p, cp.b, pl)) {  // registered items were valid; defensive
    cp.b = -1;
    cp.Lp = cp.Lt = cp.nrows = 0;
    return cp;
  }
  cp.Lp = pl.Lp;
  cp.Lt = pl.Lt;
  const long long seed = pl.Lp + p.S - pl.Lt, nwin = pl.P < p.W - 1 ? pl.P : p.W - 1;
  cp.nrows = cp.below_only ? pl.Lp - nwin - seed : pl.Lt - p.S;  // below the window, or all kept rows
  return cp;
}

}  // namespace

// The cache update into separate present buffers: the same rows as finish_kernel moves,
// as independent jobs (slice, segment of R whole rows), job = slice * segments + segment,
// taken in order from a counter (the items' row counts differ: a fixed share per block
// left blocks idle); a slice's last segment also appends the new rows.  Each block first
// computes the registered items' plans into shared memory (one load of seqlens_k per item).
__global__ void __launch_bounds__(kFinishThreads, 4) finish_copy_kernel(const Params p) {
  pdl_wait();                // the attention kernel has finished reading the cache
  const unsigned nmove = *reinterpret_cast<volatile unsigned *>(p.move_count);
  if (nmove == 0) {
    pdl_launch_dependents();
    return;
  }
  __shared__ CopyPlan s_plan[kPlanCache];
  __shared__ unsigned s_maxseg, s_job;
  __shared__ int s_last;
  const int rowb = p.rowbytes, cvec = rowb / 16;
  const long long R = kFinishThreads * kCopyVecs / cvec;  // rows per segment
  if (threadIdx.x == 0) s_maxseg = 0u;
  __syncthreads();
  for (unsigned e = threadIdx.x; e < nmove; e += kFinishThreads) {
    const CopyPlan cp = copy_plan(p, p.move_list[e]);
    if (e < kPlanCache) s_plan[e] = cp;
    if (cp.b >= 0 && cp.nrows > 0) atomicMax(&s_maxseg, (unsigned)((cp.nrows + R - 1) / R));
  }
  __syncthreads();
  const long long nseg = s_maxseg > 0u ? s_maxseg : 1u;  // segment 0 of each slice appends
  const long long nslices = (long long)nmove * p.Nkv * 2;
  for (;;) {
    if (threadIdx.x == 0) s_job = atomicAdd(p.job_count, 1u);
    __syncthreads();
    const long long job = s_job;
    __syncthreads();  // every thread has read s_job before it is written again
    if (job >= nslices * nseg) break;
    const long long slice = job / nseg, sg = job % nseg;  // slice: (list entry, kv head, K or V)
    const int tensor = (int)(slice & 1), kvh = (int)((slice >> 1) % p.Nkv);
    const long long ei = (slice >> 1) / p.Nkv;
    const CopyPlan cp = ei < kPlanCache ? s_plan[ei] : copy_plan(p, p.move_list[ei]);
    if (cp.b < 0) continue;
    const long long seed = cp.Lp + p.S - cp.Lt, kept = cp.Lt - p.S;
    const long long last = cp.nrows > 0 ? (cp.nrows + R - 1) / R - 1 : 0;
    if (sg > last) continue;
    const size_t sl = (size_t)cp.b * p.Nkv + kvh;
    const char *src = static_cast<const char *>(tensor ? p.pv : p.pk) + sl * p.C * rowb;
    char *dst = static_cast<char *>(tensor ? p.prv : p.prk) + sl * p.C * rowb;
    if (cp.nrows > 0) {
      const long long r0 = sg * R, n = cp.nrows - r0 < R ? cp.nrows - r0 : R;
      uint4 buf[kCopyVecs];
#pragma unroll
      for (int u = 0; u < kCopyVecs; ++u) {
        const int e = threadIdx.x + u * kFinishThreads;
        if (e < n * cvec) buf[u] = *reinterpret_cast<const uint4 *>(src + (r0 + e / cvec + seed) * rowb + (e % cvec) * 16);
      }
#pragma unroll
      for (int u = 0; u < kCopyVecs; ++u) {
        const int e = threadIdx.x + u * kFinishThreads;
        if (e < n * cvec) *reinterpret_cast<uint4 *>(dst + (r0 + e / cvec) * rowb + (e % cvec) * 16) = buf[u];
      }
    }
    if (cp.below_only || sg != last) continue;  // the new rows are in place already
    const long long a0 = kept > 0 ? kept : 0;
    const char *newrows = static_cast<const char *>(tensor ? p.v : p.k);
    for (long long e = threadIdx.x; e < (cp.Lt - a0) * cvec; e += kFinishThreads) {
      const long long r = a0 + e / cvec;
      const size_t off = (((size_t)cp.b * p.S + (size_t)(seed + r - cp.Lp)) * p.Nkv + kvh) * (size_t)rowb;
      *reinterpret_cast<uint4 *>(dst + r * rowb + (e % cvec) * 16) =
          *reinterpret_cast<const uint4 *>(newrows + off + (e % cvec) * 16);
    }
  }

  pdl_launch_dependents();

  // the last block resets the list for the next step
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(p.done_count, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    *p.move_count = 0u;
    *p.job_count = 0u;
    *p.done_count = 0u;
    __threadfence();
  }
}

cudaError_t launch_finish(const Params &p, int blocks, cudaStream_t stream, bool separate) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kFinishThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = separate ? cudaLaunchKernelEx(&cfg, finish_copy_kernel, p) : cudaLaunchKernelEx(&cfg, finish_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqaw
