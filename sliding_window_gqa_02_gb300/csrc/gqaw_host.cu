// gqaw_host.cu -- the C ABI of include/gqaw.h: argument checks, launch planning and
// kernel launches.  No allocation, no synchronisation (except gqaw_device_status).
//
// A step is two kernels on the caller's stream:
//   1. attention (attend_kernel): reads the pre-step cache rows and the new rows, so a
//      multi-token step that evicts rows its own queries need is handled without any
//      staging copy (onnxruntime PR #31142 "[CPU] Add windowed kv cache for GQA",
//      Key design decisions, "Staging for hazardous steps": the CPU copies into a
//      temporary cache; here the order of the two kernels makes that unnecessary);
//   2. finish (finish_kernel): split combine, block compaction, append.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "gqaw_tc.cuh"

namespace gqaw {
cudaError_t launch_attend_f32(const Params &p, int gb, int blocks, cudaStream_t stream);
cudaError_t launch_attend_bf16(const Params &p, int gb, int blocks, cudaStream_t stream);
int attend_tile_f32(int D);
int attend_tile_bf16(int D);
cudaError_t launch_finish(const Params &p, int blocks, cudaStream_t stream, bool separate);
cudaError_t launch_mma(const Params &p, const TcArgs &ta, const TcMaps &maps, int grid, cudaStream_t stream);
cudaError_t launch_rotary(const Params &p, cudaStream_t stream);
cudaError_t launch_attend_q8(const Params &p, int gb, int blocks, cudaStream_t stream);
int attend_tile_q8(int D);
cudaError_t launch_quantize(const Params &p, int max_blocks, cudaStream_t stream);
cudaError_t launch_mmad(const Params &p, const TdArgs &ta, const TdMaps &maps, int max_ctas, cudaStream_t stream);
}  // namespace gqaw

namespace {

thread_local std::string t_error;
std::atomic<unsigned long long> g_launches{0ull};

// Most attention CTAs of a step: GB300's 152 SMs x 2 resident CTAs per SM.
constexpr long long kMaxCtas = 152 * 2;
constexpr long long kSms = 152;
// Upper bound on the cache-update kernel's blocks (152 SMs x 2).
constexpr long long kFinishBlocks = 152 * 2;      // finish_kernel: two blocks per SM,
constexpr long long kFinishBlocksLong = 152 * 4;  // four for steps of 64 tokens or more
constexpr long long kFinishCopyBlocks = 152 * 4;  // finish_copy_kernel: four blocks per SM

gqaw_status fail(gqaw_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_error = buf;
  return s;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Ticket regions of caller workspaces.  Every completed step leaves its own tickets at
// zero, but where the tickets and the partial results sit depends on the step's shape
// (B, S, the kernel, the split count): a step of another shape may find its tickets
// where an earlier step left partial results, and a ticket that does not start at zero
// never reaches its count (the unit's output is never written).  So the library keeps,
// per workspace address, the ticket region of the last step enqueued on it, and clears
// a step's region first (one cudaMemsetAsync on its stream) when it differs.
struct WsRecord {
  const void *ws;
  size_t t0, t1;  // ticket region [t0, t1) of the last step; t1 == 0: the workspace is all zero
};
constexpr int kWsRecords = 64;
std::mutex g_ws_mutex;
WsRecord g_ws[kWsRecords] = {};
int g_ws_next = 0;

// Must the ticket region [t0, t1) of `ws` be cleared before this step?  Records it.
// A workspace the library has no record of (never seen, or its record was evicted by
// 64 others) is cleared to be safe.
bool tickets_need_clear(const void *ws, size_t t0, size_t t1) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (WsRecord &r : g_ws)
    if (r.ws == ws) {
      const bool clear = r.t1 != 0 && (r.t0 != t0 || r.t1 != t1);
      r.t0 = t0;
      r.t1 = t1;
      return clear;
    }
  g_ws[g_ws_next] = WsRecord{ws, t0, t1};
  g_ws_next = (g_ws_next + 1) % kWsRecords;
  return true;
}

// The workspace [ws, ws + bytes) has just been zeroed: its record says so, and records
// of workspaces inside it are dropped.
void note_zeroed(const void *ws, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  const char *lo = static_cast<const char *>(ws), *hi = lo + bytes;
  bool found = false;
  for (WsRecord &r : g_ws) {
    const char *p = static_cast<const char *>(r.ws);
    if (r.ws == ws) {
      r.t0 = r.t1 = 0;
      found = true;
    } else if (p && p >= lo && p < hi) {
      r = WsRecord{nullptr, 0, 0};
    }
  }
  if (!found) {
    g_ws[g_ws_next] = WsRecord{ws, 0, 0};
    g_ws_next = (g_ws_next + 1) % kWsRecords;
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Launch {
  int esize, rowbytes, group, gb, headblocks, tile, tpu, ncg;  // esize: cache element bytes
  int qsize;              // query/key/value/output element bytes
  int quant;              // cache_dtype of a quantized cache, or 0
  size_t off_kq, off_vq;  // quantized cache: the codes of the step's new rows
  size_t off_q16;         // quantized cache on the tensor-core kernel: the fp16 query copy
  size_t off_stash;       // small-step kernel, bf16 caches: one row stash per CTA
  long long units, ctas, ncopy, ncopy_sep;
  size_t off_list, off_tickets, off_partials, ws_bytes;
  int rot_dim;            // > 0: the rotary embedding is on, over this many dimensions
  size_t off_qrot, off_krot;  // the turned query and key rows in the workspace
  bool tc;                // multi-token step on the tensor-core kernel
  gqaw::TcArgs ta;
  long long tc_grid;
  bool td;                // small step (S x group <= 32) on the keys-as-M tensor-core kernel
  gqaw::TdArgs tda;
  long long td_ctas;
};

bool head_size_ok(int D) { return D == 8 || D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }

// Sizes only: everything gqaw_workspace_bytes needs.
gqaw_status plan_launch(const gqaw_step_args *a, Launch *L) {
  if (!a) return fail(GQAW_EINVAL, "args is NULL");
  if (a->batch_size < 0) return fail(GQAW_EINVAL, "batch_size %d < 0", a->batch_size);
  if (a->batch_size >= (1 << 30)) return fail(GQAW_EUNSUPPORTED, "batch_size %d >= 2^30", a->batch_size);
  if (a->sequence_length < 1) return fail(GQAW_EINVAL, "sequence_length %d < 1", a->sequence_length);
  if (a->num_heads < 1 || a->kv_num_heads < 1)
    return fail(GQAW_EINVAL, "num_heads %d and kv_num_heads %d must be >= 1", a->num_heads, a->kv_num_heads);
  if (a->num_heads % a->kv_num_heads != 0)
    return fail(GQAW_EINVAL, "num_heads %d is not a multiple of kv_num_heads %d", a->num_heads, a->kv_num_heads);
  if (a->dtype != GQAW_F32 && a->dtype != GQAW_BF16) return fail(GQAW_EINVAL, "unknown dtype %d", a->dtype);
  if (a->head_size < 1) return fail(GQAW_EINVAL, "head_size %d < 1", a->head_size);
  if (!head_size_ok(a->head_size))
    return fail(GQAW_EUNSUPPORTED, "head_size %d: supported are 8, 16, 32, 64, 128, 256", a->head_size);
  if (a->capacity < 1) return fail(GQAW_EINVAL, "capacity %d < 1", a->capacity);
  if (a->local_window_size < 1 || a->local_window_size > a->capacity)
    return fail(GQAW_EINVAL, "local_window_size %d must be in [1, capacity=%d]", a->local_window_size,
                a->capacity);
  if (a->total_sequence_length < a->sequence_length)
    return fail(GQAW_EINVAL, "total_sequence_length %d < sequence_length %d", a->total_sequence_length,
                a->sequence_length);
  if (!(a->scale >= 0.f) || !std::isfinite(a->scale)) return fail(GQAW_EINVAL, "scale must be finite and >= 0");
  if (!(a->softcap >= 0.f) || !std::isfinite(a->softcap))
    return fail(GQAW_EINVAL, "softcap must be finite and >= 0");
  if (a->split_keys < 0) return fail(GQAW_EINVAL, "split_keys %d < 0", a->split_keys);
  L->rot_dim = 0;
  if (a->do_rotary) {
    L->rot_dim = a->rotary_dim ? a->rotary_dim : a->head_size;
    if (L->rot_dim < 2 || L->rot_dim % 2 != 0 || L->rot_dim > a->head_size)
      return fail(GQAW_EINVAL, "rotary_dim %d must be even and in [2, head_size=%d]", a->rotary_dim, a->head_size);
    if (a->rotary_cache_len < 1) return fail(GQAW_EINVAL, "rotary_cache_len %d < 1", a->rotary_cache_len);
  }

  L->qsize = a->dtype == GQAW_F32 ? 4 : 2;
  L->quant = 0;
  if (a->cache_dtype != 0) {
    if (a->cache_dtype != GQAW_I8 && a->cache_dtype != GQAW_E4M3)
      return fail(GQAW_EINVAL, "unknown cache_dtype %d", a->cache_dtype);
    if (a->dtype != GQAW_BF16) return fail(GQAW_EUNSUPPORTED, "a quantized cache needs dtype GQAW_BF16");
    if (a->head_size != 64 && a->head_size != 128 && a->head_size != 256)
      return fail(GQAW_EUNSUPPORTED, "a quantized cache needs head_size 64, 128 or 256");
    L->quant = a->cache_dtype;
  }
  L->esize = L->quant ? 1 : L->qsize;
  L->rowbytes = a->head_size * L->esize;
  L->group = a->num_heads / a->kv_num_heads;
  L->gb = 1;  // query heads per CTA: the next power of two >= group, at most 8
  while (L->gb < L->group && L->gb < 8) L->gb *= 2;
  L->headblocks = (int)ceil_div(L->group, L->gb);
  L->tile = L->quant ? gqaw::attend_tile_q8(a->head_size)
                     : a->dtype == GQAW_F32 ? gqaw::attend_tile_f32(a->head_size) : gqaw::attend_tile_bf16(a->head_size);
  L->units = (long long)a->batch_size * a->sequence_length * a->kv_num_heads * L->headblocks;

  // Persistent stream-K attention: the step's work is units x tpu key tiles; the
  // grid has at most kMaxCtas CTAs (the launch lowers it to the resident count), each
  // taking a contiguous range of tiles.  split_keys > 0 asks for ranges of about that
  // many keys instead.
  const long long keys_max =
      a->local_window_size < a->total_sequence_length ? a->local_window_size : a->total_sequence_length;
  L->tpu = (int)ceil_div(keys_max, L->tile);
  const long long vtiles = L->units * L->tpu;
  long long ctas = std::min(vtiles, kMaxCtas);
  if (vtiles < kMaxCtas && L->units > 0) {
    // Less than one wave of tiles: latency decides.  Split each unit into k ranges
    // (k CTAs per unit), trading tiles per CTA against the merge a split unit needs
    // (about four tiles' worth of latency).
    long long best_k = 1, best_cost = L->tpu;
    for (long long k = 2; k <= L->tpu && L->units * k <= kMaxCtas; ++k) {
      const long long cost = ceil_div(L->tpu, k) + 4;
      if (cost < best_cost) {
        best_cost = cost;
        best_k = k;
      }
    }
    ctas = L->units * best_k;
  }
  if (a->split_keys > 0) ctas = std::max(1LL, std::min(ctas, ceil_div(vtiles * L->tile, a->split_keys)));
  L->ctas = ctas;

  const int nv = L->rowbytes / 16;
  // Most column groups a cache-update job may split a row into (each at least two
  // 16-byte vectors wide); the kernel picks the count from the number of moving items.
  L->ncg = 1;
  while (L->ncg * 2 <= nv / 2) L->ncg *= 2;

  // Workspace: [0, 256) status word and the three counters of the cache-update kernels;
  // the list itself (B items); per-unit tickets; two partial-result slots per
  // attention CTA.  Everything must start at zero (gqaw_workspace_init); every step
  // leaves the counters and tickets at zero again, and a step whose tickets sit
  // elsewhere than the previous step's clears them first (tickets_need_clear).
  L->off_list = 256;
  L->off_tickets = L->off_list + align256((size_t)a->batch_size * 4);
  L->off_partials = L->off_tickets + align256((size_t)L->units * 4);
  L->ws_bytes = L->off_partials + align256((size_t)L->ctas * 2 * L->gb * (a->head_size + 2) * 4);
  // Cache-update kernel: grid-stride over the jobs of the registered items.
  const long long jobs = (long long)a->batch_size * a->kv_num_heads * 2 * L->ncg;
  if (jobs > 0x7fffffffLL) return fail(GQAW_EUNSUPPORTED, "too many cache-update jobs");
  // Steps of many tokens reclaim long runs of rows in few items: more, narrower chains
  // on four blocks per SM (B=8 x 512 prefill 2.9% faster); decode steps mostly launch
  // the kernel to find nothing to move, where the larger grid costs about a microsecond.
  L->ncopy = std::min(jobs, a->sequence_length >= 64 ? kFinishBlocksLong : kFinishBlocks);
  // separate present buffers: a job per 32 KB segment of whole rows of a slice
  const long long seg_rows = 8 * 256 / (L->rowbytes / 16);  // 32 KB: 256 threads x 8 16-byte vectors
  L->ncopy_sep = std::min((long long)a->batch_size * a->kv_num_heads * 2 * ceil_div(a->capacity, seg_rows),
                          kFinishCopyBlocks);

  // Multi-token steps with bf16 caches and head size 128 run on the tensor-core
  // kernel when the query-head group tiles a 32-row lane quarter exactly.
  L->tc = a->dtype == GQAW_BF16 && a->head_size == 128 && a->sequence_length >= 2 && L->group <= 32 &&
          32 % L->group == 0;
  if (L->tc) {
    L->ta.tokens_per_tile = 128 / L->group;
    L->ta.rowtiles = (int)ceil_div(a->sequence_length, L->ta.tokens_per_tile);
    const long long base = (long long)a->batch_size * a->kv_num_heads * L->ta.rowtiles;
    // key tiles of one query tile: the window before it plus its own tokens
    const long long nt = ceil_div(std::min<long long>(a->local_window_size, a->total_sequence_length), 128) +
                         ceil_div(L->ta.tokens_per_tile, 128) + 1;
    // Key splits: the fewest waves of one-CTA-per-SM blocks, counting each block's
    // fixed cost (query load, pipeline fill, epilogue) as about two key tiles.
    long long ns = 1, best = -1;
    for (long long n = 1; n <= std::min(16LL, std::max(1LL, nt / 4)); ++n) {
      const long long cost = ceil_div(base * n, kSms) * (ceil_div(nt, n) + 2);
      if (best < 0 || cost < best) best = cost, ns = n;
    }
    if (a->split_keys > 0) ns = std::max(1LL, std::min(16LL, ceil_div(nt * 128, a->split_keys)));
    L->ta.nsplit = (int)ns;
    L->tc_grid = base * ns;  // units; the persistent kernel runs min(units, SMs) CTAs
    L->ta.units = L->tc_grid;
    if (L->tc_grid > 0x7fffffffLL) return fail(GQAW_EUNSUPPORTED, "too many attention blocks");
    L->off_tickets = L->off_list + align256((size_t)a->batch_size * 4);
    L->off_partials = L->off_tickets + align256((size_t)base * 4);
    L->ws_bytes = L->off_partials;
    if (ns > 1) L->ws_bytes += align256((size_t)L->tc_grid * 128 * gqaw::kTcPartialStride * 4);
  }
  // Steps with at most 32 query rows per (item, kv head) -- decode and short verify --
  // with bf16 caches and head size 128 run on the tensor-core kernel that puts the keys
  // on the MMA's M dimension: persistent, one CTA per SM, stream-K over (unit, 128-key
  // tile); partial results of units cut by a CTA range are merged in the kernel.
  const long long rows_all = (long long)a->batch_size * a->kv_num_heads * a->capacity;
  if (L->quant) L->tc = false;  // quantized caches: the FFMA kernel, or the small-step kernel below
  L->td = a->dtype == GQAW_BF16 && a->head_size == 128 && (long long)a->sequence_length * L->group <= 32 &&
          rows_all < 0x7fffffffLL && (long long)a->batch_size * a->sequence_length < 0x7fffffffLL;
  if (L->td) {
    L->tc = false;
    const long long nv = (long long)a->sequence_length * L->group;
    L->tda.npad = nv <= 16 ? 16 : 32;
    const long long keys = std::min<long long>(a->local_window_size - 1,
                                               (long long)a->total_sequence_length - a->sequence_length);
    L->tda.tpu = (int)std::max(1LL, ceil_div(keys, 128));
    L->tda.units = (long long)a->batch_size * a->kv_num_heads;
    const long long vt = L->tda.units * L->tda.tpu;
    long long ctas = std::min(vt, kSms);
    // Stream-K splits units at CTA range boundaries; a CTA that touches two units pays two
    // unit epilogues (dependent global round trips: the step's own keys, the partials, the
    // ticket, the merge), about kEpilogueTiles key tiles each on a busy memory system.
    // When the units fit in one wave, one whole unit per CTA can finish sooner: its CTAs
    // read TPU tiles and run one epilogue, against about V/SMs tiles and two epilogues.
    constexpr long long kEpilogueTiles = 6;
    if (a->split_keys > 0)  // the caller's chunk size overrides both choices
      ctas = std::max(1LL, std::min(ctas, ceil_div(vt * 128, a->split_keys)));
    else if (L->tda.units < kSms && L->tda.tpu + kEpilogueTiles <= ceil_div(vt, kSms) + 2 * kEpilogueTiles)
      ctas = L->tda.units;
    L->td_ctas = ctas;
    L->off_tickets = L->off_list + align256((size_t)a->batch_size * 4);
    L->off_partials = L->off_tickets + align256((size_t)L->tda.units * 4);
    L->ws_bytes = L->off_partials + align256((size_t)ctas * 2 * L->tda.npad * (128 + 2) * 4);
    L->off_stash = 0;
    if (!L->quant) {  // rows a CTA moves inside the attention pass for a later writer
      L->off_stash = L->ws_bytes;
      L->ws_bytes += align256((size_t)ctas * gqaw::kMoveStashBytes);
    }
  }
  // Rotary embedding: the turned query and key rows, in the input layouts.
  if (!L->td) L->off_stash = 0;
  L->off_qrot = L->off_krot = 0;
  if (L->rot_dim > 0) {
    const size_t tokens = (size_t)a->batch_size * a->sequence_length;
    L->off_qrot = align256(L->ws_bytes);
    L->off_krot = L->off_qrot + align256(tokens * a->num_heads * a->head_size * L->qsize);
    L->ws_bytes = L->off_krot + align256(tokens * a->kv_num_heads * a->head_size * L->qsize);
  }
  // Quantized cache: the codes of the step's new key and value rows.
  L->off_kq = L->off_vq = 0;
  if (L->quant) {
    const size_t n = (size_t)a->batch_size * a->sequence_length * a->kv_num_heads * a->head_size;
    L->off_kq = align256(L->ws_bytes);
    L->off_vq = L->off_kq + align256(n);
    L->ws_bytes = L->off_vq + align256(n);
  }
  L->off_q16 = 0;
  if (L->quant && L->td) {
    L->off_q16 = L->ws_bytes;
    L->ws_bytes += align256((size_t)a->batch_size * a->sequence_length * a->num_heads * a->head_size * 2);
  }
  return GQAW_OK;
}

bool aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

struct Range {
  const char *lo, *hi;
  const char *name;
};

bool overlap(const Range &x, const Range &y) { return x.lo < y.hi && y.lo < x.hi; }

gqaw_status check_pointers(const gqaw_step_args *a, const Launch &L) {
  struct {
    const void *p;
    const char *name;
  } req[] = {{a->query, "query"},           {a->key, "key"},
             {a->value, "value"},           {a->past_key, "past_key"},
             {a->past_value, "past_value"}, {a->present_key, "present_key"},
             {a->present_value, "present_value"}, {a->seqlens_k, "seqlens_k"},
             {a->output, "output"}};
  for (auto &r : req) {
    if (!r.p) return fail(GQAW_EINVAL, "%s is NULL", r.name);
    const size_t al = r.p == (const void *)a->seqlens_k ? 4 : 16;
    if (!aligned(r.p, al)) return fail(GQAW_EINVAL, "%s is not %zu-byte aligned", r.name, al);
  }
  if (a->attention_bias) {
    if (!aligned(a->attention_bias, 4)) return fail(GQAW_EINVAL, "attention_bias is not 4-byte aligned");
    if (a->bias_stride_b < 0 || a->bias_stride_h < 0 || a->bias_stride_s < 0)
      return fail(GQAW_EINVAL, "attention_bias strides must be >= 0");
  }
  if (a->head_sink && !aligned(a->head_sink, 4)) return fail(GQAW_EINVAL, "head_sink is not 4-byte aligned");
  if (L.quant) {
    if (!a->k_scale || !a->v_scale) return fail(GQAW_EINVAL, "a quantized cache needs k_scale and v_scale");
    if (!aligned(a->k_scale, 4) || !aligned(a->v_scale, 4))
      return fail(GQAW_EINVAL, "k_scale / v_scale are not 4-byte aligned");
  }
  if (L.rot_dim > 0) {
    if (!a->cos_cache || !a->sin_cache) return fail(GQAW_EINVAL, "do_rotary needs cos_cache and sin_cache");
    if (!aligned(a->cos_cache, L.qsize) || !aligned(a->sin_cache, L.qsize))
      return fail(GQAW_EINVAL, "cos_cache / sin_cache are not %d-byte aligned", L.qsize);
    if (a->position_ids && !aligned(a->position_ids, 8))
      return fail(GQAW_EINVAL, "position_ids is not 8-byte aligned");
  }
  if (!a->workspace) return fail(GQAW_EWORKSPACE, "workspace is NULL");
  if (!aligned(a->workspace, 256)) return fail(GQAW_EWORKSPACE, "workspace is not 256-byte aligned");
  if (a->workspace_bytes < L.ws_bytes)
    return fail(GQAW_EWORKSPACE, "workspace_bytes %zu < required %zu", a->workspace_bytes, L.ws_bytes);

  const size_t B = (size_t)a->batch_size, S = (size_t)a->sequence_length, D = (size_t)a->head_size;
  const size_t cache = B * a->kv_num_heads * (size_t)a->capacity * D * L.esize;
  const size_t qo = B * S * a->num_heads * D * L.qsize, kv = B * S * a->kv_num_heads * D * L.qsize;
  auto rng = [](const void *p, size_t n, const char *name) {
    return Range{static_cast<const char *>(p), static_cast<const char *>(p) + n, name};
  };
  const Range pk = rng(a->past_key, cache, "past_key"), pv = rng(a->past_value, cache, "past_value");
  const Range rk = rng(a->present_key, cache, "present_key"), rv = rng(a->present_value, cache, "present_value");
  const Range q = rng(a->query, qo, "query"), k = rng(a->key, kv, "key"), v = rng(a->value, kv, "value");
  const Range o = rng(a->output, qo, "output"), ws = rng(a->workspace, L.ws_bytes, "workspace");
  // present_key is past_key (in place) or disjoint from it; the same for values.
  if (a->present_key != a->past_key && overlap(rk, pk))
    return fail(GQAW_EINVAL, "present_key partially overlaps past_key");
  if (a->present_value != a->past_value && overlap(rv, pv))
    return fail(GQAW_EINVAL, "present_value partially overlaps past_value");
  const Range *written[] = {&rk, &rv, &o, &ws};
  const Range *all[] = {&pk, &pv, &rk, &rv, &q, &k, &v, &o, &ws};
  for (const Range *w : written)
    for (const Range *x : all) {
      if (w == x) continue;
      if ((w == &rk && x == &pk && a->present_key == a->past_key) ||
          (w == &rv && x == &pv && a->present_value == a->past_value))
        continue;
      if (overlap(*w, *x)) return fail(GQAW_EINVAL, "%s overlaps %s", w->name, x->name);
    }
  return GQAW_OK;
}

// Can the step leave out the cache-update kernel?  On the small-step kernel with a bf16
// cache updated in place, S <= G = C - W + 1 means a step reclaims at most one G-row
// block (seed = 0 or G); with S <= W and G <= the rows a CTA may stash, the surviving
// rows of a reclaiming item all lie in the window the step reads and the attention
// kernel moves them itself (kFused in gqaw_mmad.cuh), while a non-reclaiming item only
// appends.  So no item is ever recorded for the cache-update kernel.
bool finish_not_needed(const gqaw_step_args *a, const Launch &L) {
  const long long G = (long long)a->capacity - a->local_window_size + 1;
  return L.td && !L.quant && a->past_key == a->present_key && a->past_value == a->present_value &&
         a->sequence_length <= G && a->sequence_length <= a->local_window_size &&
         G <= gqaw::kMoveStashRows;
}

void fill_params(const gqaw_step_args *a, const Launch &L, gqaw::Params *p) {
  std::memset(p, 0, sizeof(*p));
  p->q = a->query;
  p->k = a->key;
  p->v = a->value;
  p->pk = a->past_key;
  p->pv = a->past_value;
  p->prk = a->present_key;
  p->prv = a->present_value;
  p->seqlens = a->seqlens_k;
  p->bias = a->attention_bias;
  p->bsb = a->bias_stride_b;
  p->bsh = a->bias_stride_h;
  p->bss = a->bias_stride_s;
  p->out = a->output;
  char *ws = static_cast<char *>(a->workspace);
  p->status = reinterpret_cast<uint32_t *>(ws);
  p->move_count = reinterpret_cast<uint32_t *>(ws + 4);
  p->done_count = reinterpret_cast<uint32_t *>(ws + 8);
  p->job_count = reinterpret_cast<uint32_t *>(ws + 12);
  p->move_list = reinterpret_cast<int32_t *>(ws + L.off_list);
  p->tickets = reinterpret_cast<uint32_t *>(ws + L.off_tickets);
  p->partials = reinterpret_cast<float *>(ws + L.off_partials);
  p->resident_out = a->resident_len_out;
  p->B = a->batch_size;
  p->S = a->sequence_length;
  p->Nq = a->num_heads;
  p->Nkv = a->kv_num_heads;
  p->D = a->head_size;
  p->C = a->capacity;
  p->W = a->local_window_size;
  p->total = a->total_sequence_length;
  p->group = L.group;
  p->headblocks = L.headblocks;
  p->nunits = L.units;
  p->tpu = L.tpu;
  const float scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt((float)a->head_size);
  if (a->softcap > 0.f) {
    p->qscale = scale / a->softcap;
    p->capmul = a->softcap * gqaw::kLog2e;
  } else {
    p->qscale = scale * gqaw::kLog2e;
    p->capmul = 0.f;
  }
  p->biasmul = gqaw::kLog2e;
  p->ncg = L.ncg;
  p->rowbytes = L.rowbytes;
  p->qbytes = L.qsize;
  p->sink = a->head_sink;
  p->sink_mode = a->head_sink ? 1 : (a->smooth_softmax ? 2 : 0);
  p->quant = L.quant;
  p->rot_dim = L.rot_dim;
  if (L.rot_dim > 0) {
    p->q_in = a->query;
    p->k_in = a->key;
    p->q = ws + L.off_qrot;
    p->krot = ws + L.off_krot;
    p->k = p->krot;
    p->rcos = a->cos_cache;
    p->rsin = a->sin_cache;
    p->pos_ids = reinterpret_cast<const long long *>(a->position_ids);
    p->rot_inter = a->rotary_interleaved ? 1 : 0;
    p->rot_len = a->rotary_cache_len;
  }
  if (L.quant) {  // the codes of the new rows, from the (maybe turned) rows of dtype T
    p->kq_in = p->k;
    p->vq_in = a->value;
    p->k = ws + L.off_kq;
    p->v = ws + L.off_vq;
    p->ks = a->k_scale;
    p->vs = a->v_scale;
    p->q16 = L.td ? ws + L.off_q16 : nullptr;
  }
  p->stash = L.off_stash ? reinterpret_cast<unsigned char *>(ws + L.off_stash) : nullptr;
  p->no_finish = finish_not_needed(a, L) ? 1 : 0;
}

gqaw_status prepare(const gqaw_step_args *a, Launch *L, gqaw::Params *p) {
  gqaw_status s = plan_launch(a, L);
  if (s != GQAW_OK) return s;
  if (a->batch_size == 0) return GQAW_OK;
  s = check_pointers(a, *L);
  if (s != GQAW_OK) return s;
  fill_params(a, *L, p);
  return GQAW_OK;
}

gqaw_status cuda_fail(cudaError_t e, const char *what) {
  return fail(GQAW_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled, resolved once through the runtime (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// A bf16 tensor map with 128-byte swizzle; dims/box innermost first, strides in bytes.
bool encode_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                const cuuint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, type, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gqaw_status run_mma(const gqaw_step_args *a, const Launch &L, const gqaw::Params &p, cudaStream_t st) {
  gqaw::TcMaps maps;
  const cuuint64_t D = 128, BS = (cuuint64_t)a->batch_size * a->sequence_length;
  const cuuint64_t slices = (cuuint64_t)a->batch_size * a->kv_num_heads, C = (cuuint64_t)a->capacity;
  const cuuint64_t q_dims[3] = {D, (cuuint64_t)a->num_heads, BS};
  const cuuint64_t q_str[2] = {D * 2, (cuuint64_t)a->num_heads * D * 2};
  const cuuint32_t q_box[3] = {64, (cuuint32_t)L.group, (cuuint32_t)(32 / L.group)};
  // cache as (slice, row, dim): a box that starts below row 0 reads zeros there
  const cuuint64_t c_dims[3] = {D, C, slices};
  const cuuint64_t c_str[2] = {D * 2, C * D * 2};
  const cuuint32_t c_box[3] = {64, 128, 1};
  const cuuint64_t n_dims[3] = {D, (cuuint64_t)a->kv_num_heads, BS};
  const cuuint64_t n_str[2] = {D * 2, (cuuint64_t)a->kv_num_heads * D * 2};
  const cuuint32_t n_box[3] = {64, 1, 128};
  if (!encode_map(&maps.q, p.q, 3, q_dims, q_str, q_box) ||
      !encode_map(&maps.kc, a->past_key, 3, c_dims, c_str, c_box) ||
      !encode_map(&maps.vc, a->past_value, 3, c_dims, c_str, c_box) ||
      !encode_map(&maps.kn, p.k, 3, n_dims, n_str, n_box) ||
      !encode_map(&maps.vn, a->value, 3, n_dims, n_str, n_box))
    return fail(GQAW_ECUDA, "cuTensorMapEncodeTiled failed for the multi-token kernel");
  const cudaError_t e = gqaw::launch_mma(p, L.ta, maps, (int)L.tc_grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "multi-token kernel launch");
  g_launches.fetch_add(1);
  return GQAW_OK;
}

gqaw_status run_mmad(const gqaw_step_args *a, const Launch &L, const gqaw::Params &p, cudaStream_t st) {
  gqaw::TdMaps maps;
  const cuuint64_t D = 128, BS = (cuuint64_t)a->batch_size * a->sequence_length;
  const cuuint64_t rows = (cuuint64_t)a->batch_size * a->kv_num_heads * a->capacity;
  const cuuint64_t q_dims[3] = {D, (cuuint64_t)a->num_heads, BS};
  const cuuint64_t q_str[2] = {D * 2, (cuuint64_t)a->num_heads * D * 2};
  const cuuint32_t q_box[3] = {64, (cuuint32_t)L.group, (cuuint32_t)a->sequence_length};
  const cuuint64_t c_dims[2] = {D, rows};
  const cuuint64_t c_str[1] = {D * 2};
  const cuuint32_t c_box[2] = {64, 128};
  // quantized cache: 128 one-byte codes per row, one 128 x 128 box per tile; fp16 query
  const cuuint64_t c8_str[1] = {D};
  const cuuint32_t c8_box[2] = {128, 128};
  // bf16 caches: 8-row boxes for the stores of rows moved inside the attention pass
  const cuuint32_t r8_box[2] = {64, 8};
  const bool q8 = L.quant != 0;
  const CUtensorMapDataType qt = q8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType ct = q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  std::memset(&maps.kp, 0, 4 * sizeof(maps.kp));
  if (!encode_map(&maps.q, q8 ? p.q16 : p.q, 3, q_dims, q_str, q_box, qt) ||
      !encode_map(&maps.kc, a->past_key, 2, c_dims, q8 ? c8_str : c_str, q8 ? c8_box : c_box, ct) ||
      !encode_map(&maps.vc, a->past_value, 2, c_dims, q8 ? c8_str : c_str, q8 ? c8_box : c_box, ct) ||
      (!q8 && (!encode_map(&maps.kp, a->present_key, 2, c_dims, c_str, c_box, ct) ||
               !encode_map(&maps.vp, a->present_value, 2, c_dims, c_str, c_box, ct) ||
               !encode_map(&maps.kp8, a->present_key, 2, c_dims, c_str, r8_box, ct) ||
               !encode_map(&maps.vp8, a->present_value, 2, c_dims, c_str, r8_box, ct))))
    return fail(GQAW_ECUDA, "cuTensorMapEncodeTiled failed for the small-step kernel");
  const cudaError_t e = gqaw::launch_mmad(p, L.tda, maps, (int)L.td_ctas, st);
  if (e != cudaSuccess) return cuda_fail(e, "small-step tensor-core kernel launch");
  g_launches.fetch_add(1);
  return GQAW_OK;
}

gqaw_status run_attend(const gqaw_step_args *a, const Launch &L, const gqaw::Params &p, cudaStream_t st) {
  if (L.rot_dim > 0) {
    const cudaError_t e = gqaw::launch_rotary(p, st);
    if (e != cudaSuccess) return cuda_fail(e, "rotary kernel launch");
    g_launches.fetch_add(1);
  }
  if (L.quant) {
    const cudaError_t e = gqaw::launch_quantize(p, (int)(kSms * 8), st);
    if (e != cudaSuccess) return cuda_fail(e, "quantize kernel launch");
    g_launches.fetch_add(1);
    if (L.td) return run_mmad(a, L, p, st);
    const cudaError_t e2 = gqaw::launch_attend_q8(p, L.gb, (int)L.ctas, st);
    if (e2 != cudaSuccess) return cuda_fail(e2, "attention kernel launch");
    g_launches.fetch_add(1);
    return GQAW_OK;
  }
  if (L.td) return run_mmad(a, L, p, st);
  if (L.tc) return run_mma(a, L, p, st);
  const cudaError_t e = a->dtype == GQAW_F32 ? gqaw::launch_attend_f32(p, L.gb, (int)L.ctas, st)
                                             : gqaw::launch_attend_bf16(p, L.gb, (int)L.ctas, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  g_launches.fetch_add(1);
  return GQAW_OK;
}

// Clears the step's ticket region when the workspace last served a step of another
// layout (see tickets_need_clear).
gqaw_status clear_tickets_if_needed(const gqaw_step_args *a, const Launch &L, cudaStream_t st) {
  if (!tickets_need_clear(a->workspace, L.off_tickets, L.off_partials)) return GQAW_OK;
  const cudaError_t e =
      cudaMemsetAsync(static_cast<char *>(a->workspace) + L.off_tickets, 0, L.off_partials - L.off_tickets, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (ticket region)");
  return GQAW_OK;
}

gqaw_status run_finish(const gqaw_step_args *a, const Launch &L, const gqaw::Params &p, cudaStream_t st) {
  // separate present buffers for both K and V: the copy kernel's independent jobs
  const bool separate = p.pk != p.prk && p.pv != p.prv;
  const cudaError_t e = gqaw::launch_finish(p, (int)(separate ? L.ncopy_sep : L.ncopy), st, separate);
  if (e != cudaSuccess) return cuda_fail(e, "finish kernel launch");
  g_launches.fetch_add(1);
  return GQAW_OK;
}

}  // namespace

namespace gqaw {
// Lets other translation units of the library report an error through gqaw_last_error().
void set_error(const char *msg) { t_error = msg; }

// Bytes at the start of a step's workspace that must be zero when the step starts (the
// status word, the cache-update counters and list, the tickets); 0 if the sizes are
// invalid.
size_t workspace_counter_bytes(const gqaw_step_args *args) {
  Launch L;
  if (plan_launch(args, &L) != GQAW_OK) return 0;
  return L.off_partials;
}

// A workspace was zeroed by other means than gqaw_workspace_init (see note_zeroed).
void workspace_zeroed(const void *ws, size_t bytes) { note_zeroed(ws, bytes); }
}  // namespace gqaw

extern "C" {

int64_t gqaw_resident_len(int64_t T, int64_t C, int64_t W) {
  if (T < 0 || C < 1 || W < 1 || W > C) return -1;
  if (T <= C) return T;
  const int64_t G = C - W + 1;
  return T - G * ((T - C + G - 1) / G);
}

int gqaw_rollback_exact(int64_t T, int64_t k, int64_t C, int64_t W) {
  if (k < 0 || k > T) return -1;
  const int64_t a = gqaw_resident_len(T - k, C, W), b = gqaw_resident_len(T, C, W);
  if (a < 0 || b < 0) return -1;
  return a == b - k ? 1 : 0;
}

size_t gqaw_workspace_bytes(const gqaw_step_args *args) {
  Launch L;
  if (plan_launch(args, &L) != GQAW_OK) return 0;
  return L.ws_bytes;
}

gqaw_status gqaw_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace) return fail(GQAW_EWORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(GQAW_EWORKSPACE, "workspace is not 256-byte aligned");
  if (workspace_bytes < 256) return fail(GQAW_EWORKSPACE, "workspace_bytes %zu < 256", workspace_bytes);
  const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  note_zeroed(workspace, workspace_bytes);
  return GQAW_OK;
}

gqaw_status gqa_windowed_step(const gqaw_step_args *args, void *stream) {
  Launch L;
  gqaw::Params p;
  gqaw_status s = prepare(args, &L, &p);
  if (s != GQAW_OK || args->batch_size == 0) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = clear_tickets_if_needed(args, L, st);
  if (s != GQAW_OK) return s;
  s = run_attend(args, L, p, st);
  if (s != GQAW_OK) return s;
  if (p.no_finish) return GQAW_OK;  // the attention kernel did the whole cache update
  return run_finish(args, L, p, st);
}

gqaw_status gqaw_attend(const gqaw_step_args *args, void *stream) {
  Launch L;
  gqaw::Params p;
  gqaw_status s = prepare(args, &L, &p);
  if (s != GQAW_OK || args->batch_size == 0) return s;
  s = clear_tickets_if_needed(args, L, static_cast<cudaStream_t>(stream));
  if (s != GQAW_OK) return s;
  return run_attend(args, L, p, static_cast<cudaStream_t>(stream));
}

gqaw_status gqaw_update_cache(const gqaw_step_args *args, void *stream) {
  Launch L;
  gqaw::Params p;
  gqaw_status s = prepare(args, &L, &p);
  if (s != GQAW_OK || args->batch_size == 0) return s;
  return run_finish(args, L, p, static_cast<cudaStream_t>(stream));
}

gqaw_status gqaw_device_status(void *workspace, uint32_t *flags, int reset, void *stream) {
  if (!workspace) return fail(GQAW_EWORKSPACE, "workspace is NULL");
  if (!flags) return fail(GQAW_EINVAL, "flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (reset) {
    e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  }
  if (*flags) return fail(GQAW_EDEVICE, "device status 0x%x", *flags);
  return GQAW_OK;
}

const char *gqaw_last_error(void) { return t_error.c_str(); }

uint64_t gqaw_launch_count(void) { return g_launches.load(); }

size_t gqaw_step_args_size(void) { return sizeof(gqaw_step_args); }

}  // extern "C"
