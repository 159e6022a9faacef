// gqaw_mmad.cuh -- windowed GQA attention for small steps (decode, short verify) on the
// 5th-generation tensor cores, with the keys as the MMA's M dimension.
//
// What it computes is the same as the other attention kernels: the query of token s
// (absolute position i = P + s) attends keys i - W < j <= i (onnxruntime PR #34226 "Fix
// CPU Attention causal mask for q_len=1 with past_key and kv_len > 1", Description),
// logit softcap * tanh(scale q.k / softcap) + bias[b, h, s, j] with j the absolute key
// position (PR #32419 "Specify GroupQueryAttention windowed KV cache layout contract",
// Description), keys before P from the pre-step cache rows and keys from P on from the
// step's new rows -- no staging copy (PR #31142 "[CPU] Add windowed kv cache for GQA",
// "Staging for hazardous steps"): this kernel runs before any cache row moves.
//
// Design.  A unit is (item, kv head): all S x g query rows of a step that share its
// K/V rows, at most 32, padded to NPAD = 16 or 32.  With so few query rows the usual
// orientation (query rows as M = 128) would waste most of the tensor core and leave the
// per-key work on the CUDA cores; here the contractions run transposed:
//   S^T = K Q^T      M = 128 keys of a tile, N = NPAD query rows, K = 128 dims
//   O^T += V^T P^T   M = 128 dims, N = NPAD query rows, K = 128 keys
// so one thread of the four softmax warps owns one key (a TMEM lane) and the logits of
// the unit's rows (S x g of the NPAD, rounded up to 4, 8, 16 or 32), and the fp32
// accumulator O^T lives in tensor memory (lane = head dimension).
// The online softmax keeps one reference maximum per query row, uniform over the CTA;
// it moves only when a tile's logit exceeds it by more than 2^8 (a vote through a
// reducing barrier), so the common tile needs no cross-thread reduction: each thread
// sums its own probabilities and the sums are reduced once per unit.
//
// The cache rows [lo, P) come in tiles of 128 keys by TMA (128-byte swizzle) through a
// three-stage ring; the S new rows of the step, which live in the input tensors, are
// added when the unit is finished (their logits and values are read directly), so no
// tile ever mixes the two sources.  Warp roles: four or eight softmax warps (each owning
// a quarter of the keys and half or all of the query rows), then one warp whose first
// thread is the TMA producer and one whose first thread issues the MMAs; they meet at
// mbarriers.  Persistent stream-K over the (unit, key tile) sequence, as in the decode
// kernel: a unit cut by a CTA range boundary is merged by its last contributor.
//
// Quantized caches (mobius issue #111 "GQA In-Place KV Cache: Investigation Report",
// Part 1.1, k_scale and v_scale): the TMA streams tiles of 1-byte codes (half the bytes)
// and dedicated widening warps turn each code row into an fp16 operand row of the same
// swizzled layout (int8 exactly through the fp16 mantissa, e4m3 by the hardware pair
// conversion), K into its buffer once the previous tile's S^T is done, V into one of two
// buffers once the P.V of two tiles back is done, so that widening, S^T, softmax and P.V
// of consecutive tiles overlap; the MMAs then run on fp16 operands (an fp16 copy of the
// query), the key scale is folded into the logit scale and the value scale into the
// finished rows.
//
// Every mbarrier wait is bounded; a wait that expires flags GQAW_DEV_TIMEOUT and the
// CTA winds down.  The softmax warps decide to stop only through a reducing barrier,
// so they always meet at the same named barriers.
#pragma once

#include <cuda.h>

#include <atomic>

#include "gqaw_tc.cuh"

namespace gqaw {

namespace mmad {

constexpr int kKeys = 128;                 // keys per tile (M of S^T = K Q^T)
constexpr int kD = 128;                    // head size (M of O^T = V^T P^T)
constexpr int kHalf = 16384;               // one 64-dim half of a K or V tile
constexpr int kStages = 3;
constexpr int kStageBytes = 4 * kHalf;     // K and V, two halves each
constexpr int kCodeStage = 2 * kHalf;      // quantized cache: K and V code tiles (128 x 128 bytes each)
constexpr int kK16 = kStages * kCodeStage;  // quantized cache: the widened K tile (fp16, 32 KB)
constexpr int kV16 = kK16 + 2 * kHalf;      // quantized cache: two widened V tiles (fp16, 32 KB each)
constexpr float kRescale = 8.0f;           // lazy rescale threshold (log2 units)
constexpr int kBar = 1;                    // named barrier of the softmax warps
constexpr int kNumBars = 25;
constexpr int kRow = kD * 2;               // bytes of a bf16 cache row
static_assert(kMoveStashRows <= kKeys, "a stash lies within a CTA's first tile");
static_assert(kMoveStashBytes == kMoveStashRows * 2 * kRow, "a stash holds K and V rows of head size 128");
static_assert(kV16 + 4 * kHalf == kStages * kStageBytes, "both layouts put Q at the same offset");

template <int NPAD>
struct Lay {
  static constexpr int kQHalf = NPAD * 128;                 // a 64-column half of Q or P^T
  static constexpr int kQ = kStages * kStageBytes;          // two Q buffers
  static constexpr int kP = kQ + 4 * kQHalf;                // two P^T buffers
  static constexpr int kRed = kP + 4 * kQHalf;              // float [4][NPAD]
  // The epilogue's logits of the step's own keys, float [NPAD][NPAD], live in the
  // first rows of P^T buffer 0: those rows are rewritten by every tile.
  static constexpr int kZn = kP;
  static constexpr int kFin = kRed + 4 * NPAD * 4;          // float m, l, f [3][NPAD]
  static constexpr int kBrow = kFin + 4 * NPAD * 4;         // long long [NPAD]
  static constexpr int kBars = kBrow + NPAD * 8;            // mbarriers
  static constexpr int kSlot = kBars + kNumBars * 8;        // TMEM base address
  static constexpr int kTotal = kSlot + 16;
  static constexpr int kAlloc = kTotal + 1024;              // room to align the base
  static constexpr uint32_t kCols = NPAD == 16 ? 64 : 128;  // S^T x2 and O^T
};

// Sixteen 1-byte codes (a 16-byte vector) as eight fp16 pairs, exactly.  (The general
// form is only instantiated, never run, for caches without codes.)
template <int QT>
__device__ __forceinline__ void widen16(const uint4 &u, uint32_t (&h)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = 0u;
}
template <>
__device__ __forceinline__ void widen16<GQAW_I8>(const uint4 &u, uint32_t (&h)[8]) {
  // a byte b, biased to b + 128, is the low mantissa of 1024 in fp16 (1024 + b + 128);
  // subtracting 1152 leaves b
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t wb = w[i] ^ 0x80808080u;
    uint32_t lo = __byte_perm(wb, 0x64646464u, 0x4140), hi = __byte_perm(wb, 0x64646464u, 0x4342);
    __half2 a = __hsub2(*reinterpret_cast<__half2 *>(&lo), off), b = __hsub2(*reinterpret_cast<__half2 *>(&hi), off);
    h[2 * i] = *reinterpret_cast<uint32_t *>(&a);
    h[2 * i + 1] = *reinterpret_cast<uint32_t *>(&b);
  }
}
template <>
__device__ __forceinline__ void widen16<GQAW_E4M3>(const uint4 &u, uint32_t (&h)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * i]) : "h"((uint16_t)(w[i] & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * i + 1]) : "h"((uint16_t)(w[i] >> 16)));
  }
}

// Chunks [c0, c0 + NCH) (16 codes each) of row t of a code tile (128 one-byte codes in a
// 128-byte swizzled row) into row t of an fp16 operand tile (two 64-dim halves of 128-byte
// swizzled rows, 16 KB apart); zero: write zeros (keys past the tile's valid rows).
template <int QT, int NCH = 8>
__device__ __forceinline__ void widen_row(const unsigned char *codes, unsigned char *dst, int t, bool zero, int c0 = 0) {
  const int sw = t & 7;
  uint4 u[NCH];  // all loads first: their latencies overlap
#pragma unroll
  for (int i = 0; i < NCH; ++i)
    u[i] = zero ? make_uint4(0, 0, 0, 0) : *reinterpret_cast<const uint4 *>(codes + t * 128 + (((c0 + i) ^ sw) << 4));
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = c0 + i;
    uint32_t h[8];
    widen16<QT>(u[i], h);
    unsigned char *row = dst + (c >> 2) * kHalf + t * 128;
    const int cc = (c & 3) * 2;
    *reinterpret_cast<uint4 *>(row + ((cc ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(row + (((cc + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh(x) = 1 - 2 / (e^(2x) + 1), absolute error about 1e-7.
__device__ __forceinline__ float fast_tanh(float x) {
  const float e = fast_exp2(2.8853900817779268f * fminf(fmaxf(x, -15.f), 15.f));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return fmaf(-2.f, r, 1.f);
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld<2>(uint32_t taddr, float (&v)[2]) {
  uint32_t r[2];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];\ntcgen05.wait::ld.sync.aligned;"
               : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
  v[0] = __uint_as_float(r[0]);
  v[1] = __uint_as_float(r[1]);
}
template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
  tc::tmem_ld16(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
  tc::tmem_ld32(taddr, v);
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_st<2>(uint32_t taddr, const float (&v)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
               "r"(__float_as_uint(v[1]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_st<4>(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const float (&v)[16]) {
  tc::tmem_st16(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const float (&v)[32]) {
  tc::tmem_st32(taddr, v);
}

// A unit (item, kv head) and its cache keys [lo, P) in `real` tiles of 128.
struct DUnit {
  int b, kvh;
  bool ok;
  Plan pl;
  long long lo;
  int real;
};

__device__ __forceinline__ DUnit dunit(const Params &p, long long u) {
  DUnit x;
  x.b = (int)(u / p.Nkv);
  x.kvh = (int)(u % p.Nkv);
  x.ok = plan_item(p, x.b, x.pl);
  x.lo = 0;
  x.real = 0;
  if (x.ok) {
    x.lo = x.pl.P - p.W + 1 > 0 ? x.pl.P - p.W + 1 : 0;
    x.real = (int)((x.pl.P - x.lo + kKeys - 1) / kKeys);
  }
  return x;
}

// What the kernel does with the rows of a unit's item (the same for each of its kv heads).
//  kAppend:   in place, no block reclaimed: the new rows go to [L(P), L(P) + S), which no
//             query reads, appended by the CTA holding the unit's last tile first thing.
//  kFused:    bf16 cache, and either in place with a block of seed <= kMoveStashRows
//             rows reclaimed and every surviving row [seed, L(P)) inside the window the
//             step reads, or a separate present buffer (mobius issue #111, Part 1.2,
//             "Mode A"): the mover warp writes the surviving rows of the staged tiles to
//             [0, kept) of present, and the CTA holding the unit's last tile appends the
//             new rows at [kept, L(T)) after its tiles (block compaction and append of PR
//             #31142 "[CPU] Add windowed kv cache for GQA", "Drifting layout", done inside
//             the attention pass).  With a separate present buffer nothing the step reads
//             is overwritten (no stash, no deferred rows); its surviving rows below the
//             window, which no tile holds, are left to the cache-update kernel (`below`).
//  kRegister: anything else (surviving rows below the window or a larger block in place,
//             a code cache): the item is recorded for the cache-update kernel.
enum { kAppend = 0, kFused = 1, kRegister = 2 };
struct DMove {
  int kind;
  bool sep;              // present is a separate buffer
  bool below;            // separate present: surviving rows [seed, lo_row) lie below the window
  long long seed, kept;  // rows reclaimed; rows surviving (the new rows follow them)
  long long lo_row;      // slice row of the window's first key (key position x.lo)
  long long nwin;        // keys of the window held in the cache: rows [lo_row, L(P))
};


template <int QT>
__device__ __forceinline__ DMove dmove(const Params &p, const DUnit &x) {
  DMove m;
  m.seed = x.pl.Lp + p.S - x.pl.Lt;
  m.kept = x.pl.Lt - p.S;
  m.nwin = x.pl.P - x.lo;
  m.lo_row = x.pl.Lp - m.nwin;
  const bool inplace = p.pk == p.prk && p.pv == p.prv;
  m.sep = !inplace;
  m.below = m.sep && m.kept > m.nwin;
  if (inplace && m.seed == 0)
    m.kind = kAppend;
  else if (QT == 0 && (m.sep || (m.kept >= 0 && m.kept <= m.nwin && m.seed <= kMoveStashRows)))
    m.kind = kFused;
  else
    m.kind = kRegister;
  return m;
}

// The CTA whose range holds virtual tile x (CTA c covers [c*V/G, (c+1)*V/G)).
__device__ __forceinline__ long long owner_cta(long long x, long long V, long long G) {
  return ((x + 1) * G - 1) / V;
}

// One real key tile of the CTA's sequence, as the producer and MMA threads walk it.
struct DTile {
  DUnit x;
  int lt;       // tile index within the unit
  int kc;       // index among this CTA's real tiles (ring stage, barrier phases)
  int ui;       // index among this CTA's units with real tiles (Q buffer, phases)
  bool first;   // first real tile of the unit in this CTA
  bool last;    // last one
};

struct Walker {
  long long u, ulast, tb, te, TPU;
  int lt, r1, kc, ui;
  DUnit x;
  __device__ bool next(const Params &p, DTile &t) {
    bool first = false;
    while (lt >= r1) {
      if (++u > ulast) return false;
      x = dunit(p, u);
      const long long lt0 = tb - u * TPU > 0 ? tb - u * TPU : 0;
      const long long lt1 = te - u * TPU < TPU ? te - u * TPU : TPU;
      lt = (int)lt0;
      r1 = x.ok ? (int)(lt1 < x.real ? lt1 : x.real) : 0;
      if (lt < r1) {
        ++ui;
        first = true;
      }
    }
    t.x = x;
    t.lt = lt;
    t.kc = kc++;
    t.ui = ui;
    t.first = first;
    t.last = lt + 1 == r1;
    ++lt;
    return true;
  }
};

}  // namespace mmad

// NPAD: query rows of the MMA (16 or 32); NVT: query rows the softmax warps process
// (the unit's S x g rounded up to 4, 8, 16 or 32; rows past S x g are zero); CG: column
// groups.  4 * CG softmax warps: warps w and w + 4 read the same TMEM lanes (the same
// keys, the same head dimensions) and own different query rows, NC = NVT / CG each.
// QT: 0 for bf16 caches, GQAW_I8 or GQAW_E4M3 for the codes of a quantized cache.
// Warps: 4 * CG softmax warps, 4 widening warps (quantized cache only: one per TMEM lane
// quarter; 8 for int8 codes with one column group, two per quarter, each widening one
// 64-dimension half of its rows: the int8 widening takes more arithmetic than e4m3's
// pair conversion), the TMA producer warp, the warp whose first thread issues the S^T MMAs, for
// bf16 caches the mover warp, and the warp whose first thread issues the P.V MMAs.  The two
// issuing threads sit in warps of their own: each MMA issue and each barrier wait of such a
// thread costs tens of cycles on a sub-partition shared with busy warps, and one thread
// issuing both products per tile set the pace of decode tiles.  With four column groups
// (32 query rows, softcap and bias: paced by the softmax warps) one thread issues both,
// S^T of the next tile before P.V of this one: a fifth spinning warp slowed those warps.
template <int CG, int QT>
struct Warps {
  static_assert(QT == 0 || CG <= 2, "code caches: at most two column groups");
  static constexpr int kWiden = QT == 0 ? 0 : (QT == GQAW_I8 && CG == 1 ? 8 : 4);
  static constexpr int kProducer = 4 * CG + kWiden;
  static constexpr int kMover = QT == 0 ? 1 : 0;  // bf16 caches: the warp that moves rows
  static constexpr bool kSplitMMA = CG < 4;
  static constexpr int kPV = kSplitMMA ? kProducer + 2 + kMover : kProducer + 1;
  static constexpr int kThreads = 32 * (kProducer + 2 + kMover + (kSplitMMA ? 1 : 0));
};

template <int NPAD, int NVT, int CG, int QT>
__global__ void __launch_bounds__(Warps<CG, QT>::kThreads, 1)
    mma_decode_kernel(const Params p, const TdArgs ta, const __grid_constant__ TdMaps maps) {
  using namespace mmad;
  constexpr bool kQ8 = QT != 0;
  static_assert(NVT <= NPAD && NVT % CG == 0, "processed rows within the MMA rows");
  constexpr int NC = NVT / CG;              // query rows per softmax thread
  constexpr int kSoft = 128 * CG;           // softmax threads
  constexpr int kWidenW = Warps<CG, QT>::kWiden;
  constexpr int kProducer = Warps<CG, QT>::kProducer;  // TMA producer warp; the MMA issuer is the next
  using L = Lay<NPAD>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *red = reinterpret_cast<float *>(smem + L::kRed);
  float *zn = reinterpret_cast<float *>(smem + L::kZn);
  float *fin_m = reinterpret_cast<float *>(smem + L::kFin), *fin_l = fin_m + NPAD, *fin_f = fin_l + NPAD;
  long long *brow = reinterpret_cast<long long *>(smem + L::kBrow);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
  uint64_t *full = bars, *empty = bars + 3, *s_full = bars + 6, *s_free = bars + 8;
  // p_full[2] and o_done[2] are per P^T buffer: the softmax warps may run one tile
  // ahead of the MMA thread, so a single barrier could complete two phases before the
  // MMA thread looks at it, and a parity wait cannot tell two phases apart.
  uint64_t *p_full = bars + 10, *o_done = bars + 12, *o_free = bars + 14;
  uint64_t *q_full = bars + 15, *q_free = bars + 17, *mma_done = bars + 19;
  // quantized cache: widened K tile ready, widened V tile [2] ready (both per tile parity:
  // a parity wait cannot tell apart two phases of one barrier)
  uint64_t *kconv_full = bars + 20, *vconv_full = bars + 22;
  // bf16 caches: the mover warp has written this CTA's stash (rows of its first unit whose
  // destination lies in the previous CTA's range); the softmax warps wait for it before
  // the unit's ticket
  uint64_t *stash_bar = bars + 24;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kSlot);
  __shared__ int s_abort, s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long TPU = ta.tpu, V = ta.units * TPU, G = gridDim.x, cta = blockIdx.x;
  const long long tb = cta * V / G, te = (cta + 1) * V / G;  // this CTA's virtual tiles
  const long long ufirst = tb / TPU, ulast = (te - 1) / TPU;
  const int g = p.group, S = p.S, NV = S * g;  // valid query rows of a unit

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      // codes: free once widened; bf16: once the P.V that reads V has completed and the
      // mover warp is done with the tile
      mbar_init(&empty[i], kQ8 ? 32 * kWidenW : 2);
    }
    if constexpr (!kQ8) mbar_init(stash_bar, 1);
    if constexpr (kQ8) {  // the widening warps' barriers (counts are at least 1)
      for (int i = 0; i < 2; ++i) {
        mbar_init(&kconv_full[i], 32 * kWidenW);
        mbar_init(&vconv_full[i], 32 * kWidenW);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kSoft);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_free[i], 1);
      mbar_init(&p_full[i], kSoft);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(o_free, kSoft);
    mbar_init(mma_done, Warps<CG, QT>::kSplitMMA ? 2 : 1);  // a commit from each MMA-issuing thread
    mbar_fence_init();
    s_abort = 0;
  }
  // Q and P^T rows past the unit's query rows stay zero for the whole kernel.
  for (int e = tid; e < (8 * L::kQHalf) / 16; e += blockDim.x)
    reinterpret_cast<uint4 *>(smem + L::kQ)[e] = make_uint4(0, 0, 0, 0);
  // TMEM columns: S^T (two buffers of NPAD) and O^T (NPAD); with a code cache also two
  // widened K tiles, the A operand of S^T: 128 keys (lanes) x 128 fp16 dimensions in 64
  // columns of pairs each, at columns 128 and 192
  constexpr uint32_t kTmemK = 128;
  constexpr uint32_t kTCols = kQ8 ? 256 : L::kCols;
  static_assert(3 * NPAD <= (int)kTmemK, "S^T and O^T before the K tiles");
  if (warp == 0) tc::tmem_alloc(tmem_slot, kTCols);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 2 * NPAD, tmem_k = tmem + kTmemK;
  pdl_wait();                // the previous kernel in the stream has completed

  auto stage = [&](int kc) { return smem + (kc % kStages) * (kQ8 ? kCodeStage : kStageBytes); };
  auto v16buf = [&](int kc) { return smem + kV16 + (kc & 1) * 2 * kHalf; };
  auto qbuf = [&](int ui) { return smem + L::kQ + (ui & 1) * 2 * L::kQHalf; };
  auto pbuf = [&](int kc) { return smem + L::kP + (kc & 1) * 2 * L::kQHalf; };

  if (warp == kProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first(), qpol = tc::policy_evict_last();
      Walker w{ufirst - 1, ulast, tb, te, TPU, 0, 0, 0, -1, DUnit()};
      DTile t;
      int issued = 0, qissued = -1;
      bool alive = true;
      while (alive && !*reinterpret_cast<volatile int *>(&s_abort) && w.next(p, t)) {
        const DUnit &x = t.x;
        if (t.first) {
          if (t.ui >= 2 && !mbar_wait(&q_free[t.ui & 1], ((t.ui - 2) >> 1) & 1)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[t.ui & 1], (uint32_t)(2 * NV * 128));
          tc::tma_load_3d(qbuf(t.ui), &maps.q, 0, x.kvh * g, x.b * S, &q_full[t.ui & 1], qpol);
          tc::tma_load_3d(qbuf(t.ui) + L::kQHalf, &maps.q, 64, x.kvh * g, x.b * S, &q_full[t.ui & 1], qpol);
          qissued = t.ui;
        }
        const int st = t.kc % kStages;
        if (t.kc >= kStages && !mbar_wait(&empty[st], ((t.kc / kStages) - 1) & 1)) {
          alive = false;
          break;
        }
        const int row = (int)(((long long)x.b * p.Nkv + x.kvh) * p.C + (x.lo + (long long)t.lt * kKeys - x.pl.P + x.pl.Lp));
        unsigned char *sb = stage(t.kc);
        if (kQ8) {  // one 128 x 128-byte code tile per tensor
          mbar_arrive_expect_tx(&full[st], kCodeStage);
          tc::tma_load_2d(sb, &maps.kc, 0, row, &full[st], pol);
          tc::tma_load_2d(sb + kHalf, &maps.vc, 0, row, &full[st], pol);
        } else {
          mbar_arrive_expect_tx(&full[st], kStageBytes);
          tc::tma_load_2d(sb, &maps.kc, 0, row, &full[st], pol);
          tc::tma_load_2d(sb + kHalf, &maps.kc, 64, row, &full[st], pol);
          tc::tma_load_2d(sb + 2 * kHalf, &maps.vc, 0, row, &full[st], pol);
          tc::tma_load_2d(sb + 3 * kHalf, &maps.vc, 64, row, &full[st], pol);
        }
        ++issued;
      }
      if (!alive) {
        flag(p, GQAW_DEV_TIMEOUT);
        s_abort = 1;
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (int k = issued - kStages > 0 ? issued - kStages : 0; k < issued; ++k)
        if (!mbar_wait(&full[k % kStages], (k / kStages) & 1)) flag(p, GQAW_DEV_TIMEOUT);
      for (int q = qissued - 1 > 0 ? qissued - 1 : 0; q <= qissued; ++q)
        if (q >= 0 && !mbar_wait(&q_full[q & 1], (q >> 1) & 1)) flag(p, GQAW_DEV_TIMEOUT);
    }
  } else if (warp == kProducer + 1 || warp == Warps<CG, QT>::kPV) {
    // ------------------------------------------------------------ MMA issuers
    // The first thread of warp kProducer + 1 issues S^T of every tile; the first thread of
    // warp kPV issues P.V.  They write different accumulators (S^T buffers, O^T), and
    // every order between them goes through a barrier: P.V(k) needs P(k), which the
    // softmax writes only after S^T(k) has completed, so a commit of the P.V thread also
    // covers the S^T of the same tile (the stage it freed, the last tile's Q).  A
    // tcgen05.commit tracks the MMAs of its own thread; each thread commits its own
    // barriers, and both commit mma_done before TMEM is released.
    const bool s_role = warp == kProducer + 1;
    if (lane == 0) {
      // K: K-major, Q: K-major; V^T: MN-major, P^T: K-major (fp16 operands for a quantized cache)
      constexpr uint32_t kIdescS = kQ8 ? idesc_f16_f32(kKeys, NPAD, 0, 0) : tc::idesc_bf16_f32(kKeys, NPAD, 0, 0);
      constexpr uint32_t kIdescO = kQ8 ? idesc_f16_f32(kD, NPAD, 1, 0) : tc::idesc_bf16_f32(kD, NPAD, 1, 0);
      Walker w{ufirst - 1, ulast, tb, te, TPU, 0, 0, 0, -1, DUnit()};
      auto mma_s = [&](const DTile &t) -> bool {
        if (t.first && !mbar_wait(&q_full[t.ui & 1], (t.ui >> 1) & 1)) return false;
        if (kQ8 ? !mbar_wait(&kconv_full[t.kc & 1], (t.kc >> 1) & 1)
                : !mbar_wait(&full[t.kc % kStages], (t.kc / kStages) & 1))
          return false;
        if (t.kc >= 2 && !mbar_wait(&s_free[t.kc & 1], ((t.kc - 2) >> 1) & 1)) return false;
        tc::fence_after_sync();
        // One descriptor per operand and tile; a K step adds its byte offset (over 16) to the
        // address field.  (The MMA thread shares its SM sub-partition with busy warps: every
        // instruction it saves shortens the issue of the tile's MMAs.)
        const uint64_t kd = tc::smem_desc_sw128(stage(t.kc), 16, 1024);
        const uint64_t qd = tc::smem_desc_sw128(qbuf(t.ui), 16, 1024);
        const uint32_t ds = tmem_s + (t.kc & 1) * NPAD, ka = tmem_k + (t.kc & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const int half = kk / 4, off = (kk % 4) * 32;
          const uint64_t bq = qd + (uint64_t)((half * L::kQHalf + off) >> 4);
          if (kQ8)  // K from tensor memory (buffer kc & 1): 8 columns (16 dimensions) per step
            tc::mma_bf16_ts(ds, ka + kk * 8, bq, kIdescS, kk > 0);
          else
            tc::mma_bf16_ss(ds, kd + (uint64_t)((half * kHalf + off) >> 4), bq, kIdescS, kk > 0);
        }
        tc::mma_commit(&s_full[t.kc & 1]);
        return true;
      };
      auto mma_pv = [&](const DTile &cur) -> bool {
        if (!mbar_wait(&p_full[cur.kc & 1], (cur.kc >> 1) & 1) ||
            (kQ8 && !mbar_wait(&vconv_full[cur.kc & 1], (cur.kc >> 1) & 1)) ||
            (cur.first && cur.ui >= 1 && !mbar_wait(o_free, (cur.ui - 1) & 1)))
          return false;
        tc::fence_after_sync();
        // V^T: M = dims in two 64-dim halves 16 KB apart, K = keys in 8-key groups 1 KB apart
        const uint64_t vd = tc::smem_desc_sw128(kQ8 ? v16buf(cur.kc) : stage(cur.kc) + 2 * kHalf, kHalf, 1024);
        const uint64_t pd = tc::smem_desc_sw128(pbuf(cur.kc), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc::mma_bf16_ss(tmem_o, vd + (uint64_t)((kk * 16 * 128) >> 4),
                          pd + (uint64_t)(((kk / 4) * L::kQHalf + (kk % 4) * 32) >> 4), kIdescO,
                          !(cur.first && kk == 0));
        tc::mma_commit(&o_done[cur.kc & 1]);
        if (!kQ8) tc::mma_commit(&empty[cur.kc % kStages]);
        if (cur.last) tc::mma_commit(&q_free[cur.ui & 1]);
        return true;
      };
      DTile cur, nxt;
      bool fine = true;
      if constexpr (Warps<CG, QT>::kSplitMMA) {
        if (s_role) {  // S^T of each tile, as soon as its K, Q and S^T buffer are ready
          while (fine && !*reinterpret_cast<volatile int *>(&s_abort) && w.next(p, cur)) fine = mma_s(cur);
        } else {       // P.V of each tile, as soon as its P and V are ready
          while (fine && !*reinterpret_cast<volatile int *>(&s_abort) && w.next(p, cur)) fine = mma_pv(cur);
        }
      } else {  // one thread: S^T of the next tile while this one is in softmax, then its P.V
        bool hc = w.next(p, cur);
        if (hc) fine = mma_s(cur);
        while (hc && fine && !*reinterpret_cast<volatile int *>(&s_abort)) {
          const bool hn = w.next(p, nxt);
          if (hn && !mma_s(nxt)) {
            fine = false;
            break;
          }
          fine = mma_pv(cur);
          cur = nxt;
          hc = hn;
        }
      }
      if (!fine) {
        flag(p, GQAW_DEV_TIMEOUT);
        s_abort = 1;
      }
      tc::mma_commit(mma_done);  // every MMA issued has completed before TMEM is released
      if (!mbar_wait(mma_done, 0)) flag(p, GQAW_DEV_TIMEOUT);
    }
  } else if (!kQ8 && warp == kProducer + 2) {
    // ------------------------------------------------------------ mover (bf16 caches)
    // For each staged tile of a fused unit, the tile's surviving rows go to their
    // compacted rows (destination = source row - seed): 8-row-aligned runs by tensor TMA
    // stores straight from the swizzled tile, ragged rows by the lanes (one 16-byte part of
    // a row each).  A destination in this CTA's own range was read by this CTA in an
    // earlier or the same tile, and one below the window is read by nobody; the rows whose
    // destination lies in the previous CTA's range -- the first min(seed, rows) rows of a
    // range that starts inside a unit -- go to this CTA's stash instead, for the unit's
    // last contributor.  The stage is released once the stores have read it.
    Walker w{ufirst - 1, ulast, tb, te, TPU, 0, 0, 0, -1, DUnit()};
    DTile t;
    DMove mv{};
    bool fine = true;
    const int tensor = lane >> 4, half = (lane >> 3) & 1, chunk = lane & 7;  // this lane's part of a row
    while (fine && !*reinterpret_cast<volatile int *>(&s_abort) && w.next(p, t)) {
      const int kc = t.kc, st = kc % kStages;
      if (!mbar_wait(&full[st], (kc / kStages) & 1)) {
        fine = false;
        break;
      }
      if (t.first) mv = dmove<QT>(p, t.x);
      if (mv.kind == kFused) {
        tc::fence_proxy_async_smem();  // the landed tile, as this thread saw it, to the stores
        const unsigned char *sb = stage(kc);
        const long long r0 = mv.lo_row + (long long)t.lt * kKeys;  // slice row of tile row 0
        const int nvalid = (int)(mv.nwin - (long long)t.lt * kKeys < kKeys ? mv.nwin - (long long)t.lt * kKeys : kKeys);
        const int tA = (int)(mv.seed - r0 > 0 ? mv.seed - r0 : 0);  // rows below tA are reclaimed
        const bool stash = !mv.sep && t.first && t.lt > 0;         // in place, the range starts inside the unit
        const int nst = stash ? (int)(mv.seed < nvalid ? mv.seed : nvalid) : 0;
        const long long grow0 = ((long long)t.x.b * p.Nkv + t.x.kvh) * p.C + r0 - mv.seed;
        auto part = [&](int r) {  // this lane's 16 bytes of tile row r (128-byte swizzle)
          return *reinterpret_cast<const uint4 *>(sb + tensor * 2 * kHalf + half * kHalf + r * 128 +
                                                  ((chunk ^ (r & 7)) << 4));
        };
        if (stash) {
          unsigned char *dst = p.stash + (size_t)cta * kMoveStashBytes;
          for (int r = tA; r < nst; ++r)
            *reinterpret_cast<uint4 *>(dst + (size_t)r * 2 * kRow + tensor * kRow + half * 128 + chunk * 16) = part(r);
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(stash_bar);
        }
        const int lo = tA > nst ? tA : nst, hi = nvalid;
        if (hi > lo) {
          unsigned char *gb = static_cast<unsigned char *>(tensor ? p.prv : p.prk);
          auto ragged = [&](int r) {
            *reinterpret_cast<uint4 *>(gb + (size_t)(grow0 + r) * kRow + half * 128 + chunk * 16) = part(r);
          };
          if (lo == 0 && hi == kKeys) {  // the whole tile: one 128-row box per half of K and V
            if (lane < 4)
              tc::tma_store_2d((lane >> 1) ? &maps.vp : &maps.kp, (lane & 1) * 64, (int)grow0,
                               sb + (lane >> 1) * 2 * kHalf + (lane & 1) * kHalf);
          } else {
            const int c0 = (lo + 7) & ~7, c1 = hi & ~7;  // 8-row-aligned run [c0, c1)
            if (c1 > c0) {
              for (int i = lane; i < (c1 - c0) / 2; i += 32) {  // (c1 - c0) / 8 boxes x 4 halves
                const int rr = c0 + (i >> 2) * 8, tn = (i >> 1) & 1, hf = i & 1;
                tc::tma_store_2d(tn ? &maps.vp8 : &maps.kp8, hf * 64, (int)(grow0 + rr),
                                 sb + tn * 2 * kHalf + hf * kHalf + rr * 128);
              }
              for (int r = lo; r < c0; ++r) ragged(r);
              for (int r = c1; r < hi; ++r) ragged(r);
            } else {
              for (int r = lo; r < hi; ++r) ragged(r);
            }
          }
          tc::bulk_commit();
          tc::bulk_wait_read();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!fine) {
      flag(p, GQAW_DEV_TIMEOUT);
      s_abort = 1;
    }
    tc::bulk_commit();
    tc::bulk_wait_all();  // every store of this CTA is performed before it exits
  } else if (warp >= 4 * CG) {
    // ------------------------------------------------------------ widening warps
    if constexpr (kQ8) {
      // Thread i (lane i % 32 of lane quarter i / 32) widens row i of each code tile: K(k)
      // into its lane of TMEM K buffer k & 1 (the A operand of S^T) once S^T of tile k - 2
      // is done with it, V(k) into fp16 buffer k & 1 in shared memory once P.V of tile k - 2
      // is done (keys past P as zeros).  Each wait is for a phase the barrier can have
      // reached only after the one these warps saw a tile earlier (S^T(k) needs K(k)).
      constexpr int kParts = kWidenW / 4;      // threads per row (1 or 2)
      constexpr int kChunks = 8 / kParts;      // 16-code chunks of a row per thread
      const int i0 = (warp & 3) * 32 + lane;  // key row = TMEM lane of this warp's quarter
      const int c0 = (warp - 4 * CG) / 4 * kChunks;
      const uint32_t k_lane = tmem_k + ((uint32_t)((warp & 3) * 32) << 16);
      Walker w{ufirst - 1, ulast, tb, te, TPU, 0, 0, 0, -1, DUnit()};
      DTile t;
      bool fine = true;
      while (fine && !*reinterpret_cast<volatile int *>(&s_abort) && w.next(p, t)) {
        const int kc = t.kc;
        const long long j0 = t.x.lo + (long long)t.lt * kKeys;
        const int nvalid = (int)(t.x.pl.P - j0 < kKeys ? t.x.pl.P - j0 : kKeys);
        fine = mbar_wait(&full[kc % kStages], (kc / kStages) & 1);
        if (fine && kc >= 2) fine = mbar_wait(&s_full[kc & 1], ((kc - 2) >> 1) & 1);
        tc::fence_after_sync();
        {
          const unsigned char *codes = stage(kc) + i0 * 128;
          uint4 u[kChunks];  // all loads first: their latencies overlap
#pragma unroll
          for (int i = 0; i < kChunks; ++i)
            u[i] = *reinterpret_cast<const uint4 *>(codes + (((c0 + i) ^ (i0 & 7)) << 4));
#pragma unroll
          for (int i = 0; i < kChunks; i += 2) {  // 16 codes -> 8 columns of fp16 pairs, dimension 2j low
            uint32_t h[16], h0[8], h1[8];
            widen16<QT>(u[i], h0);
            widen16<QT>(u[i + 1], h1);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              h[j] = h0[j];
              h[8 + j] = h1[j];
            }
            tc::tmem_st16_async(k_lane + (uint32_t)((kc & 1) * 64 + (c0 + i) * 8), h);
          }
          tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        mbar_arrive(&kconv_full[kc & 1]);
        if (fine && kc >= 2) fine = mbar_wait(&o_done[kc & 1], ((kc - 2) >> 1) & 1);
        tc::fence_after_sync();
        widen_row<QT, kChunks>(stage(kc) + kHalf, v16buf(kc), i0, i0 >= nvalid, c0);
        tc::fence_proxy_async_smem();
        mbar_arrive(&vconv_full[kc & 1]);
        mbar_arrive(&empty[kc % kStages]);  // both code tiles of this stage are widened
      }
      if (!fine) {
        flag(p, GQAW_DEV_TIMEOUT);
        s_abort = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = tid & 127;       // key of a tile (S^T lane) and head dimension (O^T lane)
    const int col0 = (tid >> 7) * NC;  // first query row of this thread's column group
    const int wq = warp & 3;       // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
    const __nv_bfloat16 *qin = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *kin = static_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *vin = static_cast<const __nv_bfloat16 *>(p.v);
    const bool plain = p.capmul == 0.f && p.bias == nullptr;  // logits need only the scale
    // a quantized cache's key scale joins the logit scale; its value scale multiplies the
    // finished rows
    const float qs = kQ8 ? p.qscale * *p.ks : p.qscale;
    const float vsc = kQ8 ? *p.vs : 1.f;
    int kc = 0, ui = 0;
    bool stop = false;
    for (long long u = ufirst; u <= ulast && !stop; ++u) {
      const DUnit x = dunit(p, u);
      const long long lt0 = tb - u * TPU > 0 ? tb - u * TPU : 0;
      const long long lt1 = te - u * TPU < TPU ? te - u * TPU : TPU;
      if (!x.ok) {  // every CTA touching the unit skips it: no ticket, no output
        if (lt0 == 0 && x.kvh == 0 && tid == 0) flag(p, GQAW_DEV_BAD_SEQLEN);
        continue;
      }
      const int r1 = (int)(lt1 < x.real ? lt1 : x.real);
      const int nt = r1 > (int)lt0 ? r1 - (int)lt0 : 0;  // real tiles here
      const int fx = x.real > 0 ? x.real - 1 : 0;       // the tile that adds the new keys
      const bool has_fix = lt0 <= fx && fx < lt1;
      const DMove mv = dmove<QT>(p, x);
      const long long P = x.pl.P;
      if (lt0 == 0 && x.kvh == 0 && tid == 0) {
        if (p.resident_out) p.resident_out[x.b] = (int32_t)x.pl.Lt;
        if (mv.kind == kRegister || mv.below) {
          if (p.no_finish)  // the host ruled this out: no cache-update kernel follows
            flag(p, GQAW_DEV_INTERNAL);
          else
            p.move_list[atomicAdd(p.move_count, 1u)] = mv.kind == kRegister ? x.b : (x.b | kListBelowOnly);
        }
      }
      // present rows [r_begin, r_end) <- the new rows r - kept (K and V), all softmax threads
      auto append = [&](long long r_begin, long long r_end) {
        constexpr int kRowB = kQ8 ? kD : 2 * kD, kVecs = kRowB / 16;  // row bytes, 16-byte vectors
        const int n = r_end > r_begin ? (int)(r_end - r_begin) : 0;
        for (int e = tid; e < 2 * n * kVecs; e += kSoft) {
          const int tensor = e / (n * kVecs), rem = e % (n * kVecs), rr = rem / kVecs, vec = rem % kVecs;
          const long long r = r_begin + rr;
          const size_t in_row = ((size_t)x.b * S + (size_t)(r - mv.kept)) * p.Nkv + x.kvh;
          const size_t out_row = ((size_t)x.b * p.Nkv + x.kvh) * (size_t)p.C + (size_t)r;
          reinterpret_cast<uint4 *>(static_cast<char *>(tensor ? p.prv : p.prk) + out_row * kRowB)[vec] =
              reinterpret_cast<const uint4 *>(static_cast<const char *>(tensor ? p.v : p.k) + in_row * kRowB)[vec];
        }
      };
      // append the new rows at L(P) + s (kept = L(P)): no query of this step reads them
      if (has_fix && mv.kind == kAppend) append(mv.kept, x.pl.Lt);
      for (int n = tid; n < NVT; n += kSoft)  // rows past S x g: the item's first bias row
        brow[n] = !p.bias ? 0
                          : (long long)x.b * p.bsb +
                                (n < NV ? (long long)(x.kvh * g + n % g) * p.bsh + (long long)(n / g) * p.bss : 0);
      named_barrier(kBar, kSoft);

      // Units of at most 16 query rows of a bf16 cache: what the unit's epilogue needs of
      // the step's own rows is loaded now, so that its round trip (thousands of cycles on a
      // loaded memory system) overlaps the unit's key tiles instead of lengthening the
      // epilogue, which holds up the next unit (small-slack decode 8.6 -> 7.9 us, verify4
      // 0.1024 -> 0.1005 ms; with code caches the e4m3 decode measured 8% slower: registers
      // held across the unit).  For the logits of the own keys, one warp per query row and
      // four dimensions per lane: this lane's dimensions of the first kKH key rows and of
      // its warp's query rows, and the bias of the (row, key) pair whose sum the lane will
      // hold; for their values, this thread's dimension t of the first kKH value rows.
      constexpr bool kHoist = NVT <= 16 && QT == 0;
      constexpr int kSW = kSoft / 32, kRW = (NVT + kSW - 1) / kSW, kRP = (kRW + 1) / 2;
      constexpr int kKH = NVT < 8 ? NVT : 8;  // own keys held: S <= NVT
      const int sw = tid >> 5;
      auto load_key = [&](int s2) {  // this lane's four dimensions of key row s2
        const size_t krow = ((size_t)x.b * S + (s2 < S ? s2 : S - 1)) * p.Nkv + x.kvh;
        return *reinterpret_cast<const uint2 *>(kin + krow * kD + 4 * lane);
      };
      auto load_query = [&](int r) {  // this lane's four dimensions of the warp's row r
        const int n = sw + r * kSW, nn = n < NV ? n : NV - 1;
        return *reinterpret_cast<const uint2 *>(qin + (((size_t)x.b * S + nn / g) * p.Nq + x.kvh * g + nn % g) * kD +
                                                 4 * lane);
      };
      auto load_bias = [&](int rp, int s0) {  // lane 2v: pair v = (row 2 rp + v / 8, key s0 + v % 8)
        const int n = sw + (2 * rp + (lane >> 4)) * kSW, s2 = s0 + ((lane >> 1) & 7);
        return p.bias && n < NV && s2 < S ? __ldg(p.bias + brow[n] + P + s2) : 0.f;
      };
      auto load_value = [&](int s2) {  // dimension t of value row s2
        return __bfloat162float(vin[(((size_t)x.b * S + (s2 < S ? s2 : S - 1)) * p.Nkv + x.kvh) * kD + t]);
      };
      uint2 hk[kKH], hq[kRW];
      float hv[kKH], hb[kRP];
      if (kHoist && has_fix) {
#pragma unroll
        for (int j = 0; j < kKH; ++j) {
          hk[j] = load_key(j);
          hv[j] = load_value(j);
        }
#pragma unroll
        for (int r = 0; r < kRW; ++r) hq[r] = load_query(r);
#pragma unroll
        for (int rp = 0; rp < kRP; ++rp) hb[rp] = load_bias(rp, 0);
      }

      // per query row of this thread: the reference maximum (uniform over the CTA) and
      // this thread's share of the softmax denominator
      float m_ref[NC], lsum[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        m_ref[i] = -INFINITY;
        lsum[i] = 0.f;
      }
      // Bias of this thread's key for its rows, fetched one tile ahead.  Keys past P read
      // a column that exists (P - 1): their logits are masked anyway.
      float bnext[NC];
      auto fetch_bias = [&](int lt_) {
        const long long j0_ = x.lo + (long long)lt_ * kKeys;
        const int nv_ = (int)(P - j0_ < kKeys ? P - j0_ : kKeys);
        const long long col = j0_ + (t < nv_ ? t : nv_ - 1);
#pragma unroll
        for (int i = 0; i < NC; ++i) bnext[i] = __ldg(p.bias + brow[col0 + i] + col);
      };
      // ... and brought into L2 three tiles ahead of that: under a full memory system a DRAM
      // load can take longer than a tile, and the softmax would wait for it
      auto prefetch_bias = [&](int lt_) {
        const long long j0_ = x.lo + (long long)lt_ * kKeys;
        const int nv_ = (int)(P - j0_ < kKeys ? P - j0_ : kKeys);
        const long long col = j0_ + (t < nv_ ? t : nv_ - 1);
#pragma unroll
        for (int i = 0; i < NC; ++i) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.bias + brow[col0 + i] + col));
      };
      if (p.bias && nt > 0) {
        fetch_bias((int)lt0);
        for (int l = (int)lt0 + 1; l < r1 && l <= (int)lt0 + 2; ++l) prefetch_bias(l);
      }
      for (int lt = (int)lt0; lt < r1; ++lt, ++kc) {
        const long long j0 = x.lo + (long long)lt * kKeys;
        const int nvalid = (int)(P - j0 < kKeys ? P - j0 : kKeys);
        // Key t (a cache key, so before every query) is in token s's window iff
        // t >= P + s - W + 1 - j0; rows are token-major, so the rows that see key t are
        // n < nlim.
        const int wbase = (int)(P - p.W + 1 - j0);  // <= 0
        const int nlim = (t < nvalid ? min(t - wbase + 1, S) * g : 0) - col0;
        float bv[NC];
        if (p.bias) {
#pragma unroll
          for (int i = 0; i < NC; ++i) bv[i] = bnext[i];
          if (lt + 1 < r1) fetch_bias(lt + 1);
          if (lt + 3 < r1) prefetch_bias(lt + 3);
        }
        bool ok = mbar_wait(&s_full[kc & 1], (kc >> 1) & 1);
        tc::fence_after_sync();
        float z[NC];
        tmem_ld<NC>(tmem_s + (kc & 1) * NPAD + col0 + lane_off, z);
        tc::fence_before_sync();
        mbar_arrive(&s_free[kc & 1]);
        bool exceed = false;
        if (plain) {
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            z[i] = i < nlim ? z[i] * qs : -INFINITY;
            exceed |= z[i] > m_ref[i] + kRescale;
          }
        } else {
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            float v = z[i] * qs;
            if (p.capmul != 0.f) v = p.capmul * fast_tanh(v);
            if (p.bias) v = fmaf(p.biasmul, bv[i], v);
            z[i] = i < nlim ? v : -INFINITY;
            exceed |= z[i] > m_ref[i] + kRescale;
          }
        }
        // one vote per tile: a logit above its row's reference, or a wait that expired
        const bool fail = !ok || *reinterpret_cast<volatile int *>(&s_abort);
        const bool any = named_barrier_or(kBar, kSoft, exceed || fail);
        if (any && named_barrier_or(kBar, kSoft, fail)) {
          stop = true;
          break;
        }
        // P^T buffer kc & 1 is free once the P.V of tile kc - 2 has completed
        if (kc >= 2) ok = mbar_wait(&o_done[kc & 1], ((kc - 2) >> 1) & 1);
        tc::fence_after_sync();
        if (any) {
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            float mx = z[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[wq * NPAD + col0 + i] = mx;
          }
          named_barrier(kBar, kSoft);
          float alpha[NC];
          bool resc = false;
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            const int n = col0 + i;
            const float mt = fmaxf(fmaxf(red[n], red[NPAD + n]), fmaxf(red[2 * NPAD + n], red[3 * NPAD + n]));
            alpha[i] = 1.f;
            if (mt > m_ref[i] + kRescale) {
              alpha[i] = m_ref[i] == -INFINITY ? 0.f : fast_exp2(m_ref[i] - mt);
              m_ref[i] = mt;
              lsum[i] *= alpha[i];
              resc = true;
            }
          }
          // O^T holds earlier tiles of this unit: rescale this group's columns (the
          // decision is per column group, uniform within the group's warps)
          if (resc && lt > (int)lt0) {
            if (!mbar_wait(&o_done[(kc - 1) & 1], ((kc - 1) >> 1) & 1)) ok = false;
            tc::fence_after_sync();
            float o[NC];
            tmem_ld<NC>(tmem_o + col0 + lane_off, o);
#pragma unroll
            for (int i = 0; i < NC; ++i) o[i] *= alpha[i];
            tmem_st<NC>(tmem_o + col0 + lane_off, o);
          }
        }
        // probabilities (bf16, fp16 with a quantized cache) into P^T: row n, key t,
        // 128-byte swizzled K-major
        {
          const int half = t >> 6, c = (t & 63) >> 3;
          unsigned char *pb = pbuf(kc) + half * L::kQHalf + (t & 7) * 2;
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            const int n = col0 + i;
            if (n < NV) {
              const float pr = fast_exp2(z[i] - (m_ref[i] == -INFINITY ? 0.f : m_ref[i]));
              lsum[i] += pr;
              if (kQ8)
                *reinterpret_cast<__half *>(pb + n * 128 + ((c ^ (n & 7)) << 4)) = __float2half_rn(pr);
              else
                *reinterpret_cast<__nv_bfloat16 *>(pb + n * 128 + ((c ^ (n & 7)) << 4)) = __float2bfloat16_rn(pr);
            }
          }
        }
        // keys past P in the tile: their V rows must be finite (0 * NaN is NaN)
        if (!kQ8 && nvalid < kKeys) {
          if (!mbar_wait(&full[kc % kStages], (kc / kStages) & 1)) ok = false;
          unsigned char *vb = stage(kc) + 2 * kHalf;
          for (int e = tid; e < (kKeys - nvalid) * 16; e += kSoft) {
            const int row = nvalid + e / 16, part = e % 16;
            *reinterpret_cast<uint4 *>(vb + (part / 8) * kHalf + row * 128 + (part % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        if (!ok) {
          flag(p, GQAW_DEV_TIMEOUT);
          s_abort = 1;
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        mbar_arrive(&p_full[kc & 1]);
      }
      if (stop) break;
      named_barrier(kBar, kSoft);  // every thread is done with the last tile's maxima in red
      if (has_fix && mv.kind == kFused) {
        // The new rows at [kept, L(T)), now that this CTA has read its tiles: the rows in
        // its own range (from a_fix on) or below the window; those in an earlier CTA's
        // range are written by the unit's last contributor.
        if (mv.sep) {  // nothing the step reads is overwritten
          append(mv.kept > 0 ? mv.kept : 0, x.pl.Lt);
        } else {
          const long long a_fix = mv.lo_row + (long long)lt0 * kKeys;
          append(mv.kept, x.pl.Lt < mv.lo_row ? x.pl.Lt : mv.lo_row);
          append(mv.kept > a_fix ? mv.kept : a_fix, x.pl.Lt);
        }
      }

      // ---- the unit's state in this CTA: O^T (TMEM), reference maxima, sums
      bool ok = true;
      if (nt > 0) ok = mbar_wait(&o_done[(kc - 1) & 1], ((kc - 1) >> 1) & 1);
      tc::fence_after_sync();
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        float v = lsum[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[wq * NPAD + col0 + i] = v;
        if (t == 0) fin_m[col0 + i] = m_ref[i];
      }
      if (named_barrier_or(kBar, kSoft, !ok)) {
        flag(p, GQAW_DEV_TIMEOUT);
        break;
      }
      if (has_fix) {
        // logits of the S new keys (the step's own rows) for every query row
        if constexpr (kHoist) {
          // per pair of the warp's rows and eight keys, sixteen partial dot products per
          // lane, summed over the warp by halving exchanges (lanes 2v and 2v + 1 end with
          // the sum of pair v); the first eight keys were loaded with the unit
          for (int s0 = 0; s0 < S; s0 += 8) {
            uint2 kk[8];
            float bz[kRP];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              kk[j] = s0 == 0 ? (j < kKH ? hk[j < kKH ? j : 0] : make_uint2(0u, 0u)) : load_key(s0 + j);
#pragma unroll
            for (int rp = 0; rp < kRP; ++rp) bz[rp] = s0 == 0 ? hb[rp] : load_bias(rp, s0);
#pragma unroll
            for (int rp = 0; rp < kRP; ++rp) {
              float a[16];
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * rp + rr;
                float qf[4] = {0.f, 0.f, 0.f, 0.f};
                if (r < kRW && sw + r * kSW < NV) {
                  const uint2 qw = hq[r < kRW ? r : 0];
                  qf[0] = __uint_as_float(qw.x << 16);
                  qf[1] = __uint_as_float(qw.x & 0xffff0000u);
                  qf[2] = __uint_as_float(qw.y << 16);
                  qf[3] = __uint_as_float(qw.y & 0xffff0000u);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float kf[4] = {__uint_as_float(kk[j].x << 16), __uint_as_float(kk[j].x & 0xffff0000u),
                                       __uint_as_float(kk[j].y << 16), __uint_as_float(kk[j].y & 0xffff0000u)};
                  a[rr * 8 + j] = fmaf(qf[3], kf[3], fmaf(qf[2], kf[2], fmaf(qf[1], kf[1], qf[0] * kf[0])));
                }
              }
              // halving exchanges: keep the half of the values named by this lane's bit
#pragma unroll
              for (int w = 8, o = 16; w >= 1; w >>= 1, o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                  const float send = up ? a[i] : a[w + i], keep = up ? a[w + i] : a[i];
                  a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
              }
              const float dot = a[0] + __shfl_xor_sync(0xffffffffu, a[0], 1);
              const int n = sw + (2 * rp + (lane >> 4)) * kSW, s2 = s0 + ((lane >> 1) & 7);
              if ((lane & 1) == 0 && n < NV && s2 < S) {
                const int sn = n / g;
                float zz = -INFINITY;
                if (s2 <= sn && s2 - sn > -p.W) {
                  zz = dot * qs;
                  if (p.capmul != 0.f) zz = p.capmul * fast_tanh(zz);
                  if (p.bias) zz = fmaf(p.biasmul, bz[rp], zz);
                }
                zn[n * NPAD + s2] = zz;
              }
            }
          }
        } else {
          for (int e = tid; e < NV * S; e += kSoft) {
            const int n = e / S, s2 = e % S, sn = n / g;
            const int h = x.kvh * g + n % g;
            float zz = -INFINITY;
            if (s2 <= sn && s2 - sn > -p.W) {
              const uint4 *qr = reinterpret_cast<const uint4 *>(qin + (((size_t)x.b * S + sn) * p.Nq + h) * kD);
              const size_t krow = ((size_t)x.b * S + s2) * p.Nkv + x.kvh;
              float dot = 0.f;
              if (kQ8) {  // 16 key codes per vector
                const uint4 *kr = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(p.k) + krow * kD);
#pragma unroll 4
                for (int vv = 0; vv < kD / 16; ++vv) {
                  float qa[16];
                  Elem<__nv_bfloat16>::unpack(qr[2 * vv], qa);
                  Elem<__nv_bfloat16>::unpack(qr[2 * vv + 1], qa + 8);
                  const uint4 ku = kr[vv];
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const float2 k2 = QT == GQAW_I8 ? Pairs<CodeI8>::get(ku, j) : Pairs<CodeE4M3>::get(ku, j);
                    dot = fmaf(qa[2 * j], k2.x, dot);
                    dot = fmaf(qa[2 * j + 1], k2.y, dot);
                  }
                }
              } else {
                const uint4 *kr = reinterpret_cast<const uint4 *>(kin + krow * kD);
#pragma unroll 8
                for (int vv = 0; vv < kD / 8; ++vv) {
                  float qa[8], ka[8];
                  Elem<__nv_bfloat16>::unpack(qr[vv], qa);
                  Elem<__nv_bfloat16>::unpack(kr[vv], ka);
#pragma unroll
                  for (int i = 0; i < 8; ++i) dot = fmaf(qa[i], ka[i], dot);
                }
              }
              zz = dot * qs;
              if (p.capmul != 0.f) zz = p.capmul * fast_tanh(zz);
              if (p.bias) zz = fmaf(p.biasmul, p.bias[brow[n] + P + s2], zz);
            }
            zn[n * NPAD + s2] = zz;
          }
        }
        named_barrier(kBar, kSoft);
        for (int n = tid; n < NV; n += kSoft) {
          const float m0 = fin_m[n];
          float mn = m0;
          for (int s2 = 0; s2 < S; ++s2) mn = fmaxf(mn, zn[n * NPAD + s2]);
          const float f = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mn);
          float l = (red[n] + red[NPAD + n] + red[2 * NPAD + n] + red[3 * NPAD + n]) * f;
          for (int s2 = 0; s2 < S; ++s2) {
            const float pz = fast_exp2(zn[n * NPAD + s2] - mn);
            zn[n * NPAD + s2] = pz;
            l += pz;
          }
          fin_m[n] = mn;
          fin_l[n] = l;
          fin_f[n] = f;
        }
      } else {
        for (int n = tid; n < NV; n += kSoft) {
          fin_l[n] = red[n] + red[NPAD + n] + red[2 * NPAD + n] + red[3 * NPAD + n];
          fin_f[n] = 1.f;
        }
      }
      named_barrier(kBar, kSoft);

      // ---- this thread's head dimension d = t of its query rows
      float o[NC];
      if (nt > 0) {
        tmem_ld<NC>(tmem_o + col0 + lane_off, o);
        tc::fence_before_sync();
        mbar_arrive(o_free);  // O^T may be overwritten by the next unit
        ++ui;
      } else {
#pragma unroll
        for (int i = 0; i < NC; ++i) o[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < NC; ++i) o[i] *= col0 + i < NV ? fin_f[col0 + i] : 0.f;
      if (has_fix) {
        // the step's own value rows, dimension t, eight rows per batch of independent loads
        // (a quantized cache's value codes, in code units like the accumulator; with kHoist
        // the first kKH were loaded with the unit)
        const size_t vbase = ((size_t)x.b * S * p.Nkv + x.kvh) * kD + t;
        for (int s0 = 0; s0 < S; s0 += 8) {
          float vv[8];
          if constexpr (kHoist) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              vv[j] = s0 == 0 ? (j < kKH ? hv[j < kKH ? j : 0] : 0.f) : (s0 + j < S ? load_value(s0 + j) : 0.f);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const size_t at = vbase + (size_t)(s0 + j) * p.Nkv * kD;
              if (s0 + j >= S)
                vv[j] = 0.f;
              else if (QT == GQAW_I8)
                vv[j] = (float)static_cast<const int8_t *>(p.v)[at];
              else if (QT == GQAW_E4M3)
                vv[j] = Pairs<CodeE4M3>::get(make_uint4(static_cast<const unsigned char *>(p.v)[at], 0, 0, 0), 0).x;
              else
                vv[j] = __bfloat162float(vin[at]);
            }
          }
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            const int n = col0 + i;
            if (n < NV) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (s0 + j < S) o[i] = fmaf(zn[n * NPAD + s0 + j], vv[j], o[i]);
            }
          }
        }
      }
      const long long cf = owner_cta(u * TPU, V, G), cl = owner_cta(u * TPU + TPU - 1, V, G);
      if (cf == cl) {
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int n = col0 + i;
          if (n < NV) {
            const int h = x.kvh * g + n % g;
            const size_t orow = ((size_t)x.b * S + n / g) * p.Nq + h;
            out[orow * kD + t] = __float2bfloat16_rn(sink_divide(o[i], fin_l[n], fin_m[n], sink_log2(p, h)) * vsc);
          }
        }
      } else {
        const int slot = u == ufirst ? 0 : 1;  // only a CTA's first and last unit can be shared
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int n = col0 + i;
          if (n < NV) {
            float *part = p.partials + ((cta * 2 + slot) * NPAD + n) * (kD + 2);
            part[t] = o[i];
            if (t == 0) {
              part[kD] = fin_m[n];
              part[kD + 1] = fin_l[n];
            }
          }
        }
        named_barrier(kBar, kSoft);
        if (tid == 0) {
          // a range starting inside a fused unit stashed rows for the last contributor
          if (mv.kind == kFused && !mv.sep && lt0 > 0 && nt > 0 && !mbar_wait(stash_bar, 0))
            flag(p, GQAW_DEV_TIMEOUT);
          __threadfence();
          s_last = atomicAdd(&p.tickets[u], 1u) == (unsigned)(cl - cf);
        }
        named_barrier(kBar, kSoft);
        if (s_last) {
          // merge the contributors' partial states, all of this thread's rows at once
          // (independent loads: one round trip per contributor, not one per row)
          __threadfence();
          float M[NC], Lsum[NC], A[NC];
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            M[i] = -INFINITY;
            Lsum[i] = 0.f;
            A[i] = 0.f;
          }
          for (long long c = cf; c <= cl; ++c) {
            const int sl = u == c * V / G / TPU ? 0 : 1;
            const float *part = p.partials + ((c * 2 + sl) * NPAD + col0) * (kD + 2);
#pragma unroll
            for (int i = 0; i < NC; ++i)
              if (col0 + i < NV) M[i] = fmaxf(M[i], __ldcg(part + i * (kD + 2) + kD));
          }
          for (long long c = cf; c <= cl; ++c) {
            const int sl = u == c * V / G / TPU ? 0 : 1;
            const float *part = p.partials + ((c * 2 + sl) * NPAD + col0) * (kD + 2);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
              if (col0 + i < NV) {
                const float mc = __ldcg(part + i * (kD + 2) + kD);
                const float lc = __ldcg(part + i * (kD + 2) + kD + 1);
                const float ac = __ldcg(part + i * (kD + 2) + t);
                const float f = mc == -INFINITY ? 0.f : exp2f(mc - M[i]);  // -inf: no visible key
                Lsum[i] = fmaf(f, lc, Lsum[i]);
                A[i] = fmaf(f, ac, A[i]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            const int n = col0 + i;
            if (n < NV) {
              const int h = x.kvh * g + n % g;
              const size_t orow = ((size_t)x.b * S + n / g) * p.Nq + h;
              out[orow * kD + t] = __float2bfloat16_rn(sink_divide(A[i], Lsum[i], M[i], sink_log2(p, h)) * vsc);
            }
          }
          if (mv.kind == kFused && !mv.sep) {
            // Every contributor has read its tiles: write the rows they left for the last
            // one -- each later contributor's stash (the first min(seed, rows) rows of its
            // range, moved down by seed) and the new rows in an earlier range than the
            // appending CTA's.
            for (long long c = cf + 1; c <= cl; ++c) {
              const long long lt0c = c * V / G - u * TPU;  // >= 1: c starts inside the unit
              if (lt0c >= x.real) continue;                // no key tile of the unit in c
              const long long ac = mv.lo_row + lt0c * kKeys;
              const long long nv = mv.nwin - lt0c * kKeys < kKeys ? mv.nwin - lt0c * kKeys : kKeys;
              const int nst = (int)(mv.seed < nv ? mv.seed : nv);
              const unsigned char *src = p.stash + (size_t)c * kMoveStashBytes;
              const size_t grow0 = ((size_t)x.b * p.Nkv + x.kvh) * (size_t)p.C + (size_t)(ac - mv.seed);
              for (int e = tid; e < nst * 32; e += kSoft) {  // 32 parts of 16 bytes per row (K and V)
                const int r = e >> 5, part = e & 31, tn = part >> 4, off = (part & 15) * 16;
                *reinterpret_cast<uint4 *>(static_cast<char *>(tn ? p.prv : p.prk) + (grow0 + r) * kRow + off) =
                    __ldcg(reinterpret_cast<const uint4 *>(src + (size_t)r * 2 * kRow + tn * kRow + off));
              }
            }
            const long long cfix = owner_cta(u * TPU + fx, V, G);
            const long long lt0f = cfix * V / G - u * TPU > 0 ? cfix * V / G - u * TPU : 0;
            const long long a_fix = mv.lo_row + lt0f * kKeys;
            append(mv.kept > mv.lo_row ? mv.kept : mv.lo_row, a_fix < x.pl.Lt ? a_fix : x.pl.Lt);
          }
          if (tid == 0) p.tickets[u] = 0u;  // ready for the next step
        }
      }
      named_barrier(kBar, kSoft);  // scratch (fin, zn, brow) is reused by the next unit
    }
    if (stop) flag(p, GQAW_DEV_TIMEOUT);
  }

  // release tensor memory: every MMA has completed (MMA thread) and every tcgen05.ld of
  // the softmax warps is complete (their loads wait in the same statement)
  tc::fence_before_sync();
  __syncthreads();
  pdl_launch_dependents();  // every role of this CTA is done: the cache update may be launched
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTCols);
  }
}

// One CTA per SM: a persistent grid.  The processed query rows (4, 8, 16 or 32) and the
// MMA rows (16 or 32) follow S x group; eight softmax warps from 8 rows on.
template <int QT>
cudaError_t launch_mmad_t(const Params &p, const TdArgs &ta, const TdMaps &maps, int max_ctas, cudaStream_t stream) {
  using mmad::Lay;
  constexpr int kMaxDevices = 64;
  static std::atomic<int> sms_cache[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = dev < kMaxDevices ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
  if (sms <= 0) {
    e = cudaFuncSetAttribute(mma_decode_kernel<16, 4, 2, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<16>::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mma_decode_kernel<16, 8, 2, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<16>::kAlloc);
    if (e != cudaSuccess) return e;
    if constexpr (QT == GQAW_I8) {
      e = cudaFuncSetAttribute(mma_decode_kernel<16, 4, 1, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Lay<16>::kAlloc);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(mma_decode_kernel<16, 16, 2, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<16>::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mma_decode_kernel<32, 32, QT == 0 ? 4 : 2, QT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<32>::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) sms_cache[dev].store(sms, std::memory_order_relaxed);
  }
  const long long V = ta.units * ta.tpu;
  long long grid = max_ctas < sms ? max_ctas : sms;
  if (grid > V) grid = V;
  const int nv = p.S * p.group;
  // softmax warps: 4 per column group, two groups (four for 32 bf16 rows): more warps to
  // overlap the per-row work than rows need.  int8 codes take more widening arithmetic
  // than e4m3 (the pair conversion): for units of up to 4 rows they get eight widening
  // warps and one column group (0.157 -> 0.142 ms per long-context step); e4m3 measured
  // faster with four widening warps and two groups (0.126 against 0.133 ms).
  const int cg = QT == GQAW_I8 && nv <= 4 ? 1 : nv <= 16 || QT != 0 ? 2 : 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(cg == 1 ? Warps<1, QT>::kThreads : cg == 2 ? Warps<2, QT>::kThreads : Warps<4, 0>::kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.dynamicSmemBytes = nv <= 16 ? Lay<16>::kAlloc : Lay<32>::kAlloc;
  if (nv <= 4) {
    if constexpr (QT == GQAW_I8)
      e = cg == 1 ? cudaLaunchKernelEx(&cfg, mma_decode_kernel<16, 4, 1, QT>, p, ta, maps)
                  : cudaLaunchKernelEx(&cfg, mma_decode_kernel<16, 4, 2, QT>, p, ta, maps);
    else
      e = cudaLaunchKernelEx(&cfg, mma_decode_kernel<16, 4, 2, QT>, p, ta, maps);
  } else if (nv <= 8) {
    e = cudaLaunchKernelEx(&cfg, mma_decode_kernel<16, 8, 2, QT>, p, ta, maps);
  } else if (nv <= 16) {
    e = cudaLaunchKernelEx(&cfg, mma_decode_kernel<16, 16, 2, QT>, p, ta, maps);
  } else {
    e = cudaLaunchKernelEx(&cfg, mma_decode_kernel<32, 32, QT == 0 ? 4 : 2, QT>, p, ta, maps);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqaw
