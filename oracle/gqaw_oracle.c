/*
 * gqaw_oracle.c -- reference oracle for one windowed-KV-cache GroupQueryAttention step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64-accumulating CPU
 * statement of what the step computes.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  The product path (the CUDA library)
 * shares no code, header, table or helper with it and never calls it.
 *
 * Sources (web pages; the contract is stated in prose and one formula):
 *  [P1] onnxruntime PR #32419 "Specify GroupQueryAttention windowed KV cache layout
 *       contract", Description: the resident-count formula L(T), the row layout
 *       (row i holds absolute position T - L + i), multi-token steps, the rollback
 *       rule, and attention_bias in absolute key coordinates.  Its review thread:
 *       T is taken per batch item, T_b = seqlens_k[b] + 1.
 *  [P2] onnxruntime PR #31142 "[CPU] Add windowed kv cache for GQA", Key design
 *       decisions: drifting layout, block compaction, staging; review thread:
 *       64-bit planner arithmetic, past length P = seqlens_k[b] + 1 - S.
 *  [P3] onnxruntime/mobius issue #111 "GQA In-Place KV Cache: Investigation Report",
 *       Part 1.1 (inputs/outputs) and 1.3 (num_heads, kv_num_heads, scale, softcap).
 *  [P4] onnxruntime PR #34226 "Fix CPU Attention causal mask for q_len=1 with
 *       past_key and kv_len > 1", Description: key j is visible to query i iff
 *       j <= i + past_sequence_length.
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *  - window: query at absolute position i sees keys j with i - W < j <= i (W keys
 *    including itself), the causal rule of [P4] combined with the local window;
 *  - logit order: z = softcap * tanh(scale * q.k / softcap) (if softcap > 0),
 *    then + attention_bias[b, h, s, j];
 *  - head grouping: query head h reads kv head h / (num_heads / kv_num_heads);
 *  - multi-token steps with batch > 1 are allowed; every item uses the same S and
 *    its own P_b = T_b - S; P_b < 0 is an error;
 *  - the output is rounded once, from fp64, to the cache dtype (round to nearest
 *    even);
 *  - head_sink / smooth_softmax ([P3] Part 1.1 input 11 and Part 1.3, named only):
 *    a sink is one more logit per head that joins the softmax denominator and has no
 *    value row; it is taken as given (not scaled, capped or biased); smooth_softmax is
 *    a sink of 0 for every head; head_sink wins when both are given;
 *  - rotary embedding ([P3] Part 1.1 inputs cos_cache, sin_cache, position_ids and
 *    Part 1.3 attributes do_rotary, rotary_interleaved; named only): the rotary
 *    position embedding of RoFormer (Su et al.), each pair of dimensions (x1, x2)
 *    turned by the angle of its position, y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin,
 *    with cos/sin read from row `pos` of the caches at column i for the i-th pair.
 *    Pairs are (i, i + rd/2) by default and (2i, 2i + 1) when interleaved; rd is
 *    twice the cache width (head_size unless given), dimensions from rd on pass
 *    through.  pos = position_ids[b, s] if given, else the absolute position P_b + s.
 *    The new query and key rows of the step are turned before use; the turned key
 *    rows are what the cache stores (rounded once to the cache dtype), the turned
 *    query stays in double.  Values are not turned;
 *  - quantized cache ([P3] Part 1.1 inputs k_scale and v_scale, "KV cache quantization
 *    scale", named only): the caches hold int8 or fp8 e4m3 codes, one scale per tensor;
 *    a code c stands for c * scale.  The step's new key and value rows (turned and
 *    rounded to the step's dtype first, if rotary) are quantized once: x / scale in
 *    float (one IEEE division: the code is an integer decision, taken in the kernel's
 *    precision), rounded to nearest even and saturated to the type (int8 [-128, 127];
 *    e4m3 per the OCP 8-bit floating-point format, finite values up to 448, NaN kept).
 *    The cache stores the codes and attention reads every key and value, new ones
 *    included, as code * scale.
 *
 * Precision: every input element is widened exactly to double; dot products,
 * softcap, softmax and the weighted sum are evaluated in double in ascending key
 * order; present rows are bit copies.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_I8 = 2, ORACLE_E4M3 = 3 };

enum {
  ORACLE_OK = 0,
  ORACLE_EARGS = 1,     /* malformed sizes */
  ORACLE_EPAST = 2,     /* seqlens_k[b] + 1 - S < 0 for some item */
  ORACLE_ETOTAL = 3,    /* T_b > total_sequence_length for some item */
  ORACLE_ENOMEM = 4,
  ORACLE_EPOS = 5       /* a rotary position outside [0, rotary_cache_len) */
};

typedef struct oracle_args {
  int64_t batch_size;        /* B */
  int64_t sequence_length;   /* S, new tokens in this step */
  int64_t num_heads;         /* Nq */
  int64_t kv_num_heads;      /* Nkv */
  int64_t head_size;         /* D */
  int64_t capacity;          /* C, dimension 2 of past_key */
  int64_t local_window_size; /* W */
  double scale;              /* already resolved: the caller passes 1/sqrt(D) for the default */
  double softcap;            /* 0: disabled */
  int64_t dtype;             /* ORACLE_F32 or ORACLE_BF16; all tensors but bias share it */
  const void *query;         /* (B, S, Nq*D) */
  const void *key;           /* (B, S, Nkv*D) */
  const void *value;         /* (B, S, Nkv*D) */
  const void *past_key;      /* (B, Nkv, C, D), read only */
  const void *past_value;    /* (B, Nkv, C, D), read only */
  void *present_key;         /* (B, Nkv, C, D), distinct from past; rows [0, L) written */
  void *present_value;       /* (B, Nkv, C, D) */
  const int32_t *seqlens_k;  /* (B,) */
  int64_t total_sequence_length;
  const float *attention_bias; /* NULL or element [b*sb + h*sh + s*ss + j] */
  int64_t bias_stride_b, bias_stride_h, bias_stride_s;
  void *output;              /* (B, S, Nq*D) in dtype */
  double *output_f64;        /* NULL or (B, S, Nq*D), before the final rounding */
  int32_t *resident_len;     /* NULL or (B,), L(T_b) after the step */
  int64_t s_begin, s_end;    /* attention is evaluated for new tokens s in [s_begin, s_end)
                                only (outputs of other rows are left as they are); the
                                present rows are always written */
  const float *head_sink;    /* NULL or (Nq,): a sink logit per query head */
  int64_t smooth_softmax;    /* non-zero: a sink logit of 0 for every head (if no head_sink) */
  int64_t do_rotary;         /* non-zero: turn the new query and key rows (rotary embedding) */
  int64_t rotary_interleaved; /* non-zero: pairs (2i, 2i+1); else (i, i + rd/2) */
  int64_t rotary_dim;        /* rd, even, 0 < rd <= D */
  int64_t rotary_cache_len;  /* rows of cos_cache / sin_cache */
  const void *cos_cache;     /* (rotary_cache_len, rd/2) in dtype */
  const void *sin_cache;     /* (rotary_cache_len, rd/2) in dtype */
  const int64_t *position_ids; /* NULL or (B, S) */
  int64_t cache_dtype;       /* 0: the caches hold dtype; ORACLE_I8 or ORACLE_E4M3: codes */
  float k_scale, v_scale;    /* scales of the quantized caches */
} oracle_args;

/* [P1] Description, resident-count formula:
 *   L(T) = T                          if T <= C
 *   L(T) = T - G * ceil((T - C) / G)  otherwise,   G = C - W + 1.
 * Evaluated in 64-bit integers ([P2] review thread). */
int64_t oracle_resident_len(int64_t T, int64_t C, int64_t W) {
  int64_t G, blocks;
  if (T <= C) return T;
  G = C - W + 1;
  blocks = (T - C + G - 1) / G; /* ceil for positive operands */
  return T - G * blocks;
}

/* Round a double to the nearest bfloat16, ties to even, in one step.
 * bfloat16 keeps 8 significant bits and the float exponent range. */
uint16_t oracle_round_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x), r, y;
  int e, q;
  float f;
  uint32_t bits;
  if (isnan(x)) return 0x7fc0u;
  if (a == 0.0) return sign;
  if (isinf(x)) return (uint16_t)(sign | 0x7f80u);
  frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
  q = e - 8;               /* spacing of 8-significant-bit numbers near a */
  if (q < -133) q = -133;  /* spacing of bfloat16 subnormals */
  r = nearbyint(ldexp(a, -q)); /* default rounding mode: nearest, ties to even */
  y = ldexp(r, q);
  if (y > 3.38953138925153547590470800371487867e38) return (uint16_t)(sign | 0x7f80u);
  f = (float)y; /* exact: y has at most 9 significant bits */
  memcpy(&bits, &f, 4);
  return (uint16_t)(sign | (bits >> 16));
}

/* fp8 e4m3 (OCP 8-bit floating point, "E4M3FN"): sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent 0 holds subnormals m * 2^-9; S.1111.111 is NaN; no
 * infinities; the largest finite value is 1.75 * 2^8 = 448. */
double oracle_decode_e4m3(uint8_t c) {
  const double sign = (c & 0x80) ? -1.0 : 1.0;
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) return sign * ldexp((double)m, -9);
  return sign * ldexp(1.0 + m / 8.0, e - 7);
}

/* The e4m3 code nearest to x (ties to even), saturated to +-448; NaN gives NaN. */
uint8_t oracle_round_e4m3(float x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  const double a = fabs((double)x);
  int e, r;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {                    /* subnormal range: steps of 2^-9 */
    r = (int)nearbyint(ldexp(a, 9));           /* 0 .. 8, ties to even */
    return (uint8_t)(sign | r);                /* r == 8 is the smallest normal, code 0x08 */
  }
  frexp(a, &e);                                /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;                                      /* a = (1 + t) * 2^e, t in [0, 1) */
  r = (int)nearbyint((ldexp(a, -e) - 1.0) * 8.0); /* 0 .. 8, ties to even */
  if (r == 8) {
    r = 0;
    e += 1;
  }
  if (e + 7 > 15 || (e + 7 == 15 && r == 7)) return (uint8_t)(sign | 0x7E);
  return (uint8_t)(sign | ((e + 7) << 3) | r);
}

/* The quantized code of x: x / scale in float, rounded to nearest even, saturated. */
uint8_t oracle_quantize(float x, float scale, int64_t cache_dtype) {
  const float q = x / scale;
  if (cache_dtype == ORACLE_E4M3) return oracle_round_e4m3(q);
  if (isnan(q)) return 0;
  if (q >= 127.0f) return (uint8_t)127;
  if (q <= -128.0f) return (uint8_t)(int8_t)-128;
  return (uint8_t)(int8_t)(int)nearbyintf(q);
}

static double load_elem(const void *base, int64_t idx, int64_t dtype) {
  if (dtype == ORACLE_F32) {
    float f;
    memcpy(&f, (const char *)base + idx * 4, 4);
    return (double)f;
  } else {
    uint16_t h;
    uint32_t bits;
    float f;
    memcpy(&h, (const char *)base + idx * 2, 2);
    bits = ((uint32_t)h) << 16;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
}

static void store_elem(void *base, int64_t idx, int64_t dtype, double v) {
  if (dtype == ORACLE_F32) {
    float f = (float)v; /* C conversion: round to nearest even */
    memcpy((char *)base + idx * 4, &f, 4);
  } else {
    uint16_t h = oracle_round_bf16(v);
    memcpy((char *)base + idx * 2, &h, 2);
  }
}

/* Element idx of a key or value row of the cache's type, as a number: the element
 * itself, or code * scale for a quantized cache. */
static double load_kv(const oracle_args *a, const void *base, int64_t idx, float scale) {
  if (a->cache_dtype == ORACLE_I8) return (double)((const int8_t *)base)[idx] * (double)scale;
  if (a->cache_dtype == ORACLE_E4M3) return oracle_decode_e4m3(((const uint8_t *)base)[idx]) * (double)scale;
  return load_elem(base, idx, a->dtype);
}

/* Element offset of row r (0-based) of slice (b, kvh) in a (B, Nkv, C, D) cache. */
static int64_t cache_row(const oracle_args *a, int64_t b, int64_t kvh, int64_t r) {
  return ((b * a->kv_num_heads + kvh) * a->capacity + r) * a->head_size;
}

/* Element offset of new token s of kv head kvh in a (B, S, Nkv*D) input. */
static int64_t input_row(const oracle_args *a, int64_t b, int64_t s, int64_t kvh) {
  return ((b * a->sequence_length + s) * a->kv_num_heads + kvh) * a->head_size;
}

/* The rotary embedding of one row of D elements at element offset `off` of `src`,
 * turned by the angles of position `pos` (reading above), into y[0..D) in double. */
static void rotate_row(const oracle_args *a, const void *src, int64_t off, int64_t pos, double *y) {
  const int64_t D = a->head_size, half = a->rotary_dim / 2;
  int64_t i;
  for (i = 0; i < D; ++i) y[i] = load_elem(src, off + i, a->dtype);
  for (i = 0; i < half; ++i) {
    const double c = load_elem(a->cos_cache, pos * half + i, a->dtype);
    const double sn = load_elem(a->sin_cache, pos * half + i, a->dtype);
    const int64_t i1 = a->rotary_interleaved ? 2 * i : i;
    const int64_t i2 = a->rotary_interleaved ? 2 * i + 1 : i + half;
    const double x1 = y[i1], x2 = y[i2];
    y[i1] = x1 * c - x2 * sn;
    y[i2] = x2 * c + x1 * sn;
  }
}

/* Turns the S new query and key rows of item b (reading above): the query rows into
 * qrot (B, S, Nq*D) doubles, the key rows into krot (B, S, Nkv*D) in the cache dtype. */
static int rotate_item(const oracle_args *a, int64_t b, double *qrot, void *krot, double *y) {
  const int64_t S = a->sequence_length, D = a->head_size;
  const int64_t P = (int64_t)a->seqlens_k[b] + 1 - S;
  int64_t s, h, d;
  for (s = 0; s < S; ++s) {
    const int64_t pos = a->position_ids ? a->position_ids[b * S + s] : P + s;
    if (pos < 0 || pos >= a->rotary_cache_len) return ORACLE_EPOS;
    for (h = 0; h < a->num_heads; ++h) {
      const int64_t off = ((b * S + s) * a->num_heads + h) * D;
      rotate_row(a, a->query, off, pos, qrot + off);
    }
    for (h = 0; h < a->kv_num_heads; ++h) {
      const int64_t off = input_row(a, b, s, h);
      rotate_row(a, a->key, off, pos, y);
      for (d = 0; d < D; ++d) store_elem(krot, off + d, a->dtype, y[d]);
    }
  }
  return ORACLE_OK;
}

/* One step for one batch item.  The virtual sequence X of item b has Lp + S rows:
 * X[r] = past row r for r < Lp, else new token r - Lp.  X[r] holds absolute
 * position P - Lp + r ([P1] row layout applied to the past length P). */
static int step_item(const oracle_args *a, int64_t b, double *z, double *acc, const double *qrot,
                     const void *knew, const void *vnew) {
  const int64_t S = a->sequence_length, D = a->head_size, W = a->local_window_size;
  const int64_t Nq = a->num_heads, Nkv = a->kv_num_heads, C = a->capacity;
  const int64_t group = Nq / Nkv;
  const int64_t esize = a->cache_dtype ? 1 : (a->dtype == ORACLE_F32 ? 4 : 2); /* cache element */
  const int64_t T = (int64_t)a->seqlens_k[b] + 1; /* [P1] review: T_b = seqlens_k[b] + 1 */
  const int64_t P = T - S;                         /* [P2] review: past length */
  int64_t Lp, Lt, first_pos, s, h, kvh, r, d, j;

  const void *key = knew, *value = vnew; /* the new rows as the cache holds them */

  if (P < 0) return ORACLE_EPAST;
  if (T > a->total_sequence_length) return ORACLE_ETOTAL;
  Lp = oracle_resident_len(P, C, W);
  Lt = oracle_resident_len(T, C, W);
  first_pos = P - Lp; /* absolute position of X[0] */

  /* Attention ([P4] causal rule, local window of W keys, [P3] scale/softcap,
   * [P1] absolute-column attention_bias). */
  for (s = a->s_begin; s < a->s_end && s < S; ++s) {
    const int64_t i = P + s; /* absolute position of query s */
    int64_t jlo = i - W + 1;
    if (jlo < 0) jlo = 0;
    if (jlo < first_pos) jlo = first_pos; /* never taken: Lp >= min(P, W) */
    for (h = 0; h < Nq; ++h) {
      const int64_t qoff = ((b * S + s) * Nq + h) * D;
      double zmax = -INFINITY, denom = 0.0;
      kvh = h / group;
      for (j = jlo; j <= i; ++j) {
        const int64_t xr = j - first_pos;
        const void *kb = xr < Lp ? a->past_key : key;
        const int64_t koff = xr < Lp ? cache_row(a, b, kvh, xr) : input_row(a, b, xr - Lp, kvh);
        double dot = 0.0, zj;
        for (d = 0; d < D; ++d)
          dot += (qrot ? qrot[qoff + d] : load_elem(a->query, qoff + d, a->dtype)) * load_kv(a, kb, koff + d, a->k_scale);
        zj = a->scale * dot;
        if (a->softcap > 0.0) zj = a->softcap * tanh(zj / a->softcap);
        if (a->attention_bias)
          zj += (double)a->attention_bias[b * a->bias_stride_b + h * a->bias_stride_h +
                                          s * a->bias_stride_s + j];
        z[j - jlo] = zj;
        if (zj > zmax) zmax = zj;
      }
      /* the sink logit, if any, joins the maximum and the denominator */
      if (a->head_sink || a->smooth_softmax) {
        const double sink = a->head_sink ? (double)a->head_sink[h] : 0.0;
        if (sink > zmax) zmax = sink;
        denom += exp(sink - zmax);
      }
      for (d = 0; d < D; ++d) acc[d] = 0.0;
      for (j = jlo; j <= i; ++j) {
        const int64_t xr = j - first_pos;
        const void *vb = xr < Lp ? a->past_value : value;
        const int64_t voff = xr < Lp ? cache_row(a, b, kvh, xr) : input_row(a, b, xr - Lp, kvh);
        const double p = exp(z[j - jlo] - zmax);
        denom += p;
        for (d = 0; d < D; ++d) acc[d] += p * load_kv(a, vb, voff + d, a->v_scale);
      }
      for (d = 0; d < D; ++d) {
        const double o = acc[d] / denom;
        store_elem(a->output, qoff + d, a->dtype, o);
        if (a->output_f64) a->output_f64[qoff + d] = o;
      }
    }
  }

  /* Present layout ([P1] row layout): row r holds absolute position T - Lt + r,
   * i.e. X[Lp + S - Lt + r].  Bit copies; rows [Lt, C) are left as they are. */
  for (kvh = 0; kvh < Nkv; ++kvh) {
    for (r = 0; r < Lt; ++r) {
      const int64_t xr = Lp + S - Lt + r;
      const int64_t src = xr < Lp ? cache_row(a, b, kvh, xr) : input_row(a, b, xr - Lp, kvh);
      const void *ksrc = xr < Lp ? a->past_key : key;
      const void *vsrc = xr < Lp ? a->past_value : value;
      const int64_t dst = cache_row(a, b, kvh, r);
      memcpy((char *)a->present_key + dst * esize, (const char *)ksrc + src * esize, D * esize);
      memcpy((char *)a->present_value + dst * esize, (const char *)vsrc + src * esize, D * esize);
    }
  }
  if (a->resident_len) a->resident_len[b] = (int32_t)Lt;
  return ORACLE_OK;
}

/* The S new key and value rows of item b as a quantized cache holds them (reading above):
 * knew, vnew (B, S, Nkv*D) codes; ksrc is the key input, or the turned keys. */
static void quantize_item(const oracle_args *a, int64_t b, const void *ksrc, uint8_t *knew, uint8_t *vnew) {
  const int64_t n = a->kv_num_heads * a->head_size, off = b * a->sequence_length * n;
  int64_t e;
  for (e = 0; e < a->sequence_length * n; ++e) {
    knew[off + e] = oracle_quantize((float)load_elem(ksrc, off + e, a->dtype), a->k_scale, a->cache_dtype);
    vnew[off + e] = oracle_quantize((float)load_elem(a->value, off + e, a->dtype), a->v_scale, a->cache_dtype);
  }
}

/* Items are independent; the step is item by item.  Returns ORACLE_OK or the first
 * error met (items before it are already written). */
int oracle_step(const oracle_args *a) {
  int64_t b, nz;
  double *z, *acc, *qrot = NULL;
  void *krot = NULL;
  uint8_t *knew = NULL, *vnew = NULL;
  const int quant = a->cache_dtype == ORACLE_I8 || a->cache_dtype == ORACLE_E4M3;
  int rc = ORACLE_OK;
  if (a->batch_size < 0 || a->sequence_length < 1 || a->num_heads < 1 || a->kv_num_heads < 1 ||
      a->num_heads % a->kv_num_heads != 0 || a->head_size < 1 || a->capacity < 1 ||
      a->local_window_size < 1 || a->local_window_size > a->capacity ||
      (a->dtype != ORACLE_F32 && a->dtype != ORACLE_BF16))
    return ORACLE_EARGS;
  if (a->cache_dtype != 0 && (!quant || !(a->k_scale > 0.0f) || !(a->v_scale > 0.0f))) return ORACLE_EARGS;
  if (a->do_rotary && (a->rotary_dim < 2 || a->rotary_dim % 2 != 0 || a->rotary_dim > a->head_size ||
                       a->rotary_cache_len < 0 || !a->cos_cache || !a->sin_cache))
    return ORACLE_EARGS;
  nz = a->local_window_size;
  z = (double *)malloc(sizeof(double) * (size_t)nz);
  acc = (double *)malloc(sizeof(double) * (size_t)a->head_size);
  if (a->do_rotary) {
    const size_t rows = (size_t)(a->batch_size * a->sequence_length);
    qrot = (double *)malloc(sizeof(double) * rows * (size_t)(a->num_heads * a->head_size) + 8);
    krot = malloc(8 * rows * (size_t)(a->kv_num_heads * a->head_size) + 8);
  }
  if (quant) {
    const size_t n = (size_t)(a->batch_size * a->sequence_length * a->kv_num_heads * a->head_size) + 8;
    knew = (uint8_t *)malloc(n);
    vnew = (uint8_t *)malloc(n);
  }
  if (!z || !acc || (a->do_rotary && (!qrot || !krot)) || (quant && (!knew || !vnew))) {
    free(z);
    free(acc);
    free(qrot);
    free(krot);
    free(knew);
    free(vnew);
    return ORACLE_ENOMEM;
  }
  for (b = 0; b < a->batch_size && rc == ORACLE_OK; ++b) {
    const void *ksrc = a->key;
    if (a->do_rotary) {
      rc = rotate_item(a, b, qrot, krot, acc);
      ksrc = krot;
    }
    if (rc == ORACLE_OK && quant) quantize_item(a, b, ksrc, knew, vnew);
    if (rc == ORACLE_OK)
      rc = step_item(a, b, z, acc, qrot, quant ? (const void *)knew : ksrc, quant ? (const void *)vnew : a->value);
  }
  free(z);
  free(acc);
  free(qrot);
  free(krot);
  free(knew);
  free(vnew);
  return rc;
}
