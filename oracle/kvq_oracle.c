/*
 * kvq_oracle.c -- CPU reference for decode attention over a quantized, paged
 * KV cache.  TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product path never does.  It shares
 * no code, header or table with the CUDA library.
 *
 * Plain C11, double precision for every floating-point step that the pages do
 * not fix to fp32.  Slow and obvious on purpose.
 *
 * Sources (web pages on quantized-KV decode attention):
 *  - "kv-quant-attn" page, section "Method": every K and V row carries its own
 *    absmax scale computed when the row is written; decode is flash-decoding
 *    with a fixed-order merge of split partials.
 *  - onnxruntime PR #29912 "[CUDA] PagedAttention: quantized KV cache, XQA
 *    decode, MLA, QK-Norm and head sink", Summary of Changes: ReshapeAndCache
 *    quantizes on write; reads dequantize with k_scale / v_scale under
 *    PER_TENSOR or PER_CHANNEL granularity; slot_mapping places each new token;
 *    ApplyHeadSink rescales the output by 1/(1+exp(s_h - lse)); the paged
 *    decode kernel supports softcap and a sliding window.
 *  - onnxruntime PR #32515 "[CUDA] Add INT4 paged KV cache with per-channel
 *    scales", Description: signed 4-bit values packed two per byte, cache head
 *    dimension (head_size+1)/2; int8 step max/127, int4 step max/7.
 *  - onnxruntime issue #29783: per-token (per-position) scales, so appending
 *    never re-quantizes earlier entries.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  R1 round half to even; R2 a true division x/scale (never a reciprocal
 *  multiply); R3 symmetric code range [-qmax, qmax]; R4 an all-zero row gets
 *  scale 0 and all-zero codes; R5 a "row" is one (token, kv head) vector, K and
 *  V scaled separately; R6 fp32 scales; R7 e4m3fn saturates finite overflow to
 *  +-448, NaN stays NaN; R8 low nibble holds the even channel; R10 query head
 *  i reads kv head i / (Hq/Hkv); R11 seq_lens include the T new tokens and
 *  draft tau sits at position L - T + tau, causal among drafts; R12 a window W
 *  keeps exactly the W most recent keys including the query's own position;
 *  R13 sm_scale defaults to 1/sqrt(D); R14 softcap c*tanh(s/c) acts on the
 *  scaled logit, the sink logit is neither scaled nor capped; R15 one sink per
 *  query head for every query token; R16 an empty key set gives o = 0 and
 *  lse = -inf.  For the prologue before the cache write: R19 RMSNorm, then
 *  RoPE; R20 RMSNorm per (token, head) over the D channels with one bf16 weight
 *  vector per side, evaluated here in fp64 from the definition (the pages fix
 *  no evaluation order) with a single bf16 rounding at the end;
 *  R21 RoPE angles come as caller tables cos/sin [max_pos, rotary_dim/2]
 *  indexed by the token's position, half-split pairs unless interleaved is
 *  asked for; R22 on the cache side only K takes the prologue, V is written as
 *  given; R23 the optional Walsh-Hadamard rotation (onnxruntime PR #32515,
 *  note on the stacked change that adds it) comes after RoPE, on Q and K
 *  alike (so dot products are unchanged), in Sylvester order, orthonormal
 *  (entries +-1/sqrt(D)).  For the
 *  group-wise scales the kv-quant-attn page lists as not done (section
 *  "Requirements and limits"): R25 a group is a run of group_size consecutive channels of
 *  one (token, kv head) row (group_size divides D), quantized exactly like a
 *  PER_ROW row of group_size values (absmax / qmax, R1-R4), one fp32 scale
 *  per group stored [num_blocks, Hkv, block_size, D / group_size]; PER_ROW is
 *  the case group_size = D.
 *
 * Parity pins live in tests/ (format table of e4m3 against torch's
 * float8_e4m3fn, brute-force nearest-code search, round-trip bounds, the
 * library SDPA routine, closed forms and invariants).  The int4 nibble order
 * (R8) is this library's own definition: parity unpinned beyond that.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_INT8 1
#define ORC_FP8_E4M3 2
#define ORC_INT4 3

#define ORC_PER_ROW 1
#define ORC_PER_TENSOR 2
#define ORC_PER_CHANNEL 3
#define ORC_PER_GROUP 4

/* ------------------------------------------------------------------ */
/* scalar helpers                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Correctly rounded binary32 quotient.  The double quotient is rounded once
 * more to float; for two binary32 operands this double rounding is innocuous
 * (53 >= 2*24 + 2), so the result equals IEEE single division. */
static float orc_fdiv(float a, float b) { return (float)((double)a / (double)b); }

/* Round half to even, written out so it does not depend on the FP
 * environment's rounding mode (reading R1). */
static double orc_rne(double v) {
  double f = floor(v);
  double r = v - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* E4M3 (e4m3fn) decode from the format definition: 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent 0 is subnormal (m * 2^-9);
 * S.1111.111 is NaN; there is no infinity.  Largest finite value 448. */
double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* E4M3 encode: nearest representable value, ties to the even mantissa,
 * finite overflow saturated to +-448 (reading R7).  NaN maps to 0x7F/0xFF. */
uint8_t orc_e4m3_encode(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range, step 2^-9; a carry to 8 lands on the smallest normal,
     * whose code (exponent 1, mantissa 0) is also 8 */
    int q = (int)orc_rne(a * 512.0);
    return (uint8_t)(sign | q);
  }
  int e2;
  (void)frexp(a, &e2);       /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;            /* a in [2^e, 2^(e+1)) */
  double q = ldexp(a, 3 - e); /* in [8, 16), exact */
  int mm = (int)orc_rne(q);
  if (mm == 16) {
    e += 1;
    mm = 8;
  }
  int code = ((e + 7) << 3) | (mm - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

/* Element-wise batch forms of the codec (used for dense format sweeps). */
void orc_e4m3_encode_n(const float* x, uint8_t* out, long n) {
  for (long k = 0; k < n; ++k) out[k] = orc_e4m3_encode(x[k]);
}
void orc_e4m3_decode_n(const uint8_t* c, double* out, long n) {
  for (long k = 0; k < n; ++k) out[k] = orc_e4m3_decode(c[k]);
}

static double orc_qmax(int dtype) {
  switch (dtype) {
    case ORC_INT8: return 127.0;
    case ORC_INT4: return 7.0;
    default: return 448.0;
  }
}

int orc_row_bytes(int dtype, int D) { return dtype == ORC_INT4 ? (D + 1) / 2 : D; }

/* ------------------------------------------------------------------ */
/* quantize one row (append)                                            */
/* ------------------------------------------------------------------ */

/* Quantize one (token, kv head) row of D bf16 values.
 *   PER_ROW:     scale = absmax / qmax (fp32 division), stored to scale_out[0]
 *   PER_GROUP:   the same for each run of group_size channels (R25): group
 *                g's scale = absmax of channels [g G, (g+1) G) / qmax, stored to
 *                scale_out[g]
 *   PER_TENSOR:  scale = static_scale[0]
 *   PER_CHANNEL: scale_d = static_scale[d]  (this head's D values)
 * int8 / int4: code = clamp(rne(x / scale), -qmax, qmax); e4m3: encode(x/scale).
 * int4 codes are packed two per byte, even channel in the low nibble. */
void orc_quantize_row_g(const uint16_t* x_bf16, int D, int dtype, int mode, const float* static_scale,
                        int group_size, uint8_t* codes, float* scale_out) {
  float qmaxf = (float)orc_qmax(dtype);
  int absmax_mode = mode == ORC_PER_ROW || mode == ORC_PER_GROUP;
  int G = mode == ORC_PER_GROUP ? group_size : D;
  float grp_scale = 0.0f;
  int nbytes = orc_row_bytes(dtype, D);
  if (dtype == ORC_INT4) memset(codes, 0, (size_t)nbytes);
  for (int d = 0; d < D; ++d) {
    if (absmax_mode && d % G == 0) {
      float amax = 0.0f;
      for (int k = d; k < d + G && k < D; ++k) {
        float a = fabsf(orc_bf16_to_f32(x_bf16[k]));
        if (a > amax) amax = a;
      }
      grp_scale = orc_fdiv(amax, qmaxf);
      if (scale_out) scale_out[d / G] = grp_scale;
    }
    float s = absmax_mode ? grp_scale
              : mode == ORC_PER_TENSOR ? static_scale[0]
                                        : static_scale[d];
    float x = orc_bf16_to_f32(x_bf16[d]);
    int code = 0;
    uint8_t byte = 0;
    if (s != 0.0f) {
      float v = orc_fdiv(x, s);
      if (dtype == ORC_FP8_E4M3) {
        byte = orc_e4m3_encode(v);
      } else {
        double r = orc_rne((double)v);
        double qm = orc_qmax(dtype);
        if (r > qm) r = qm;
        if (r < -qm) r = -qm;
        code = (int)r;
      }
    }
    if (dtype == ORC_INT8) {
      codes[d] = (uint8_t)(int8_t)code;
    } else if (dtype == ORC_INT4) {
      uint8_t nib = (uint8_t)(code & 0xF);
      codes[d / 2] |= (d & 1) ? (uint8_t)(nib << 4) : nib;
    } else {
      codes[d] = byte;
    }
  }
}

void orc_quantize_row(const uint16_t* x_bf16, int D, int dtype, int mode, const float* static_scale,
                      uint8_t* codes, float* scale_out) {
  orc_quantize_row_g(x_bf16, D, dtype, mode, static_scale, D, codes, scale_out);
}

/* Code value of channel d in a row (int8 / int4 sign-extended / e4m3). */
static double orc_code_value(const uint8_t* codes, int d, int dtype) {
  if (dtype == ORC_INT8) return (double)(int8_t)codes[d];
  if (dtype == ORC_INT4) {
    int nib = (codes[d / 2] >> ((d & 1) * 4)) & 0xF;
    return (double)(nib >= 8 ? nib - 16 : nib);
  }
  return orc_e4m3_decode(codes[d]);
}

/* ------------------------------------------------------------------ */
/* paged cache                                                          */
/* ------------------------------------------------------------------ */

typedef struct {
  int dtype, k_mode, v_mode;
  int num_blocks, block_size, num_kv_heads, head_dim;
  uint8_t *k_codes, *v_codes; /* [NB, Hkv, bs, Dp] */
  float *k_scale, *v_scale;   /* PER_ROW [NB, Hkv, bs]; PER_TENSOR [1]; PER_CHANNEL [Hkv, D];
                                 PER_GROUP [NB, Hkv, bs, D / group_size] */
  int group_size;             /* PER_GROUP: channels per scale group (divides D) */
} orc_cache;

/* fp32 scales per cached row of a side in this mode (0: static scales). */
static int orc_scales_per_row(const orc_cache* c, int mode) {
  return mode == ORC_PER_ROW ? 1 : mode == ORC_PER_GROUP ? c->head_dim / c->group_size : 0;
}

static size_t orc_row_index(const orc_cache* c, int blk, int h, int row) {
  return ((size_t)blk * c->num_kv_heads + h) * c->block_size + row;
}

/* Append N tokens: token n's (K, V) rows for every kv head are quantized
 * into slot slot_mapping[n] = block * block_size + row.  A negative slot is
 * skipped; a slot past the pool is counted in the return value and skipped. */
int orc_append(const orc_cache* c, const uint16_t* k_new, const uint16_t* v_new,
               const int64_t* slot_mapping, int n_tokens) {
  int bad = 0;
  int H = c->num_kv_heads, D = c->head_dim, Dp = orc_row_bytes(c->dtype, D);
  for (int n = 0; n < n_tokens; ++n) {
    int64_t slot = slot_mapping[n];
    if (slot < 0) continue;
    if (slot >= (int64_t)c->num_blocks * c->block_size) {
      ++bad;
      continue;
    }
    int blk = (int)(slot / c->block_size), row = (int)(slot % c->block_size);
    for (int h = 0; h < H; ++h) {
      size_t ri = orc_row_index(c, blk, h, row);
      const uint16_t* kx = k_new + ((size_t)n * H + h) * D;
      const uint16_t* vx = v_new + ((size_t)n * H + h) * D;
      const float* ks = c->k_mode == ORC_PER_TENSOR ? c->k_scale
                        : c->k_mode == ORC_PER_CHANNEL ? c->k_scale + (size_t)h * D
                                                       : NULL;
      const float* vs = c->v_mode == ORC_PER_TENSOR ? c->v_scale
                        : c->v_mode == ORC_PER_CHANNEL ? c->v_scale + (size_t)h * D
                                                       : NULL;
      int nk = orc_scales_per_row(c, c->k_mode), nv = orc_scales_per_row(c, c->v_mode);
      orc_quantize_row_g(kx, D, c->dtype, c->k_mode, ks, c->group_size, c->k_codes + ri * Dp,
                         nk ? c->k_scale + ri * nk : NULL);
      orc_quantize_row_g(vx, D, c->dtype, c->v_mode, vs, c->group_size, c->v_codes + ri * Dp,
                         nv ? c->v_scale + ri * nv : NULL);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* QK-RMSNorm + RoPE before the cache write (onnxruntime PR #29912,     */
/* Summary of Changes: q_norm_weight / k_norm_weight inputs,            */
/* qk_norm_epsilon with default 1e-6, rotary_offset; "QkNormRotaryTNH"  */
/* fuses QK-RMSNorm and RoPE into one pass, in that order).             */
/* ------------------------------------------------------------------ */

/* The bf16 value nearest to v, ties to even, from the format definition:
 * 8 significant bits for |v| >= 2^-126, a fixed quantum of 2^-133 below that
 * (subnormals), and infinity once the rounded magnitude reaches 2^128. */
uint16_t orc_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  int e;
  frexp(fabs(v), &e); /* |v| in [2^(e-1), 2^e) */
  int lead = e - 1 > -126 ? e - 1 : -126;
  int qe = lead - 7;
  double r = ldexp(orc_rne(ldexp(v, -qe)), qe); /* both scalings exact */
  if (r == 0.0) return signbit(v) ? 0x8000 : 0x0000; /* underflow keeps the sign */
  if (fabs(r) >= ldexp(1.0, 128)) return v > 0 ? 0x7F80 : 0xFF80;
  float f = (float)r; /* exact: at most 8 significant bits, inside the float range */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* One row of D values, written out from the definitions in double precision
 * (reading R20: the pages state the operations, not an evaluation order; fp64
 * leaves any order's rounding far below one bf16 unit):
 *   RMSNorm (w != NULL): y_d = x_d * r * w_d, r = 1 / sqrt(sum_d x_d^2 / D + eps);
 *   RoPE (rd > 0) on channels [off, off + rd), angle index i in [0, rd/2):
 *     the pair (a, b) = (off + i, off + i + rd/2) (half split) or
 *     (off + 2i, off + 2i + 1) (interleaved) becomes
 *     (a cos_i - b sin_i, b cos_i + a sin_i), cos_i = cs[i], sin_i = sn[i]
 *     (the caller's table row of the token's position);
 *   Walsh-Hadamard (hadamard != 0): y <- H y with the Sylvester-order matrix
 *     H[i][j] = (-1)^popcount(i & j) / sqrt(D), a plain matrix-vector product;
 * then one round-to-nearest-even to bf16 per value.  out64 (may be NULL)
 * receives the values before that rounding. */
void orc_norm_rope_row(const uint16_t* x, int D, const uint16_t* w, double eps, int rd, int off,
                       int interleaved, const float* cs, const float* sn, int hadamard, uint16_t* out,
                       double* out64) {
  double y[1024];
  for (int d = 0; d < D; ++d) y[d] = (double)orc_bf16_to_f32(x[d]);
  if (w) {
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += y[d] * y[d];
    double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int d = 0; d < D; ++d) y[d] = y[d] * r * (double)orc_bf16_to_f32(w[d]);
  }
  if (rd > 0) {
    double z[1024];
    memcpy(z, y, sizeof(double) * (size_t)D);
    for (int i = 0; i < rd / 2; ++i) {
      int a = interleaved ? off + 2 * i : off + i;
      int b = interleaved ? a + 1 : a + rd / 2;
      double c = (double)cs[i], s = (double)sn[i];
      z[a] = y[a] * c - y[b] * s;
      z[b] = y[b] * c + y[a] * s;
    }
    memcpy(y, z, sizeof(double) * (size_t)D);
  }
  if (hadamard) {
    double z[1024];
    double inv = 1.0 / sqrt((double)D);
    for (int i = 0; i < D; ++i) {
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -y[j] : y[j];
      z[i] = acc * inv;
    }
    memcpy(y, z, sizeof(double) * (size_t)D);
  }
  for (int d = 0; d < D; ++d) {
    out[d] = orc_f64_to_bf16(y[d]);
    if (out64) out64[d] = y[d];
  }
}

/* The prologue over x [n_tokens, H, D] -> out (same shape, bf16 bits; out64,
 * if not NULL, the same values before the bf16 rounding).  The RoPE tables are
 * [max_pos, rd/2]; a token whose position lies outside [0, max_pos) while
 * rd > 0 is left untouched in out and counted in the return value. */
int orc_norm_rope(const uint16_t* x, int n_tokens, int H, int D, const uint16_t* w, double eps, int rd,
                  int off, int interleaved, const float* cos_tab, const float* sin_tab, int max_pos,
                  const int64_t* positions, int hadamard, uint16_t* out, double* out64) {
  int bad = 0;
  if (D <= 0 || D > 1024 || rd < 0 || rd % 2 || off < 0 || off + rd > D || (hadamard && (D & (D - 1))))
    return -1;
  for (int n = 0; n < n_tokens; ++n) {
    int64_t pos = rd > 0 ? positions[n] : 0;
    if (rd > 0 && (pos < 0 || pos >= max_pos)) {
      ++bad;
      continue;
    }
    const float* cs = rd > 0 ? cos_tab + (size_t)pos * (rd / 2) : NULL;
    const float* sn = rd > 0 ? sin_tab + (size_t)pos * (rd / 2) : NULL;
    for (int h = 0; h < H; ++h) {
      size_t o = ((size_t)n * H + h) * D;
      orc_norm_rope_row(x + o, D, w, eps, rd, off, interleaved, cs, sn, hadamard, out + o,
                        out64 ? out64 + o : NULL);
    }
  }
  return bad;
}

/* Dequantize one cached row (token position t of sequence with block-table
 * row bt) in fp64: code * row scale, * group scale, * tensor scale, or *
 * channel scale. */
static void orc_dequant_row(const orc_cache* c, const uint8_t* codes_base, const float* scale,
                            int mode, const int32_t* bt, int h, int t, double* out) {
  int D = c->head_dim, Dp = orc_row_bytes(c->dtype, D);
  int blk = bt[t / c->block_size], row = t % c->block_size;
  size_t ri = orc_row_index(c, blk, h, row);
  const uint8_t* codes = codes_base + ri * Dp;
  for (int d = 0; d < D; ++d) {
    double s = mode == ORC_PER_ROW ? (double)scale[ri]
               : mode == ORC_PER_GROUP ? (double)scale[ri * (size_t)(D / c->group_size) + d / c->group_size]
               : mode == ORC_PER_TENSOR ? (double)scale[0]
                                         : (double)scale[(size_t)h * D + d];
    out[d] = orc_code_value(codes, d, c->dtype) * s;
  }
}

/* Dequantized K and V rows 0..L-1 of one sequence (block-table row bt) and
 * kv head h, in fp64: kout/vout [L, D]. */
void orc_dequant_seq(const orc_cache* c, const int32_t* bt, int h, int L, double* kout,
                     double* vout) {
  int D = c->head_dim;
  for (int t = 0; t < L; ++t) {
    orc_dequant_row(c, c->k_codes, c->k_scale, c->k_mode, bt, h, t, kout + (size_t)t * D);
    orc_dequant_row(c, c->v_codes, c->v_scale, c->v_mode, bt, h, t, vout + (size_t)t * D);
  }
}

/* ------------------------------------------------------------------ */
/* attention                                                            */
/* ------------------------------------------------------------------ */

typedef struct {
  int batch, num_q_heads, q_tokens, max_blocks_per_seq;
  double sm_scale; /* <= 0: 1/sqrt(D) */
  double softcap;  /* 0: off */
  int window;      /* 0: off */
  int nsplit;      /* 1: one softmax over the key set; >1: split + LSE merge */
} orc_params;

/* softmax attention of one query row over keys [lo, hi] (inclusive); returns
 * lse (natural log) and writes o (unnormalised sums are kept in fp64). */
static double orc_attend_range(const orc_cache* c, const orc_params* p, const int32_t* bt, int h,
                               const double* q, int lo, int hi, double* o, double* kbuf,
                               double* vbuf, double* s) {
  int D = c->head_dim;
  double scale = p->sm_scale > 0 ? p->sm_scale : 1.0 / sqrt((double)D);
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (hi < lo) return -INFINITY;
  double m = -INFINITY;
  for (int j = lo; j <= hi; ++j) {
    orc_dequant_row(c, c->k_codes, c->k_scale, c->k_mode, bt, h, j, kbuf);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * kbuf[d];
    double sj = scale * dot;
    if (p->softcap > 0) sj = p->softcap * tanh(sj / p->softcap);
    s[j - lo] = sj;
    if (sj > m) m = sj;
  }
  double l = 0.0;
  for (int j = lo; j <= hi; ++j) {
    double w = exp(s[j - lo] - m);
    l += w;
    orc_dequant_row(c, c->v_codes, c->v_scale, c->v_mode, bt, h, j, vbuf);
    for (int d = 0; d < D; ++d) o[d] += w * vbuf[d];
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  return m + log(l);
}

/* One output row (b, tau, i).  Key set: 0 <= j <= pos, pos = L_b - T + tau,
 * and j > pos - W when a window W is set.  Optional split of the key set into
 * nsplit contiguous ranges merged by the log-sum-exp rule in range order. */
static void orc_attend_one(const orc_cache* c, const orc_params* p, const int32_t* block_table,
                           const int32_t* seq_lens, const uint16_t* q_bf16, const float* head_sink,
                           int b, int tau, int i, double* out, double* lse_out, double* work) {
  int D = c->head_dim, Hq = p->num_q_heads, T = p->q_tokens;
  int G = Hq / c->num_kv_heads, h = i / G;
  const int32_t* bt = block_table + (size_t)b * p->max_blocks_per_seq;
  double* q = work;
  double* kbuf = q + D;
  double* vbuf = kbuf + D;
  double* o_part = vbuf + D;
  double* s = o_part + D;
  const uint16_t* qrow = q_bf16 + (((size_t)b * T + tau) * Hq + i) * D;
  for (int d = 0; d < D; ++d) q[d] = (double)orc_bf16_to_f32(qrow[d]);

  int pos = seq_lens[b] - T + tau;
  int lo = 0;
  if (p->window > 0 && pos - p->window + 1 > lo) lo = pos - p->window + 1;
  int hi = pos;
  double lse;
  if (hi < lo || pos < 0) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    lse = -INFINITY;
  } else if (p->nsplit <= 1) {
    lse = orc_attend_range(c, p, bt, h, q, lo, hi, out, kbuf, vbuf, s);
  } else {
    /* split-KV: partial (lse_s, o_s) per range, merged in fixed order:
     * M = max lse_s, w_s = exp(lse_s - M), o = sum w_s o_s / sum w_s,
     * lse = M + log(sum w_s) */
    int n = hi - lo + 1, S = p->nsplit;
    double* lse_s = (double*)malloc(sizeof(double) * S);
    double* o_s = (double*)malloc(sizeof(double) * (size_t)S * D);
    double M = -INFINITY;
    for (int k = 0; k < S; ++k) {
      int a = lo + (int)((long long)n * k / S), e = lo + (int)((long long)n * (k + 1) / S) - 1;
      lse_s[k] = orc_attend_range(c, p, bt, h, q, a, e, o_s + (size_t)k * D, kbuf, vbuf, s);
      if (lse_s[k] > M) M = lse_s[k];
    }
    double wsum = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int k = 0; k < S; ++k) {
      if (lse_s[k] == -INFINITY) continue;
      double w = exp(lse_s[k] - M);
      wsum += w;
      for (int d = 0; d < D; ++d) out[d] += w * o_s[(size_t)k * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= wsum;
    lse = M + log(wsum);
    free(lse_s);
    free(o_s);
  }
  if (head_sink && lse != -INFINITY) {
    /* exact post-hoc sink rescale: o *= 1 / (1 + exp(sink_i - lse)) */
    double f = 1.0 / (1.0 + exp((double)head_sink[i] - lse));
    for (int d = 0; d < D; ++d) out[d] *= f;
  }
  *lse_out = lse;
}

typedef struct {
  const orc_cache* c;
  const orc_params* p;
  const int32_t *block_table, *seq_lens, *rows;
  const uint16_t* q;
  const float* sink;
  double *out, *lse;
  int nrows, first, stride;
  size_t work_len;
} orc_job;

static void* orc_worker(void* arg) {
  orc_job* jb = (orc_job*)arg;
  double* work = (double*)malloc(sizeof(double) * jb->work_len);
  int T = jb->p->q_tokens, Hq = jb->p->num_q_heads, D = jb->c->head_dim;
  for (int r = jb->first; r < jb->nrows; r += jb->stride) {
    int b, tau, i;
    size_t oidx;
    if (jb->rows) {
      b = jb->rows[3 * r];
      tau = jb->rows[3 * r + 1];
      i = jb->rows[3 * r + 2];
      oidx = (size_t)r;
    } else {
      i = r % Hq;
      tau = (r / Hq) % T;
      b = r / (Hq * T);
      oidx = (size_t)r;
    }
    orc_attend_one(jb->c, jb->p, jb->block_table, jb->seq_lens, jb->q, jb->sink, b, tau, i,
                   jb->out + oidx * D, jb->lse + oidx, work);
  }
  free(work);
  return NULL;
}

/* Attention for every output row (rows == NULL: out [B, T, Hq, D] and
 * lse [B, T, Hq]) or for the listed (b, tau, i) triples (out [nrows, D]).
 * nthreads POSIX threads share the rows round-robin. */
int orc_attend(const orc_cache* c, const orc_params* p, const int32_t* block_table,
               const int32_t* seq_lens, const uint16_t* q_bf16, const float* head_sink,
               const int32_t* rows, int nrows, double* out, double* lse, int nthreads) {
  int total = rows ? nrows : p->batch * p->q_tokens * p->num_q_heads;
  int cap = p->max_blocks_per_seq * c->block_size;
  for (int b = 0; b < p->batch; ++b) {
    if (seq_lens[b] > cap || seq_lens[b] < 0) return -1;
    const int32_t* bt = block_table + (size_t)b * p->max_blocks_per_seq;
    for (int pg = 0; pg * c->block_size < seq_lens[b]; ++pg)
      if (bt[pg] < 0 || bt[pg] >= c->num_blocks) return -2;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > total && total > 0) nthreads = total;
  size_t work_len = (size_t)4 * c->head_dim + (size_t)(cap > 0 ? cap : 1);
  orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    orc_job j = {c, p, block_table, seq_lens, rows, q_bf16, head_sink, out, lse,
                 total, t, nthreads, work_len};
    jobs[t] = j;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
  orc_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  return 0;
}
