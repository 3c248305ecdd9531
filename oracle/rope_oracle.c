/*
 * rope_oracle.c -- reference oracle for rotary position embedding (RoPE),
 * multimodal RoPE (M-RoPE), the on-the-fly cos/sin variant and the cos/sin
 * cache build.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The product path (the
 * CUDA library and its Python binding) never calls it, and the two share no
 * code: no header, no helper, no table, no constant generator.
 *
 * Plain, single-threaded and slow on purpose. Every loop follows the operator
 * definition element by element. Arithmetic is binary64 wherever the
 * definition does not fix a narrower type, and each output is rounded once,
 * to nearest-even, to the storage type T (float32, float16 or bfloat16). The only steps
 * done in binary32 are the ones the modelling code fixes to float32 (the
 * angle product and the cos/sin values of the on-the-fly variant).
 *
 * Sources (web pages, cited by title and section):
 *  [RE] "ai.onnx.RotaryEmbedding" WebGPU kernel manifest (manifest.json):
 *       "description", "inputs" (X, cos_cache, sin_cache, position_ids),
 *       "attributeDescriptions" (interleaved, num_heads,
 *       rotary_embedding_dim), "derive" (rank3Contract, rank4Contract,
 *       rank3PosContract, rank4PosContract) and the Params fields of
 *       "bindingSets".
 *  [MR] "com.microsoft.MRotaryEmbedding" README: Description, Inputs
 *       (positionIds, cos), Attributes (interleaved, mrope_layout,
 *       mrope_section, rotary_embedding_dim, scale), Implementation variants
 *       (pairs4).
 *  [PR] onnxruntime pull request "Add RotaryEmbedding fusion for Qwen3
 *       on-the-fly RoPE patterns": Motivation and Context; Modeling Code
 *       Alignment Check (Qwen3RotaryEmbedding.forward, rotate_half,
 *       apply_rotary_pos_emb); Critical Issues 1 (positions beyond the
 *       cache); Medium Issues 4 (the cache is cos(freqs) * scaling).
 *  [SA] "com.microsoft.SparseAttention" README: Attributes
 *       (rotary_interleaved rotates adjacent pairs, 0 is the NeoX half split).
 *
 * Readings where the pages leave a step open are stated beside the code.
 * Parity unpinned: the interleaved M-RoPE stream order (mrope_layout = 1)
 * for sections where the two readings below differ; only the reading itself
 * is pinned (counts honour mrope_section, and both readings agree where the
 * page's own example applies).
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16, written out from the format: 1 sign bit, 5 exponent   */
/* bits (bias 15), 10 fraction bits; exponent field 0 is subnormal (unit    */
/* 2^-24), field 31 is infinity or NaN.                                     */
/* ------------------------------------------------------------------------ */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(m + 1024), e - 25);
  }
  return sign ? -v : v;
}

/* Round a binary64 value to binary16, nearest-even, in one step. */
uint16_t oracle_double_to_half(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | 0x7e00);
  /* 65504 is the largest finite half; 65520 is the midpoint to 2^16 and ties
     go to the even neighbour, which is the overflow to infinity. */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: an integer number of 2^-24 units (1024 is the
       smallest normal, which the encoding below gives for free) */
    double r = nearbyint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)r);
  }
  int e;
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): unbiased exponent e-1 */
  int E = e - 1;
  double r = nearbyint(ldexp(a, 10 - E)); /* significand in [1024, 2048] */
  if (r == 2048.0) {
    r = 1024.0;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* ------------------------------------------------------------------------ */
/* bfloat16, written out from the format: 1 sign bit, 8 exponent bits      */
/* (bias 127), 7 fraction bits; exponent field 0 is subnormal (unit        */
/* 2^-133), field 255 is infinity or NaN. (The pages list only float32 and  */
/* float16; bfloat16 storage is offered beyond them with the same          */
/* arithmetic and one final rounding.)                                     */
/* ------------------------------------------------------------------------ */
double oracle_bf16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int m = h & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133);
  } else if (e == 255) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(m + 128), e - 134);
  }
  return sign ? -v : v;
}

/* Round a binary64 value to bfloat16, nearest-even, in one step. */
uint16_t oracle_double_to_bf16(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | 0x7fc0);
  /* 255 * 2^120 is the largest finite value; 255.5 * 2^120, the midpoint to
     2^128, ties to the even neighbour, which is the overflow to infinity. */
  if (a >= ldexp(255.5, 120)) return (uint16_t)(sign | 0x7f80);
  if (a < ldexp(1.0, -126)) {
    /* subnormal range: an integer number of 2^-133 units (128 is the
       smallest normal, which the encoding below gives for free) */
    double r = nearbyint(ldexp(a, 133));
    return (uint16_t)(sign | (uint16_t)r);
  }
  int e;
  (void)frexp(a, &e);
  int E = e - 1;
  double r = nearbyint(ldexp(a, 7 - E)); /* significand in [128, 256] */
  if (r == 256.0) {
    r = 128.0;
    E += 1;
  }
  if (E > 127) return (uint16_t)(sign | 0x7f80);
  return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)(r - 128.0));
}

/* Element access by storage type T. */
static double ld(int dt, const void* base, int64_t i) {
  if (dt == ORC_F16) return oracle_half_to_double(((const uint16_t*)base)[i]);
  if (dt == ORC_BF16) return oracle_bf16_to_double(((const uint16_t*)base)[i]);
  return (double)((const float*)base)[i];
}

static void st(int dt, void* base, int64_t i, double v) {
  if (dt == ORC_F16)
    ((uint16_t*)base)[i] = oracle_double_to_half(v);
  else if (dt == ORC_BF16)
    ((uint16_t*)base)[i] = oracle_double_to_bf16(v);
  else
    ((float*)base)[i] = (float)v;
}

/* Bit-exact copy of one element: pass-through never re-rounds. */
static void cp(int dt, const void* src, int64_t si, void* dst, int64_t di) {
  if (dt == ORC_F16 || dt == ORC_BF16)
    ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
  else
    memcpy((float*)dst + di, (const float*)src + si, sizeof(float));
}

/* The value of v after rounding to T. */
static double round_to(int dt, double v) {
  if (dt == ORC_F16) return oracle_half_to_double(oracle_double_to_half(v));
  if (dt == ORC_BF16) return oracle_bf16_to_double(oracle_double_to_bf16(v));
  return (double)(float)v;
}

/* ------------------------------------------------------------------------ */
/* Geometry of X.                                                           */
/* [RE] inputs/X: rank 3 is (batch, sequence, hidden) with hidden =         */
/* num_heads * head_size; rank 4 is (batch, num_heads, sequence, head_size).*/
/* The Params fields (numHeads, sequenceLength, headSize) of "bindingSets"  */
/* give the same decomposition. Row (b, s, n) starts at                     */
/*   rank 3: ((b*S + s)*N + n)*H        rank 4: ((b*N + n)*S + s)*H.        */
/* ------------------------------------------------------------------------ */
typedef struct {
  int64_t B, S, N, H;
  int rank;
} geom;

static int make_geom(int rank, const int64_t* xs, int64_t num_heads, geom* g) {
  g->rank = rank;
  if (rank == 3) {
    if (num_heads <= 0 || xs[2] % num_heads != 0) return 1;
    g->B = xs[0];
    g->S = xs[1];
    g->N = num_heads;
    g->H = xs[2] / num_heads;
  } else if (rank == 4) {
    g->B = xs[0];
    g->N = xs[1];
    g->S = xs[2];
    g->H = xs[3];
  } else {
    return 1;
  }
  return 0;
}

static int64_t row_start(const geom* g, int64_t b, int64_t s, int64_t n) {
  if (g->rank == 3) return ((b * g->S + s) * g->N + n) * g->H;
  return ((b * g->N + n) * g->S + s) * g->H;
}

/* The two elements of rotation pair i inside a head of rotary width rd.
   [RE] attributeDescriptions/interleaved: 0 splits the rotated part into two
   contiguous halves, so pair i is (i, i + rd/2) -- the rotate_half form of
   [PR] Modeling Code Alignment Check; 1 pairs even/odd elements, so pair i is
   (2i, 2i+1) -- [SA] rotary_interleaved "adjacent pairs". Reading: pair i
   uses coefficient index i in both pairings. */
static void pair_elems(int interleaved, int64_t half, int64_t i, int64_t* j0, int64_t* j1) {
  if (interleaved) {
    *j0 = 2 * i;
    *j1 = 2 * i + 1;
  } else {
    *j0 = i;
    *j1 = i + half;
  }
}

/* One rotation of the pair (x0, x1) by (c, s):
     y0 = x0*c - x1*s,   y1 = x1*c + x0*s.
   [PR] apply_rotary_pos_emb: q*cos + rotate_half(q)*sin with
   rotate_half(q) = cat(-q2, q1) and cos = cat(freqs, freqs): element i of the
   first half gets x_i*c_i - x_{i+h}*s_i, element i+h gets x_{i+h}*c_i + x_i*s_i.
   Computed in binary64 and rounded once to T. */
static void rotate_store(int dt, void* y, int64_t j0, int64_t j1, double x0, double x1, double c,
                         double s) {
  double y0 = x0 * c - x1 * s;
  double y1 = x1 * c + x0 * s;
  st(dt, y, j0, y0);
  st(dt, y, j1, y1);
}

/* ------------------------------------------------------------------------ */
/* RotaryEmbedding.                                                         */
/* [RE] inputs: with position_ids the (max_sequence_length, rotary_dim/2)   */
/* tables are gathered at position_ids[b, s]; without, the tables are       */
/* (batch, sequence, rotary_dim/2) and row (b, s) is used directly.         */
/* [RE] attributeDescriptions/rotary_embedding_dim: 0 rotates the whole     */
/* head, otherwise only the leading rd elements; the rest pass through.     */
/* Reading for a position outside [0, cache_rows): [RE] says valid          */
/* positions are non-negative cache rows and [PR] Critical Issues 1 shows   */
/* the damage of reading past the cache; the token's heads are copied       */
/* through unchanged, as [MR] Description does for an out-of-range pair.    */
/* Returns 0, or 1 on a malformed geometry. *n_oor counts tokens whose      */
/* position was out of range.                                               */
/* ------------------------------------------------------------------------ */
int oracle_rope(int dt, int rank, const int64_t* xs, int64_t num_heads, int interleaved,
                int64_t rotary_dim, const void* x, const void* cos_t, const void* sin_t,
                int64_t cache_rows, const int64_t* pos, void* y, int64_t* n_oor) {
  geom g;
  if (make_geom(rank, xs, num_heads, &g)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : g.H;
  int64_t half = rd / 2;
  if (rd % 2 || rd > g.H || rd <= 0) return 1;
  int64_t oor = 0;
  for (int64_t b = 0; b < g.B; ++b) {
    for (int64_t s = 0; s < g.S; ++s) {
      int64_t tok = b * g.S + s;
      int64_t crow;
      int valid = 1;
      if (pos) {
        int64_t p = pos[tok];
        valid = (p >= 0 && p < cache_rows);
        crow = p * half;
      } else {
        crow = tok * half;
      }
      if (!valid) ++oor;
      for (int64_t n = 0; n < g.N; ++n) {
        int64_t base = row_start(&g, b, s, n);
        if (!valid) {
          for (int64_t j = 0; j < g.H; ++j) cp(dt, x, base + j, y, base + j);
          continue;
        }
        for (int64_t i = 0; i < half; ++i) {
          int64_t j0, j1;
          pair_elems(interleaved, half, i, &j0, &j1);
          double c = ld(dt, cos_t, crow + i);
          double sn = ld(dt, sin_t, crow + i);
          rotate_store(dt, y, base + j0, base + j1, ld(dt, x, base + j0), ld(dt, x, base + j1), c,
                       sn);
        }
        for (int64_t j = rd; j < g.H; ++j) cp(dt, x, base + j, y, base + j);
      }
    }
  }
  if (n_oor) *n_oor = oor;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* M-RoPE stream maps: which of the temporal (0), height (1) and width (2)  */
/* position streams drives coefficient index i, for i < rd/2.               */
/* [MR] Attributes/mrope_section: three non-negative counts that divide     */
/* the half-rotary axis among t, h, w and sum to rd/2.                      */
/* [MR] Attributes/mrope_layout: 0 is the sectioned (chunked) layout, 1 the */
/* interleaved one.                                                         */
/* ------------------------------------------------------------------------ */

/* Layout 0: the first sec_t indices use t, the next sec_h use h, the rest w. */
static int map_chunked(const int32_t* sec, int64_t half, uint8_t* map) {
  int64_t i = 0;
  for (int st = 0; st < 3; ++st)
    for (int32_t k = 0; k < sec[st]; ++k) {
      if (i >= half) return 1;
      map[i++] = (uint8_t)st;
    }
  return i == half ? 0 : 1;
}

/* Layout 1, primary reading: deal the indices round by round, t then h then
   w, each stream taking part in as many rounds as its section count, so the
   counts per stream are exactly mrope_section (the page says the sections
   divide the axis). For sections with sec_h == sec_w <= sec_t this gives
   t,h,w,t,h,w,... then t to the end. */
static int map_interleaved(const int32_t* sec, int64_t half, uint8_t* map) {
  int64_t i = 0;
  int32_t rounds = sec[0];
  if (sec[1] > rounds) rounds = sec[1];
  if (sec[2] > rounds) rounds = sec[2];
  for (int32_t r = 0; r < rounds; ++r)
    for (int st = 0; st < 3; ++st)
      if (r < sec[st]) {
        if (i >= half) return 1;
        map[i++] = (uint8_t)st;
      }
  return i == half ? 0 : 1;
}

/* Layout 1, alternative reading: fixed stride-3 slots capped at three
   times the section, i.e. index i goes to h when i % 3 == 1 and
   i < 3*sec_h, to w when i % 3 == 2 and i < 3*sec_w, else to t. The
   counts can differ from mrope_section when 3*sec_h or 3*sec_w exceed rd/2. */
static int map_interleaved_stride3(const int32_t* sec, int64_t half, uint8_t* map) {
  for (int64_t i = 0; i < half; ++i) {
    uint8_t st = 0;
    if (i % 3 == 1 && i < 3 * (int64_t)sec[1])
      st = 1;
    else if (i % 3 == 2 && i < 3 * (int64_t)sec[2])
      st = 2;
    map[i] = st;
  }
  return 0;
}

/* layout: 0 chunked, 1 interleaved (primary reading), 2 interleaved
   stride-3 reading. Returns 0 on success, 1 when the sections do not add
   up to half (layouts 0 and 1) or a section is negative. */
int oracle_mrope_stream_map(const int32_t* sec, int layout, int64_t half, uint8_t* map) {
  if (sec[0] < 0 || sec[1] < 0 || sec[2] < 0) return 1;
  if (layout == 0) return map_chunked(sec, half, map);
  if (layout == 1) return map_interleaved(sec, half, map);
  if (layout == 2) return map_interleaved_stride3(sec, half, map);
  return 1;
}

/* ------------------------------------------------------------------------ */
/* MRotaryEmbedding with an explicit stream map.                            */
/* [MR] Inputs/positionIds: (3, batch, sequence) int64, streams t, h, w;    */
/* negative or out-of-cache ids copy their pair through unchanged (also     */
/* [MR] Description). Int32 storage saturates large ids on the page; a      */
/* saturated id is still >= the cache rows, so comparing the int64 value    */
/* gives the same copy-through.                                             */
/* [MR] Inputs/cos: one (max_sequence_length, rd/2) table shared by all     */
/* three streams.                                                           */
/* [MR] Attributes/scale and Implementation variants/pairs4: the gathered   */
/* cos and sin are multiplied by scale and rounded to T before rotating.    */
/* Reading: the product c*scale is exact in binary64 and rounded once.      */
/* *n_oor counts pairs copied through (per head).                           */
/* ------------------------------------------------------------------------ */
int oracle_mrope_map(int dt, int rank, const int64_t* xs, int64_t num_heads, int interleaved,
                     int64_t rotary_dim, const void* x, const void* cos_t, const void* sin_t,
                     int64_t cache_rows, const int64_t* pos3, const uint8_t* map, float scale,
                     void* y, int64_t* n_oor) {
  geom g;
  if (make_geom(rank, xs, num_heads, &g)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : g.H;
  int64_t half = rd / 2;
  if (rd % 2 || rd > g.H || rd <= 0) return 1;
  int64_t ntok = g.B * g.S;
  int64_t oor = 0;
  for (int64_t b = 0; b < g.B; ++b) {
    for (int64_t s = 0; s < g.S; ++s) {
      int64_t tok = b * g.S + s;
      int64_t p3[3];
      for (int k = 0; k < 3; ++k) p3[k] = pos3[k * ntok + tok];
      for (int64_t n = 0; n < g.N; ++n) {
        int64_t base = row_start(&g, b, s, n);
        for (int64_t i = 0; i < half; ++i) {
          int64_t j0, j1;
          pair_elems(interleaved, half, i, &j0, &j1);
          int64_t p = p3[map[i]];
          if (p < 0 || p >= cache_rows) {
            cp(dt, x, base + j0, y, base + j0);
            cp(dt, x, base + j1, y, base + j1);
            ++oor;
            continue;
          }
          double c = round_to(dt, ld(dt, cos_t, p * half + i) * (double)scale);
          double sn = round_to(dt, ld(dt, sin_t, p * half + i) * (double)scale);
          rotate_store(dt, y, base + j0, base + j1, ld(dt, x, base + j0), ld(dt, x, base + j1), c,
                       sn);
        }
        for (int64_t j = rd; j < g.H; ++j) cp(dt, x, base + j, y, base + j);
      }
    }
  }
  if (n_oor) *n_oor = oor;
  return 0;
}

/* MRotaryEmbedding with the map given by mrope_section and mrope_layout. */
int oracle_mrope(int dt, int rank, const int64_t* xs, int64_t num_heads, int interleaved,
                 int64_t rotary_dim, const void* x, const void* cos_t, const void* sin_t,
                 int64_t cache_rows, const int64_t* pos3, const int32_t* sec, int layout,
                 float scale, void* y, int64_t* n_oor) {
  geom g;
  if (make_geom(rank, xs, num_heads, &g)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : g.H;
  int64_t half = rd / 2;
  if (half <= 0 || half > 65536) return 1;
  uint8_t map[65536];
  if (oracle_mrope_stream_map(sec, layout, half, map)) return 1;
  return oracle_mrope_map(dt, rank, xs, num_heads, interleaved, rotary_dim, x, cos_t, sin_t,
                          cache_rows, pos3, map, scale, y, n_oor);
}

/* ------------------------------------------------------------------------ */
/* On-the-fly coefficients.                                                 */
/* [PR] Motivation and Context and Modeling Code Alignment Check:           */
/*   freqs = inv_freq @ position_ids in float32, i.e. freqs[p, i] =         */
/*   float(p) * inv_freq[i]; emb = cat(freqs, freqs); cos = emb.cos() *     */
/*   attention_scaling, sin likewise; then cast to the dtype of x.          */
/* [PR] Medium Issues 4: the first rd/2 columns of cat(freqs, freqs) are    */
/* freqs itself, so coefficient i is a function of freqs[p, i] alone.       */
/* Reading: each float32 step is one correctly rounded float32 operation;   */
/* cos and sin of the float32 angle are evaluated in binary64 and rounded   */
/* to float32, the product with attention_scaling is a float32 product, and */
/* the result is rounded to T.                                              */
/* ------------------------------------------------------------------------ */
static void coef_on_the_fly(int dt, int64_t p, float inv, float scaling, double* c, double* s) {
  float pf = (float)p;
  float theta = pf * inv;
  float c32 = (float)cos((double)theta);
  float s32 = (float)sin((double)theta);
  float cs = c32 * scaling;
  float ss = s32 * scaling;
  *c = round_to(dt, (double)cs);
  *s = round_to(dt, (double)ss);
}

/* Rotation with coefficients computed from inv_freq at each token's
   position ([PR] Motivation and Context); no cache, so no position is out of
   range. inv_freq has rd/2 float32 entries. */
int oracle_rope_fused(int dt, int rank, const int64_t* xs, int64_t num_heads, int interleaved,
                      int64_t rotary_dim, const void* x, const float* inv_freq, float scaling,
                      const int64_t* pos, void* y) {
  geom g;
  if (make_geom(rank, xs, num_heads, &g)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : g.H;
  int64_t half = rd / 2;
  if (rd % 2 || rd > g.H || rd <= 0) return 1;
  for (int64_t b = 0; b < g.B; ++b) {
    for (int64_t s = 0; s < g.S; ++s) {
      int64_t p = pos[b * g.S + s];
      for (int64_t n = 0; n < g.N; ++n) {
        int64_t base = row_start(&g, b, s, n);
        for (int64_t i = 0; i < half; ++i) {
          int64_t j0, j1;
          pair_elems(interleaved, half, i, &j0, &j1);
          double c, sn;
          coef_on_the_fly(dt, p, inv_freq[i], scaling, &c, &sn);
          rotate_store(dt, y, base + j0, base + j1, ld(dt, x, base + j0), ld(dt, x, base + j1), c,
                       sn);
        }
        for (int64_t j = rd; j < g.H; ++j) cp(dt, x, base + j, y, base + j);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* MRotaryEmbedding with on-the-fly coefficients.                           */
/* [MR] Description and Inputs: coefficient index i follows one of the t,   */
/* h, w position streams (mrope_section, mrope_layout) and the cached cos   */
/* and sin are scaled by `scale` and rounded to T; [PR] Motivation and      */
/* Context: the cache is cos/sin(p * inv_freq) * attention_scaling, which   */
/* the on-the-fly form computes where it is used.                           */
/* Reading: index i of token (b, s) takes the coefficients the cache build  */
/* would store at row p = pos3[map[i], b, s] (coef_on_the_fly), then the    */
/* scale step of oracle_mrope_map; with no table, no position is out of     */
/* range (as oracle_rope_fused). For in-range positions this equals         */
/* oracle_mrope over the oracle_cache_build table, bit for bit.             */
/* ------------------------------------------------------------------------ */
int oracle_mrope_fused(int dt, int rank, const int64_t* xs, int64_t num_heads, int interleaved,
                       int64_t rotary_dim, const void* x, const float* inv_freq, float scaling,
                       const int64_t* pos3, const int32_t* sec, int layout, float scale, void* y) {
  geom g;
  if (make_geom(rank, xs, num_heads, &g)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : g.H;
  int64_t half = rd / 2;
  if (rd % 2 || rd > g.H || rd <= 0 || half > 65536) return 1;
  uint8_t map[65536];
  if (oracle_mrope_stream_map(sec, layout, half, map)) return 1;
  int64_t ntok = g.B * g.S;
  for (int64_t b = 0; b < g.B; ++b) {
    for (int64_t s = 0; s < g.S; ++s) {
      int64_t tok = b * g.S + s;
      for (int64_t n = 0; n < g.N; ++n) {
        int64_t base = row_start(&g, b, s, n);
        for (int64_t i = 0; i < half; ++i) {
          int64_t j0, j1;
          pair_elems(interleaved, half, i, &j0, &j1);
          int64_t p = pos3[(int64_t)map[i] * ntok + tok];
          double c, sn;
          coef_on_the_fly(dt, p, inv_freq[i], scaling, &c, &sn);
          c = round_to(dt, c * (double)scale);
          sn = round_to(dt, sn * (double)scale);
          rotate_store(dt, y, base + j0, base + j1, ld(dt, x, base + j0), ld(dt, x, base + j1), c,
                       sn);
        }
        for (int64_t j = rd; j < g.H; ++j) cp(dt, x, base + j, y, base + j);
      }
    }
  }
  return 0;
}

/* The (rows, half) cos and sin tables: row p holds the on-the-fly
   coefficients of position p ([PR] Medium Issues 4: cos(freqs) * scaling). */
int oracle_cache_build(int dt, const float* inv_freq, int64_t half, int64_t rows, float scaling,
                       void* cos_out, void* sin_out) {
  if (half <= 0 || rows < 0) return 1;
  for (int64_t p = 0; p < rows; ++p)
    for (int64_t i = 0; i < half; ++i) {
      double c, s;
      coef_on_the_fly(dt, p, inv_freq[i], scaling, &c, &s);
      st(dt, cos_out, p * half + i, c);
      st(dt, sin_out, p * half + i, s);
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Q and K rotation for grouped-query attention, with the optional key/     */
/* value cache append.                                                      */
/* [SA] Description: grouped-query heads, separate or packed [Q|K|V] input, */
/* partial or full rotary embedding in NeoX or interleaved layout; the past */
/* key and value tensors are updated in place.                              */
/* [SA] Inputs: query (B, S, Nq*H), or packed (B, S, (Nq + 2*Nkv)*H) when   */
/* key and value are omitted; key and value (B, S, Nkv*H); past_key and     */
/* past_value (B, Nkv, max_cache_sequence_length, H).                       */
/* [SA] Attributes: do_rotary rotates Q, and K before it enters the cache;  */
/* kv_num_heads divides num_heads.                                          */
/* [PR] Verification and Qwen3 Architecture: RoPE is applied to both the Q  */
/* and the K path of every layer, and GQA has fewer K/V heads than Q heads. */
/* Readings:                                                                */
/*  - every Q and K head is rotated exactly as oracle_rope rotates one head */
/*    of a rank-3 X: same tables, positions, pairing, rotary width,         */
/*    pass-through tail, and an out-of-range position copies the token's    */
/*    heads through;                                                        */
/*  - cache mode (k_cache given): new token s of batch b goes to cache row  */
/*    past[b] + s of both caches (rotated K, V unchanged); rows outside the */
/*    new tokens are left as they are; a token whose row falls outside      */
/*    [0, max_len) is not stored (counted in *n_skip);                      */
/*  - without position_ids the position of token s is past[b] + s, or s    */
/*    when past is NULL (the new tokens follow the cached ones);            */
/*  - without a cache the rotated K goes to k_out (B, S, Nkv*H) and V is    */
/*    not touched.                                                          */
/* Returns 0, or 1 on a malformed argument set.                             */
/* ------------------------------------------------------------------------ */
static void rope_one_head(int dt, int interleaved, int64_t H, int64_t rd, const void* x, int64_t xb,
                          void* y, int64_t yb, const void* cos_t, const void* sin_t, int64_t crow,
                          int valid) {
  int64_t half = rd / 2;
  if (!valid) {
    for (int64_t j = 0; j < H; ++j) cp(dt, x, xb + j, y, yb + j);
    return;
  }
  for (int64_t i = 0; i < half; ++i) {
    int64_t j0, j1;
    pair_elems(interleaved, half, i, &j0, &j1);
    rotate_store(dt, y, yb + j0, yb + j1, ld(dt, x, xb + j0), ld(dt, x, xb + j1),
                 ld(dt, cos_t, crow + i), ld(dt, sin_t, crow + i));
  }
  for (int64_t j = rd; j < H; ++j) cp(dt, x, xb + j, y, yb + j);
}

/* One head rotated as oracle_mrope_map rotates it: pair i takes the
   position of its stream map[i] (p3[0..2] = t, h, w); a position outside
   [0, cache_rows) copies the pair through (counted in *oor); otherwise the
   coefficients are scaled and rounded to T before the rotation. */
static void mrope_one_head(int dt, int interleaved, int64_t H, int64_t rd, const void* x, int64_t xb,
                           void* y, int64_t yb, const void* cos_t, const void* sin_t, int64_t cache_rows,
                           const int64_t* p3, const uint8_t* map, float scale, int64_t* oor) {
  int64_t half = rd / 2;
  for (int64_t i = 0; i < half; ++i) {
    int64_t j0, j1;
    pair_elems(interleaved, half, i, &j0, &j1);
    const int64_t p = p3[map[i]];
    if (p < 0 || p >= cache_rows) {
      cp(dt, x, xb + j0, y, yb + j0);
      cp(dt, x, xb + j1, y, yb + j1);
      ++*oor;
      continue;
    }
    const double c = round_to(dt, ld(dt, cos_t, p * half + i) * (double)scale);
    const double sn = round_to(dt, ld(dt, sin_t, p * half + i) * (double)scale);
    rotate_store(dt, y, yb + j0, yb + j1, ld(dt, x, xb + j0), ld(dt, x, xb + j1), c, sn);
  }
  for (int64_t j = rd; j < H; ++j) cp(dt, x, xb + j, y, yb + j);
}

/* RMS normalisation of one head (H elements at x + xb) followed by the
   per-channel weight, into z[0..H): z_j = T(w_j * T(x_j * r)) with
   r = 1 / sqrt(mean_j(x_j^2) + eps), the mean and r in binary64. */
static void rms_norm_head(int dt, const void* x, int64_t xb, int64_t H, const void* w, double eps,
                          void* z) {
  double ss = 0.0;
  for (int64_t j = 0; j < H; ++j) {
    double v = ld(dt, x, xb + j);
    ss += v * v;
  }
  double r = 1.0 / sqrt(ss / (double)H + eps);
  for (int64_t j = 0; j < H; ++j) {
    double n = round_to(dt, ld(dt, x, xb + j) * r);
    st(dt, z, j, n * ld(dt, w, j));
  }
}

/* pos3 non-NULL: M-RoPE heads (mrope_one_head with map and scale; pos is
   not used and *n_oor counts pairs); otherwise RotaryEmbedding heads. */
static int qkv_core(int dt, int64_t B, int64_t S, int64_t Nq, int64_t Nkv, int64_t H, int interleaved,
                    int64_t rotary_dim, const void* q, const void* k, const void* v,
                    const void* q_weight, const void* k_weight, double eps, const void* cos_t,
                    const void* sin_t, int64_t cache_rows, const int64_t* pos, const int64_t* pos3,
                    const uint8_t* map, float scale, const int32_t* past, void* q_out, void* k_out,
                    void* k_cache, void* v_cache, int64_t max_len, int64_t* n_oor, int64_t* n_skip) {
  if (B < 0 || S < 0 || Nq < 1 || Nkv < 1 || Nq % Nkv || H < 2 || H % 2) return 1;
  int64_t rd = rotary_dim ? rotary_dim : H;
  if (rd % 2 || rd > H || rd <= 0) return 1;
  int packed = (k == NULL && v == NULL);
  int cache = (k_cache != NULL);
  if (cache && (v_cache == NULL || past == NULL || max_len < 1)) return 1;
  if (!cache && k_out == NULL) return 1;
  if (!packed && (k == NULL || (cache && v == NULL))) return 1;
  int norm = (q_weight != NULL);
  if (norm && (k_weight == NULL || !(eps >= 0))) return 1;
  int64_t half = rd / 2;
  int64_t Ntot = Nq + 2 * Nkv;
  int64_t oor = 0, skip = 0;
  /* normalised head (rotation input) when RMSNorm comes first */
  void* zq = norm ? malloc((size_t)H * 8) : NULL;
  if (norm && zq == NULL) return 1;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t s = 0; s < S; ++s) {
      int64_t tok = b * S + s;
      int64_t p = pos ? pos[tok] : (past ? (int64_t)past[b] + s : s);
      int64_t p3[3] = {0, 0, 0};
      if (pos3)
        for (int st3 = 0; st3 < 3; ++st3) p3[st3] = pos3[st3 * B * S + tok];
      int valid = (p >= 0 && p < cache_rows);
      if (!valid && !pos3) ++oor;
      int64_t crow = p * half;
      for (int64_t n = 0; n < Nq; ++n) {
        int64_t src = packed ? (tok * Ntot + n) * H : (tok * Nq + n) * H;
        const void* qs = q;
        if (norm) {
          rms_norm_head(dt, q, src, H, q_weight, eps, zq);
          qs = zq;
          src = 0;
        }
        if (pos3)
          mrope_one_head(dt, interleaved, H, rd, qs, src, q_out, (tok * Nq + n) * H, cos_t, sin_t,
                         cache_rows, p3, map, scale, &oor);
        else
          rope_one_head(dt, interleaved, H, rd, qs, src, q_out, (tok * Nq + n) * H, cos_t, sin_t, crow,
                        valid);
      }
      int64_t row = cache ? (int64_t)past[b] + s : 0;
      int store = !cache || (row >= 0 && row < max_len);
      if (cache && !store) ++skip;
      for (int64_t n = 0; n < Nkv; ++n) {
        const void* ks = packed ? q : k;
        int64_t ksrc = packed ? (tok * Ntot + Nq + n) * H : (tok * Nkv + n) * H;
        if (norm && (!cache || store)) {
          rms_norm_head(dt, ks, ksrc, H, k_weight, eps, zq);
          ks = zq;
          ksrc = 0;
        }
        if (!cache) {
          if (pos3)
            mrope_one_head(dt, interleaved, H, rd, ks, ksrc, k_out, (tok * Nkv + n) * H, cos_t, sin_t,
                           cache_rows, p3, map, scale, &oor);
          else
            rope_one_head(dt, interleaved, H, rd, ks, ksrc, k_out, (tok * Nkv + n) * H, cos_t, sin_t,
                          crow, valid);
          continue;
        }
        if (!store) continue;
        int64_t dst = ((b * Nkv + n) * max_len + row) * H;
        if (pos3)
          mrope_one_head(dt, interleaved, H, rd, ks, ksrc, k_cache, dst, cos_t, sin_t, cache_rows, p3, map,
                         scale, &oor);
        else
          rope_one_head(dt, interleaved, H, rd, ks, ksrc, k_cache, dst, cos_t, sin_t, crow, valid);
        const void* vs = packed ? q : v;
        int64_t vsrc = packed ? (tok * Ntot + Nq + Nkv + n) * H : (tok * Nkv + n) * H;
        for (int64_t j = 0; j < H; ++j) cp(dt, vs, vsrc + j, v_cache, dst + j);
      }
    }
  }
  free(zq);
  if (n_oor) *n_oor = oor;
  if (n_skip) *n_skip = skip;
  return 0;
}

int oracle_rope_qkv(int dt, int64_t B, int64_t S, int64_t Nq, int64_t Nkv, int64_t H,
                    int interleaved, int64_t rotary_dim, const void* q, const void* k,
                    const void* v, const void* cos_t, const void* sin_t, int64_t cache_rows,
                    const int64_t* pos, const int32_t* past, void* q_out, void* k_out,
                    void* k_cache, void* v_cache, int64_t max_len, int64_t* n_oor,
                    int64_t* n_skip) {
  return qkv_core(dt, B, S, Nq, Nkv, H, interleaved, rotary_dim, q, k, v, NULL, NULL, 0.0, cos_t,
                  sin_t, cache_rows, pos, NULL, NULL, 1.0f, past, q_out, k_out, k_cache, v_cache, max_len,
                  n_oor, n_skip);
}

/* ------------------------------------------------------------------------ */
/* The same, with each Q and K head RMS-normalised before the rotation.     */
/* [PR] Qwen3 Architecture (QK-Norm): Qwen3 applies RMSNorm to Q and K      */
/* after the projection and reshape and before RoPE; Verification counts    */
/* the SimplifiedLayerNormalization (RMSNorm) nodes it fuses.               */
/* Reading (the pages name RMSNorm without printing it): over the head's H  */
/* elements, r = 1/sqrt(mean(x^2) + eps); the normalised value x*r is       */
/* rounded to T, multiplied by the head-size weight (q_weight for Q heads,  */
/* k_weight for K heads) and rounded to T again -- the modelling code casts */
/* back to the activation type before the weight -- and that z is what the  */
/* rotation of oracle_rope_qkv receives (an out-of-range position copies z  */
/* through; the tail past rd is z). V is not normalised.                    */
/* ------------------------------------------------------------------------ */
int oracle_rope_qkv_rmsnorm(int dt, int64_t B, int64_t S, int64_t Nq, int64_t Nkv, int64_t H,
                            int interleaved, int64_t rotary_dim, const void* q, const void* k,
                            const void* v, const void* q_weight, const void* k_weight, double eps,
                            const void* cos_t, const void* sin_t, int64_t cache_rows,
                            const int64_t* pos, const int32_t* past, void* q_out, void* k_out,
                            void* k_cache, void* v_cache, int64_t max_len, int64_t* n_oor,
                            int64_t* n_skip) {
  if (q_weight == NULL || k_weight == NULL) return 1;
  return qkv_core(dt, B, S, Nq, Nkv, H, interleaved, rotary_dim, q, k, v, q_weight, k_weight, eps,
                  cos_t, sin_t, cache_rows, pos, NULL, NULL, 1.0f, past, q_out, k_out, k_cache, v_cache,
                  max_len, n_oor, n_skip);
}

/* ------------------------------------------------------------------------ */
/* Q and K rotation with M-RoPE, grouped-query heads and the cache append.  */
/* [MR] Description, Inputs/positionIds and Attributes: multimodal RoPE     */
/* with three position streams (t, h, w) that mrope_section / mrope_layout  */
/* assign to the half-rotary indices, the scale applied to the gathered     */
/* coefficient, and pairs whose stream position is out of range copied     */
/* through. [SA] Description, Inputs and Attributes: Q and K rotated in one */
/* pass for grouped-query heads, K and V appended to the caches. [PR] Qwen3 */
/* Architecture: QK-Norm (RMSNorm on Q and K) before the rotary step.       */
/* Reading: every Q and K head is rotated exactly as oracle_mrope_map       */
/* rotates one head of a rank-3 X with the token's three positions          */
/* pos3[k, b, s]; with q_weight and k_weight the head is first normalised   */
/* as in oracle_rope_qkv_rmsnorm; the cache append, the k_out form and V    */
/* are those of oracle_rope_qkv. Positions are required (three streams      */
/* cannot follow from the past lengths). *n_oor counts Q and K pairs copied */
/* through (in the K heads that are written).                               */
/* ------------------------------------------------------------------------ */
int oracle_mrope_qkv(int dt, int64_t B, int64_t S, int64_t Nq, int64_t Nkv, int64_t H, int interleaved,
                     int64_t rotary_dim, const void* q, const void* k, const void* v,
                     const void* q_weight, const void* k_weight, double eps, const void* cos_t,
                     const void* sin_t, int64_t cache_rows, const int64_t* pos3, const int32_t* sec,
                     int layout, float scale, const int32_t* past, void* q_out, void* k_out,
                     void* k_cache, void* v_cache, int64_t max_len, int64_t* n_oor, int64_t* n_skip) {
  if (pos3 == NULL || sec == NULL || H < 2) return 1;
  if ((q_weight == NULL) != (k_weight == NULL)) return 1;
  int64_t rd = rotary_dim ? rotary_dim : H;
  int64_t half = rd / 2;
  if (half <= 0 || half > 65536) return 1;
  uint8_t* map = malloc((size_t)half);
  if (map == NULL) return 1;
  int rc = oracle_mrope_stream_map(sec, layout, half, map);
  if (rc == 0)
    rc = qkv_core(dt, B, S, Nq, Nkv, H, interleaved, rotary_dim, q, k, v, q_weight, k_weight, eps, cos_t,
                  sin_t, cache_rows, NULL, pos3, map, scale, past, q_out, k_out, k_cache, v_cache, max_len,
                  n_oor, n_skip);
  free(map);
  return rc;
}
