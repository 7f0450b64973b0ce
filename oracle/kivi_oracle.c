/*
 * kivi_oracle.c -- plain, slow, single-threaded CPU oracle for KIVI-style
 * group-affine KV-cache quantization and decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it follows (VeloxQuant-MLX pages):
 *  - Changelog, v0.8.0 "New", KIVI entry: keys are quantized per channel,
 *    values per token, asymmetric group quantization, an fp16 residual window
 *    (`residual_length`) and a group size (`kivi_group_size`, default 32).
 *  - Changelog, v0.42.0 "Added", scalar_fused_decode_attend: the cache is
 *    integer codes plus one (scale, zero) pair per group from the group's
 *    min/max; attention runs over k_hat/v_hat rebuilt from those codes, with
 *    softmax accumulated in higher precision than fp16.
 *  - Method overview, AgeTieredKV entry: the residual window is gated purely
 *    by recency and the group quantizer is a shared min/max quantizer.
 *  - Changelog, v0.28.0 (NSNQuant-adapted): the fp16 residual buffer is
 *    flushed in whole chunks ("chunk-flush ... KIVI's idiom"), and prefill
 *    and decode produce identical quantized state.
 * The pages print no formula; the fp32 formula used here is the plain reading
 * (scale = (max-min)/(2^b-1); code = clamp(rint((x-min)/scale), 0, 2^b-1);
 * scale stored as fp16 round-to-nearest-even, zero = min stored exactly,
 * with a minimum of -0.0 stored as +0.0 and a zero range as the scale +0.0).
 *
 * Precision: quantization arithmetic in IEEE fp32 exactly as written (this
 * file must be compiled without fast-math and with -ffp-contract=off);
 * dequantization and attention in double (k_hat = code*scale + zero is exact
 * in double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef _Float16 half_t;

static float h2f(uint16_t bits) {
  half_t h;
  memcpy(&h, &bits, sizeof h);
  return (float)h;
}

static uint16_t f2h(float f) {
  half_t h = (half_t)f; /* IEEE conversion, round to nearest even */
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

/* ------------------------------------------------------------------------ */
/* The group quantizer (one group of n values).                              */
/* ------------------------------------------------------------------------ */

/* x[i*stride], i < n: fp32 copies of fp16 inputs.  Writes codes[i*cstride],
 * the fp32 scale, and the stored fp16 scale / zero bit patterns. */
static void quant_group(const float *x, long stride, int n, int bits,
                        uint8_t *codes, long cstride, float *scale32,
                        uint16_t *s16, uint16_t *z16) {
  const int levels = (1 << bits) - 1;
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    float v = x[(long)i * stride];
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  /* A group minimum of -0.0 is stored as +0.0 (the pages leave signed zero
   * open; -0 + +0 = +0 under round-to-nearest).  No code changes: x - min
   * is the same number either way.  Likewise a zero range (a constant
   * group, possibly of mixed-sign zeros) gives the scale +0.0 whatever the
   * order of its elements: mx - mn alone is -0.0 when the first element,
   * which the scan keeps as the maximum among equal zeros, is -0.0. */
  mn = mn + 0.0f;
  float range = (mx - mn) + 0.0f;
  float scale = range / (float)levels;
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if (scale != 0.0f) {
      float diff = x[(long)i * stride] - mn;
      float t = diff / scale;
      float r = nearbyintf(t); /* default rounding mode: ties to even */
      if (r < 0.0f) r = 0.0f;
      if (r > (float)levels) r = (float)levels;
      c = (int)r;
    }
    codes[(long)i * cstride] = (uint8_t)c;
  }
  if (scale32) *scale32 = scale;
  *s16 = f2h(scale);
  *z16 = f2h(mn);
}

void orc_quant_group_f32(const float *x, int n, int bits, uint8_t *codes,
                         float *scale32, uint16_t *s16, uint16_t *z16) {
  quant_group(x, 1, n, bits, codes, 1, scale32, s16, z16);
}

/* Sub-byte packing: the code of element e of a row sits in byte e*b/8 at bit
 * (e*b) mod 8, least significant bits first (2-bit: 4 per byte, 4-bit: 2 per
 * byte, 8-bit: 1 per byte). */
void orc_pack_codes(const uint8_t *codes, int n, int bits, uint8_t *out) {
  int nbytes = (n * bits + 7) / 8;
  memset(out, 0, (size_t)nbytes);
  for (int e = 0; e < n; ++e) {
    int bit = e * bits;
    out[bit / 8] |= (uint8_t)(codes[e] << (bit % 8));
  }
}

void orc_unpack_codes(const uint8_t *packed, int n, int bits, uint8_t *codes) {
  int mask = (1 << bits) - 1;
  for (int e = 0; e < n; ++e) {
    int bit = e * bits;
    codes[e] = (uint8_t)((packed[bit / 8] >> (bit % 8)) & mask);
  }
}

/* ------------------------------------------------------------------------ */
/* The cache.                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct orc_cache {
  int B, Hq, Hkv, D, bits, g, R, max_seq;
  int Tcap; /* quantized-token capacity, a multiple of g */
  int Rcap; /* residual capacity, R + g */
  int row;  /* packed bytes per token row: D*bits/8 */
  uint8_t *Kc, *Vc;        /* [B][Hkv][Tcap][row] */
  uint16_t *Ks, *Kz;       /* [B][Hkv][Tcap/g][D] */
  uint16_t *Vs, *Vz;       /* [B][Hkv][Tcap][D/g] */
  uint16_t *Kr, *Vr;       /* [B][Hkv][Rcap][D]; slot i holds token Tq+i */
  int32_t *S, *Tq, *nres;  /* [B] */
  /* KIVI-Sink (0 sinks = plain KIVI): per (b, h) the positions of the sink
   * tokens, ascending, -1 in unused slots, and their fp16 key / value rows */
  int n_sink;
  int32_t *sink_pos;       /* [B][Hkv][n_sink] */
  uint16_t *sink_k, *sink_v; /* [B][Hkv][n_sink][D] */
  /* Kitty (0 = plain KIVI): kitty_hi channels of every key group get 4-bit
   * codes, the other D - kitty_hi 2-bit; values stay fp16.  Per (b, h,
   * channel) the running sums of the quantized keys as integers in units of
   * 2^-24 (every fp16 value is an integer multiple of 2^-24). */
  int kitty_hi;
  int krow;                /* key code bytes per token row */
  uint32_t *Kmask;         /* [B][Hkv][Tcap/g][D/32] 4-bit channels */
  uint16_t *Vf;            /* [B][Hkv][Tcap][D] fp16 values */
  int64_t *ksum;           /* [B][Hkv][D] */
  unsigned __int128 *ksq;  /* [B][Hkv][D] */
  /* AgeTieredKV (tier == NULL: off): a quantized group's width follows its
   * age, counted from its newest token: age < age_b1 -> age_bits[0], age <
   * age_b2 -> age_bits[1], else age_bits[2].  Codes sit in the first
   * D * bits / 8 bytes of a D-byte row (the rest zero); tier[] is each
   * group's current tier. */
  int age_b1, age_b2, age_bits[3];
  int8_t *tier;            /* [B][Hkv][Tcap/g] */
} orc_cache;

static int n_quantized(int S, int R, int g) {
  /* Quantized prefix length for a sequence of S tokens: whole groups only,
   * leaving between R and R+g-1 tokens (or all S, when S < R) in fp16. */
  if (S < R) return 0;
  return g * ((S - R) / g);
}

orc_cache *orc_new(int B, int Hq, int Hkv, int D, int bits, int g, int R,
                   int max_seq) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || g <= 0 || R < 0 ||
      max_seq < 0)
    return NULL;
  if (bits != 2 && bits != 4 && bits != 8) return NULL;
  if (Hq % Hkv != 0 || D % g != 0 || (D * bits) % 8 != 0) return NULL;
  if (D > 4096) return NULL; /* per-row scratch below is sized for 4096 */
  orc_cache *c = (orc_cache *)calloc(1, sizeof *c);
  if (!c) return NULL;
  c->B = B; c->Hq = Hq; c->Hkv = Hkv; c->D = D; c->bits = bits; c->g = g;
  c->R = R; c->max_seq = max_seq;
  c->Tcap = ((max_seq + g - 1) / g) * g;
  if (c->Tcap == 0) c->Tcap = g;
  c->Rcap = R + g;
  c->row = D * bits / 8;
  size_t bh = (size_t)B * Hkv;
  c->Kc = (uint8_t *)calloc(bh * c->Tcap * c->row, 1);
  c->Vc = (uint8_t *)calloc(bh * c->Tcap * c->row, 1);
  c->Ks = (uint16_t *)calloc(bh * (c->Tcap / g) * D, 2);
  c->Kz = (uint16_t *)calloc(bh * (c->Tcap / g) * D, 2);
  c->Vs = (uint16_t *)calloc(bh * c->Tcap * (D / g), 2);
  c->Vz = (uint16_t *)calloc(bh * c->Tcap * (D / g), 2);
  c->Kr = (uint16_t *)calloc(bh * c->Rcap * D, 2);
  c->Vr = (uint16_t *)calloc(bh * c->Rcap * D, 2);
  c->S = (int32_t *)calloc(B, 4);
  c->Tq = (int32_t *)calloc(B, 4);
  c->nres = (int32_t *)calloc(B, 4);
  if (!c->Kc || !c->Vc || !c->Ks || !c->Kz || !c->Vs || !c->Vz || !c->Kr ||
      !c->Vr || !c->S || !c->Tq || !c->nres) {
    free(c->Kc); free(c->Vc); free(c->Ks); free(c->Kz); free(c->Vs);
    free(c->Vz); free(c->Kr); free(c->Vr); free(c->S); free(c->Tq);
    free(c->nres); free(c);
    return NULL;
  }
  return c;
}

void orc_free(orc_cache *c) {
  if (!c) return;
  free(c->Kc); free(c->Vc); free(c->Ks); free(c->Kz); free(c->Vs);
  free(c->Vz); free(c->Kr); free(c->Vr); free(c->S); free(c->Tq);
  free(c->nres); free(c->sink_pos); free(c->sink_k); free(c->sink_v);
  free(c->Kmask); free(c->Vf); free(c->ksum); free(c->ksq); free(c->tier);
  free(c);
}

/* AgeTieredKV (method overview, AgeTieredKV entry): three tiers of the
 * shared min/max group quantizer chosen by token age against two
 * boundaries.  Call on a fresh cache of bits = 8 (its rows hold the widest
 * tier) before orc_quantize.  0 < b1 < b2, multiples of g; widths from
 * {2, 4, 8}, non-increasing.  Returns 0, or -1. */
int orc_set_age(orc_cache *c, int b1, int b2, int bits0, int bits1, int bits2) {
  const int ok_bits[3] = {bits0, bits1, bits2};
  if (c->bits != 8 || c->n_sink || c->Kmask || c->tier) return -1;
  if (b1 <= 0 || b2 <= b1 || b1 % c->g || b2 % c->g) return -1;
  for (int i = 0; i < 3; ++i) {
    if (ok_bits[i] != 2 && ok_bits[i] != 4 && ok_bits[i] != 8) return -1;
    if (i && ok_bits[i] > ok_bits[i - 1]) return -1;
    c->age_bits[i] = ok_bits[i];
  }
  c->age_b1 = b1;
  c->age_b2 = b2;
  c->tier = (int8_t *)calloc((size_t)c->B * c->Hkv * (c->Tcap / c->g), 1);
  return c->tier ? 0 : -1;
}

static int age_tier(const orc_cache *c, int S, int G) {
  const int age = S - (G + 1) * c->g; /* tokens newer than the group's last */
  return age < c->age_b1 ? 0 : (age < c->age_b2 ? 1 : 2);
}

/* codes of a row at width w (LSB-first, D * w / 8 bytes), rest zero */
static void age_put_row(uint8_t *row, const uint8_t *codes, int D, int w) {
  memset(row, 0, (size_t)D);
  orc_pack_codes(codes, D, w, row);
}

/* Move group G of (b, h) one tier down: rebuild its keys and values in fp32
 * (code * scale rounded, then + zero rounded) and quantize them again at
 * the next tier's width with the same group quantizer. */
static void age_demote(orc_cache *c, int b, int h, int G) {
  const int D = c->D, g = c->g;
  size_t bh = (size_t)b * c->Hkv + h;
  int8_t *tr = c->tier + bh * (c->Tcap / g) + G;
  const int wf = c->age_bits[*tr], wt = c->age_bits[*tr + 1];
  float *x = (float *)malloc(sizeof(float) * (size_t)g * D);
  uint8_t *codes = (uint8_t *)malloc((size_t)g * D);
  uint8_t row[4096];
  /* keys, per channel */
  for (int i = 0; i < g; ++i) {
    const uint8_t *r = c->Kc + (bh * c->Tcap + (size_t)G * g + i) * c->row;
    orc_unpack_codes(r, D, wf, row);
    for (int ch = 0; ch < D; ++ch) {
      float sc = h2f(c->Ks[(bh * (c->Tcap / g) + G) * D + ch]);
      float z = h2f(c->Kz[(bh * (c->Tcap / g) + G) * D + ch]);
      float prod = (float)row[ch] * sc;
      x[(size_t)i * D + ch] = prod + z;
    }
  }
  for (int ch = 0; ch < D; ++ch) {
    uint16_t s16, z16;
    quant_group(x + ch, D, g, wt, codes + ch, D, NULL, &s16, &z16);
    c->Ks[(bh * (c->Tcap / g) + G) * D + ch] = s16;
    c->Kz[(bh * (c->Tcap / g) + G) * D + ch] = z16;
  }
  for (int i = 0; i < g; ++i)
    age_put_row(c->Kc + (bh * c->Tcap + (size_t)G * g + i) * c->row,
                codes + (size_t)i * D, D, wt);
  /* values, per token over groups of g channels */
  for (int i = 0; i < g; ++i) {
    size_t t = (size_t)G * g + i;
    uint8_t *r = c->Vc + (bh * c->Tcap + t) * c->row;
    orc_unpack_codes(r, D, wf, row);
    float xv[4096];
    uint8_t cv[4096];
    for (int ch = 0; ch < D; ++ch) {
      float sc = h2f(c->Vs[(bh * c->Tcap + t) * (D / g) + ch / g]);
      float z = h2f(c->Vz[(bh * c->Tcap + t) * (D / g) + ch / g]);
      float prod = (float)row[ch] * sc;
      xv[ch] = prod + z;
    }
    for (int j = 0; j < D / g; ++j) {
      uint16_t s16, z16;
      quant_group(xv + j * g, 1, g, wt, cv + j * g, 1, NULL, &s16, &z16);
      c->Vs[(bh * c->Tcap + t) * (D / g) + j] = s16;
      c->Vz[(bh * c->Tcap + t) * (D / g) + j] = z16;
    }
    age_put_row(r, cv, D, wt);
  }
  *tr += 1;
  free(x);
  free(codes);
}

/* after a change of length: every group of b demoted to its age's tier */
static void age_update(orc_cache *c, int b) {
  if (!c->tier) return;
  for (int h = 0; h < c->Hkv; ++h)
    for (int G = 0; G < c->Tq[b] / c->g; ++G) {
      const int want = age_tier(c, c->S[b], G);
      while (c->tier[((size_t)b * c->Hkv + h) * (c->Tcap / c->g) + G] < want)
        age_demote(c, b, h, G);
    }
}

/* Kitty (changelog v0.11.0 "New"): channel-wise mixed-precision keys.  For
 * every key group the hi channels with the largest running variance get
 * 4-bit codes, the rest 2-bit; values are kept in fp16.  Call on a fresh
 * cache of bits = 2, before orc_quantize.  hi in [0, D], a multiple of 8.
 * Returns 0, or -1 on bad arguments or a failed allocation. */
int orc_set_kitty(orc_cache *c, int hi) {
  if (hi < 0 || hi > c->D || hi % 8 != 0 || c->bits != 2 || c->n_sink != 0 ||
      c->D % 32 != 0 || c->max_seq > (1 << 20) || c->Kmask)
    return -1;
  c->kitty_hi = hi;
  c->krow = (hi * 4 + (c->D - hi) * 2) / 8;
  size_t bh = (size_t)c->B * c->Hkv;
  free(c->Kc);
  c->Kc = (uint8_t *)calloc(bh * c->Tcap * c->krow, 1);
  c->Kmask = (uint32_t *)calloc(bh * (c->Tcap / c->g) * (c->D / 32), 4);
  c->Vf = (uint16_t *)calloc(bh * c->Tcap * c->D, 2);
  c->ksum = (int64_t *)calloc(bh * c->D, 8);
  c->ksq = (unsigned __int128 *)calloc(bh * c->D, sizeof(unsigned __int128));
  if (!c->Kc || !c->Kmask || !c->Vf || !c->ksum || !c->ksq) return -1;
  return 0;
}

/* fp16 bits -> the value as an integer multiple of 2^-24 (exact) */
static int64_t f16_units(uint16_t bits) {
  int e = (bits >> 10) & 31;
  int64_t m = bits & 1023;
  if (e == 0) return (bits & 0x8000) ? -m : m;      /* subnormal: m 2^-24 */
  int64_t v = (m | 1024) << (e - 1);                /* (1024 + m) 2^(e-25) */
  return (bits & 0x8000) ? -v : v;
}

/* Kitty: rank the channels of key group G of (b, h) after adding the
 * group's keys (rows krow(ctx, i)) to the running sums: the hi channels
 * with the largest N sum(x^2) - (sum x)^2 (N times the population
 * variance, exact in 128-bit integers; the smaller channel first on equal
 * values), as a bit mask in mask[D/32]. */
static void kitty_rank(orc_cache *c, int b, int h, int G, const uint16_t **rows,
                       uint32_t *mask) {
  const int D = c->D, g = c->g;
  size_t bh = (size_t)b * c->Hkv + h;
  int64_t *ks = c->ksum + bh * D;
  unsigned __int128 *kq = c->ksq + bh * D;
  unsigned __int128 *var = (unsigned __int128 *)malloc(sizeof(unsigned __int128) * D);
  const unsigned __int128 N = (unsigned __int128)((G + 1) * g);
  for (int ch = 0; ch < D; ++ch) {
    for (int i = 0; i < g; ++i) {
      int64_t m = f16_units(rows[i][ch]);
      ks[ch] += m;
      kq[ch] += (unsigned __int128)((__int128)m * m);
    }
    __int128 sm = ks[ch];
    unsigned __int128 s2 = (unsigned __int128)(sm < 0 ? -sm : sm);
    var[ch] = N * kq[ch] - s2 * s2;
  }
  for (int w = 0; w < D / 32; ++w) mask[w] = 0;
  for (int ch = 0; ch < D; ++ch) {
    int rank = 0; /* channels ranked before ch */
    for (int o = 0; o < D; ++o)
      if (var[o] > var[ch] || (var[o] == var[ch] && o < ch)) ++rank;
    if (rank < c->kitty_hi) mask[ch / 32] |= 1u << (ch % 32);
  }
  free(var);
}

/* KIVI-Sink (changelog v0.9.0 "New"): tokens with the largest key L2 norms
 * are kept in fp16 and left out of the groups' min/max.  Call before
 * orc_quantize; n_sink = 0 is plain KIVI.  Returns 0, or -1 on a bad count
 * or a failed allocation. */
int orc_set_sinks(orc_cache *c, int n_sink) {
  if (n_sink < 0 || n_sink > 64) return -1;
  free(c->sink_pos); free(c->sink_k); free(c->sink_v);
  c->sink_pos = NULL; c->sink_k = NULL; c->sink_v = NULL;
  c->n_sink = n_sink;
  if (n_sink == 0) return 0;
  size_t slots = (size_t)c->B * c->Hkv * n_sink;
  c->sink_pos = (int32_t *)malloc(4 * slots);
  c->sink_k = (uint16_t *)calloc(slots * c->D, 2);
  c->sink_v = (uint16_t *)calloc(slots * c->D, 2);
  if (!c->sink_pos || !c->sink_k || !c->sink_v) return -1;
  for (size_t i = 0; i < slots; ++i) c->sink_pos[i] = -1;
  return 0;
}

static int is_sink(const orc_cache *c, int b, int h, int t) {
  const int32_t *sp = c->sink_pos + ((size_t)b * c->Hkv + h) * c->n_sink;
  for (int k = 0; k < c->n_sink; ++k)
    if (sp[k] == t) return 1;
  return 0;
}

/* Squared L2 norm of an fp16 key row in fp32, channel 0 first (each square
 * of an fp16 value is exact in fp32; the sums round to nearest). */
static float key_norm2(const uint16_t *row, int D) {
  float acc = 0.0f;
  for (int ch = 0; ch < D; ++ch) {
    float x = h2f(row[ch]);
    acc = acc + x * x;
  }
  return acc;
}

/* Sinks of one (b, h): the min(n_sink, S) tokens among the S prefill tokens
 * with the largest key norms (a larger norm first, an earlier position on
 * equal norms), stored by ascending position with their fp16 rows. */
static void pick_sinks(orc_cache *c, int b, int h, const uint16_t *Kbh,
                       const uint16_t *Vbh, int S) {
  const int D = c->D, n = c->n_sink;
  size_t base = ((size_t)b * c->Hkv + h) * n;
  int32_t *sp = c->sink_pos + base;
  int count = 0;
  for (int k = 0; k < n; ++k) sp[k] = -1;
  char *taken = (char *)calloc(S > 0 ? S : 1, 1);
  for (int k = 0; k < n && k < S; ++k) {
    int best = -1;
    float bn = 0.0f;
    for (int t = 0; t < S; ++t) {
      if (taken[t]) continue;
      float nt = key_norm2(Kbh + (size_t)t * D, D);
      if (best < 0 || nt > bn) { best = t; bn = nt; }
    }
    taken[best] = 1;
    sp[count++] = best;
  }
  free(taken);
  /* ascending positions */
  for (int i = 1; i < count; ++i)
    for (int j = i; j > 0 && sp[j - 1] > sp[j]; --j) {
      int32_t tmp = sp[j]; sp[j] = sp[j - 1]; sp[j - 1] = tmp;
    }
  for (int k = 0; k < count; ++k) {
    memcpy(c->sink_k + (base + k) * D, Kbh + (size_t)sp[k] * D, 2 * (size_t)D);
    memcpy(c->sink_v + (base + k) * D, Vbh + (size_t)sp[k] * D, 2 * (size_t)D);
  }
}

/* Quantize one key group (g tokens, all D channels, per channel) and the
 * values of the same g tokens (per token, groups of g channels).  ktok/vtok
 * return a pointer to the fp16 row of token i of the group. */
typedef const uint16_t *(*row_fn)(const void *ctx, int i);

static void quantize_group_of_tokens(orc_cache *c, int b, int h, int G,
                                     row_fn krow, row_fn vrow,
                                     const void *ctx) {
  const int D = c->D, g = c->g;
  size_t bh = (size_t)b * c->Hkv + h;
  if (c->Kmask) {
    /* Kitty: rank, then per channel 4- or 2-bit codes over the g tokens;
     * row layout: the 4-bit channels' codes in ascending channel order
     * (LSB-first), then the 2-bit channels' */
    const uint16_t *rows[4096];
    for (int i = 0; i < g; ++i) rows[i] = krow(ctx, i);
    uint32_t *mask = c->Kmask + (bh * (c->Tcap / g) + G) * (D / 32);
    kitty_rank(c, b, h, G, rows, mask);
    float *xk = (float *)malloc(sizeof(float) * g);
    uint8_t *ck = (uint8_t *)malloc((size_t)g * D);
    for (int ch = 0; ch < D; ++ch) {
      const int hi = (mask[ch / 32] >> (ch % 32)) & 1;
      uint16_t s16, z16;
      for (int i = 0; i < g; ++i) xk[i] = h2f(rows[i][ch]);
      uint8_t cc[4096];
      quant_group(xk, 1, g, hi ? 4 : 2, cc, 1, NULL, &s16, &z16);
      for (int i = 0; i < g; ++i) ck[(size_t)i * D + ch] = cc[i];
      c->Ks[(bh * (c->Tcap / g) + G) * D + ch] = s16;
      c->Kz[(bh * (c->Tcap / g) + G) * D + ch] = z16;
    }
    for (int i = 0; i < g; ++i) {
      size_t t = (size_t)G * g + i;
      uint8_t *row = c->Kc + (bh * c->Tcap + t) * c->krow;
      int bit = 0;
      memset(row, 0, (size_t)c->krow);
      for (int pass = 0; pass < 2; ++pass)   /* 4-bit channels, then 2-bit */
        for (int ch = 0; ch < D; ++ch) {
          const int hi = (mask[ch / 32] >> (ch % 32)) & 1;
          if (hi != (pass == 0)) continue;
          row[bit / 8] |= (uint8_t)(ck[(size_t)i * D + ch] << (bit % 8));
          bit += hi ? 4 : 2;
        }
      memcpy(c->Vf + (bh * c->Tcap + t) * D, vrow(ctx, i), 2 * (size_t)D);
    }
    free(xk);
    free(ck);
    return;
  }
  float *x = (float *)malloc(sizeof(float) * (size_t)g * D);
  uint8_t *codes = (uint8_t *)malloc((size_t)g * D);
  if (c->tier) {
    /* AgeTieredKV: a new group enters at the top tier */
    const int w = c->age_bits[0];
    uint8_t *codes2 = (uint8_t *)malloc((size_t)g * D);
    float *xk = (float *)malloc(sizeof(float) * (size_t)g * D);
    for (int i = 0; i < g; ++i) {
      const uint16_t *r = krow(ctx, i);
      for (int ch = 0; ch < D; ++ch) xk[(size_t)i * D + ch] = h2f(r[ch]);
    }
    for (int ch = 0; ch < D; ++ch) {
      uint16_t s16, z16;
      quant_group(xk + ch, D, g, w, codes2 + ch, D, NULL, &s16, &z16);
      c->Ks[(bh * (c->Tcap / g) + G) * D + ch] = s16;
      c->Kz[(bh * (c->Tcap / g) + G) * D + ch] = z16;
    }
    for (int i = 0; i < g; ++i)
      age_put_row(c->Kc + (bh * c->Tcap + (size_t)G * g + i) * c->row,
                  codes2 + (size_t)i * D, D, w);
    for (int i = 0; i < g; ++i) {
      const uint16_t *r = vrow(ctx, i);
      size_t t = (size_t)G * g + i;
      float xv[4096];
      uint8_t cv[4096];
      for (int ch = 0; ch < D; ++ch) xv[ch] = h2f(r[ch]);
      for (int j = 0; j < D / g; ++j) {
        uint16_t s16, z16;
        quant_group(xv + j * g, 1, g, w, cv + j * g, 1, NULL, &s16, &z16);
        c->Vs[(bh * c->Tcap + t) * (D / g) + j] = s16;
        c->Vz[(bh * c->Tcap + t) * (D / g) + j] = z16;
      }
      age_put_row(c->Vc + (bh * c->Tcap + t) * c->row, cv, D, w);
    }
    c->tier[bh * (c->Tcap / g) + G] = 0;
    free(codes2);
    free(xk);
    free(x);
    free(codes);
    return;
  }
  /* sink tokens of this group (KIVI-Sink): left out of every min/max,
   * their codes 0 and their own value groups empty */
  char sink[4096];
  int n_keep = 0;
  for (int i = 0; i < g; ++i) {
    sink[i] = c->n_sink > 0 && is_sink(c, b, h, G * g + i);
    if (!sink[i]) ++n_keep;
  }
  /* keys: per channel over the group's (non-sink) tokens */
  for (int i = 0, k = 0; i < g; ++i) {
    if (sink[i]) continue;
    const uint16_t *r = krow(ctx, i);
    for (int ch = 0; ch < D; ++ch) x[(size_t)k * D + ch] = h2f(r[ch]);
    ++k;
  }
  uint8_t *kept = (uint8_t *)malloc((size_t)(n_keep ? n_keep : 1) * D);
  for (int ch = 0; ch < D; ++ch) {
    uint16_t s16 = 0, z16 = 0; /* a group of sinks only: scale and zero +0 */
    if (n_keep > 0)
      quant_group(x + ch, D, n_keep, c->bits, kept + ch, D, NULL, &s16, &z16);
    c->Ks[(bh * (c->Tcap / g) + G) * D + ch] = s16;
    c->Kz[(bh * (c->Tcap / g) + G) * D + ch] = z16;
  }
  for (int i = 0, k = 0; i < g; ++i) {
    for (int ch = 0; ch < D; ++ch)
      codes[(size_t)i * D + ch] = sink[i] ? 0 : kept[(size_t)k * D + ch];
    if (!sink[i]) ++k;
  }
  free(kept);
  for (int i = 0; i < g; ++i) {
    size_t t = (size_t)G * g + i;
    orc_pack_codes(codes + (size_t)i * D, D, c->bits,
                   c->Kc + (bh * c->Tcap + t) * c->row);
  }
  /* values: per token over groups of g consecutive channels */
  for (int i = 0; i < g; ++i) {
    const uint16_t *r = vrow(ctx, i);
    size_t t = (size_t)G * g + i;
    float xv[4096];
    uint8_t cv[4096];
    for (int ch = 0; ch < D; ++ch) xv[ch] = h2f(r[ch]);
    for (int j = 0; j < D / g; ++j) {
      uint16_t s16 = 0, z16 = 0;
      if (sink[i]) {
        memset(cv + j * g, 0, (size_t)g); /* no member left: scale, zero +0 */
      } else {
        quant_group(xv + j * g, 1, g, c->bits, cv + j * g, 1, NULL, &s16, &z16);
      }
      c->Vs[(bh * c->Tcap + t) * (D / g) + j] = s16;
      c->Vz[(bh * c->Tcap + t) * (D / g) + j] = z16;
    }
    orc_pack_codes(cv, D, c->bits, c->Vc + (bh * c->Tcap + t) * c->row);
  }
  free(x);
  free(codes);
}

typedef struct {
  const uint16_t *base; /* [S_max][D] block of one (b, h) */
  int D, first;
} dense_ctx;

static const uint16_t *dense_row(const void *ctx, int i) {
  const dense_ctx *d = (const dense_ctx *)ctx;
  return d->base + (size_t)(d->first + i) * d->D;
}

typedef struct {
  const dense_ctx *kd, *vd;
} kv_pair_ctx;

static const uint16_t *pair_k(const void *ctx, int i) {
  const kv_pair_ctx *p = (const kv_pair_ctx *)ctx;
  return dense_row(p->kd, i);
}
static const uint16_t *pair_v(const void *ctx, int i) {
  const kv_pair_ctx *p = (const kv_pair_ctx *)ctx;
  return dense_row(p->vd, i);
}

/* Prefill: K, V fp16 [B][Hkv][s_stride][D]; sequence b has seq_lens[b]
 * tokens.  Replaces the whole cache state.  Returns 0, or -1 on a bad length. */
int orc_quantize(orc_cache *c, const uint16_t *K, const uint16_t *V,
                 long s_stride, const int32_t *seq_lens) {
  for (int b = 0; b < c->B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > c->max_seq || seq_lens[b] > s_stride)
      return -1;
  if (c->Kmask) { /* Kitty: the running sums start over */
    memset(c->ksum, 0, sizeof(int64_t) * (size_t)c->B * c->Hkv * c->D);
    memset(c->ksq, 0, sizeof(unsigned __int128) * (size_t)c->B * c->Hkv * c->D);
  }
  for (int b = 0; b < c->B; ++b) {
    int S = seq_lens[b];
    int Tq = n_quantized(S, c->R, c->g);
    c->S[b] = S;
    c->Tq[b] = Tq;
    c->nres[b] = S - Tq;
    for (int h = 0; h < c->Hkv; ++h) {
      size_t off = ((size_t)b * c->Hkv + h) * (size_t)s_stride * c->D;
      if (c->n_sink > 0) pick_sinks(c, b, h, K + off, V + off, S);
      for (int G = 0; G < Tq / c->g; ++G) {
        dense_ctx kd = {K + off, c->D, G * c->g};
        dense_ctx vd = {V + off, c->D, G * c->g};
        kv_pair_ctx p = {&kd, &vd};
        quantize_group_of_tokens(c, b, h, G, pair_k, pair_v, &p);
      }
      size_t bh = (size_t)b * c->Hkv + h;
      for (int i = 0; i < S - Tq; ++i) {
        memcpy(c->Kr + (bh * c->Rcap + i) * c->D,
               K + off + (size_t)(Tq + i) * c->D, 2 * (size_t)c->D);
        memcpy(c->Vr + (bh * c->Rcap + i) * c->D,
               V + off + (size_t)(Tq + i) * c->D, 2 * (size_t)c->D);
      }
    }
    age_update(c, b);
  }
  return 0;
}

/* Decode-time append, done the incremental way: push the new tokens onto
 * the fp16 residual, then flush the oldest whole groups while at least R+g
 * tokens are waiting.  Kn, Vn fp16 [B][Hkv][n_stride][D]. */
int orc_append(orc_cache *c, const uint16_t *Kn, const uint16_t *Vn,
               long n_stride, const int32_t *n_new) {
  for (int b = 0; b < c->B; ++b)
    if (n_new[b] < 0 || n_new[b] > n_stride ||
        (long)c->S[b] + n_new[b] > c->max_seq)
      return -1;
  const int D = c->D;
  for (int b = 0; b < c->B; ++b) {
    int n = n_new[b];
    for (int h = 0; h < c->Hkv; ++h) {
      size_t bh = (size_t)b * c->Hkv + h;
      /* a growing fp16 staging list: old residual followed by new tokens */
      int total = c->nres[b] + n;
      uint16_t *ks = (uint16_t *)malloc(2 * (size_t)D * (total ? total : 1));
      uint16_t *vs = (uint16_t *)malloc(2 * (size_t)D * (total ? total : 1));
      memcpy(ks, c->Kr + bh * c->Rcap * D, 2 * (size_t)D * c->nres[b]);
      memcpy(vs, c->Vr + bh * c->Rcap * D, 2 * (size_t)D * c->nres[b]);
      const uint16_t *kin = Kn + bh * (size_t)n_stride * D;
      const uint16_t *vin = Vn + bh * (size_t)n_stride * D;
      memcpy(ks + (size_t)c->nres[b] * D, kin, 2 * (size_t)D * n);
      memcpy(vs + (size_t)c->nres[b] * D, vin, 2 * (size_t)D * n);
      int head = 0; /* index of the oldest unflushed staged token */
      int Tq = c->Tq[b];
      while (total - head >= c->R + c->g) {
        dense_ctx kd = {ks, D, head};
        dense_ctx vd = {vs, D, head};
        kv_pair_ctx p = {&kd, &vd};
        quantize_group_of_tokens(c, b, h, Tq / c->g, pair_k, pair_v, &p);
        head += c->g;
        Tq += c->g;
      }
      for (int i = 0; i < total - head; ++i) {
        memcpy(c->Kr + (bh * c->Rcap + i) * D, ks + (size_t)(head + i) * D,
               2 * (size_t)D);
        memcpy(c->Vr + (bh * c->Rcap + i) * D, vs + (size_t)(head + i) * D,
               2 * (size_t)D);
      }
      if (h == c->Hkv - 1) {
        c->Tq[b] = Tq;
        c->nres[b] = total - head;
        c->S[b] += n;
      }
      free(ks);
      free(vs);
    }
    age_update(c, b);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization and attention (double).                                   */
/* ------------------------------------------------------------------------ */

/* k_hat and v_hat of token t of sequence (b, h), all D channels, in double. */
static void token_hat(const orc_cache *c, int b, int h, int t, double *k,
                      double *v) {
  const int D = c->D, g = c->g;
  size_t bh = (size_t)b * c->Hkv + h;
  if (t < c->Tq[b] && c->n_sink > 0 && is_sink(c, b, h, t)) {
    /* a sink token of the quantized region: its exact fp16 rows */
    const int32_t *sp = c->sink_pos + bh * c->n_sink;
    int slot = 0;
    while (sp[slot] != t) ++slot;
    for (int ch = 0; ch < D; ++ch) {
      k[ch] = h2f(c->sink_k[(bh * c->n_sink + slot) * D + ch]);
      v[ch] = h2f(c->sink_v[(bh * c->n_sink + slot) * D + ch]);
    }
    return;
  }
  if (t < c->Tq[b] && c->Kmask) {
    const int G = t / g;
    const uint32_t *mask = c->Kmask + (bh * (c->Tcap / g) + G) * (D / 32);
    const uint8_t *row = c->Kc + (bh * c->Tcap + t) * c->krow;
    int bit = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int ch = 0; ch < D; ++ch) {
        const int hi = (mask[ch / 32] >> (ch % 32)) & 1;
        if (hi != (pass == 0)) continue;
        const int w = hi ? 4 : 2;
        const int code = (row[bit / 8] >> (bit % 8)) & ((1 << w) - 1);
        bit += w;
        double sc = h2f(c->Ks[(bh * (c->Tcap / g) + G) * D + ch]);
        double z = h2f(c->Kz[(bh * (c->Tcap / g) + G) * D + ch]);
        k[ch] = (double)code * sc + z;
      }
    for (int ch = 0; ch < D; ++ch) v[ch] = h2f(c->Vf[(bh * c->Tcap + t) * D + ch]);
    return;
  }
  if (t < c->Tq[b]) {
    uint8_t codes[4096];
    int G = t / g;
    const int w = c->tier ? c->age_bits[c->tier[bh * (c->Tcap / g) + G]] : c->bits;
    orc_unpack_codes(c->Kc + (bh * c->Tcap + t) * c->row, D, w, codes);
    for (int ch = 0; ch < D; ++ch) {
      double s = h2f(c->Ks[(bh * (c->Tcap / g) + G) * D + ch]);
      double z = h2f(c->Kz[(bh * (c->Tcap / g) + G) * D + ch]);
      k[ch] = (double)codes[ch] * s + z;
    }
    orc_unpack_codes(c->Vc + (bh * c->Tcap + t) * c->row, D, w, codes);
    for (int ch = 0; ch < D; ++ch) {
      double s = h2f(c->Vs[(bh * c->Tcap + t) * (D / g) + ch / g]);
      double z = h2f(c->Vz[(bh * c->Tcap + t) * (D / g) + ch / g]);
      v[ch] = (double)codes[ch] * s + z;
    }
  } else {
    int i = t - c->Tq[b];
    for (int ch = 0; ch < D; ++ch) {
      k[ch] = h2f(c->Kr[(bh * c->Rcap + i) * D + ch]);
      v[ch] = h2f(c->Vr[(bh * c->Rcap + i) * D + ch]);
    }
  }
}

/* One query head: softmax(scale * q . k_hat_t) over every token t of
 * sequence b (quantized prefix and fp16 residual; no mask), weighted sum of
 * v_hat_t.  Query head hq reads kv head hq / (Hq/Hkv).  out: D doubles.
 * Returns 0, or -1 for an empty sequence (out is then all zero). */
int orc_attend_one(const orc_cache *c, int b, int hq, const uint16_t *q_row,
                   double scale, double *out) {
  const int D = c->D;
  const int h = hq / (c->Hq / c->Hkv);
  const int S = c->S[b];
  for (int ch = 0; ch < D; ++ch) out[ch] = 0.0;
  if (S == 0) return -1;
  double *q = (double *)malloc(sizeof(double) * D);
  double *k = (double *)malloc(sizeof(double) * D);
  double *v = (double *)malloc(sizeof(double) * D);
  double *s = (double *)malloc(sizeof(double) * (size_t)S);
  for (int ch = 0; ch < D; ++ch) q[ch] = h2f(q_row[ch]);
  double m = -INFINITY;
  for (int t = 0; t < S; ++t) {
    token_hat(c, b, h, t, k, v);
    double dot = 0.0;
    for (int ch = 0; ch < D; ++ch) dot += q[ch] * k[ch];
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int t = 0; t < S; ++t) {
    double p = exp(s[t] - m);
    l += p;
    token_hat(c, b, h, t, k, v);
    for (int ch = 0; ch < D; ++ch) out[ch] += p * v[ch];
  }
  for (int ch = 0; ch < D; ++ch) out[ch] /= l;
  free(q); free(k); free(v); free(s);
  return 0;
}

/* Several query tokens per sequence (multi-query decode, chunked
 * prefill-attend): the S_q queries of sequence b are its newest S_q tokens,
 * already in the cache, so query i sits at position S[b] - S_q + i and
 * attends every token t <= that position (causal; the S_q = 1 case is
 * orc_attend_one).  q fp16 [B][Hq][S_q][D] -> out fp32 [B][Hq][S_q][D], the
 * softmax in double as in orc_attend_one.  Returns 0, or -1 when some
 * sequence holds fewer than S_q tokens (out untouched). */
/* One query of head hq of sequence b attending tokens 0 ... last (the
 * causal prefix of the query at position last); out: D doubles.  Returns
 * 0, or -1 when last is outside [0, S - 1]. */
int orc_attend_prefix(const orc_cache *c, int b, int hq, const uint16_t *q_row,
                      int last, double scale, double *out) {
  const int D = c->D;
  const int h = hq / (c->Hq / c->Hkv);
  if (last < 0 || last >= c->S[b]) return -1;
  double *qd = (double *)malloc(sizeof(double) * D);
  double *k = (double *)malloc(sizeof(double) * D);
  double *v = (double *)malloc(sizeof(double) * D);
  double *s = (double *)malloc(sizeof(double) * (size_t)(last + 1));
  for (int ch = 0; ch < D; ++ch) qd[ch] = h2f(q_row[ch]);
  double m = -INFINITY;
  for (int t = 0; t <= last; ++t) {
    token_hat(c, b, h, t, k, v);
    double dot = 0.0;
    for (int ch = 0; ch < D; ++ch) dot += qd[ch] * k[ch];
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int ch = 0; ch < D; ++ch) out[ch] = 0.0;
  for (int t = 0; t <= last; ++t) {
    double p = exp(s[t] - m);
    l += p;
    token_hat(c, b, h, t, k, v);
    for (int ch = 0; ch < D; ++ch) out[ch] += p * v[ch];
  }
  for (int ch = 0; ch < D; ++ch) out[ch] /= l;
  free(qd); free(k); free(v); free(s);
  return 0;
}

int orc_attend_multi(const orc_cache *c, const uint16_t *q, int S_q,
                     double scale, float *out) {
  const int D = c->D;
  if (S_q <= 0) return -1;
  for (int b = 0; b < c->B; ++b)
    if (c->S[b] < S_q) return -1;
  double *o = (double *)malloc(sizeof(double) * D);
  for (int b = 0; b < c->B; ++b)
    for (int hq = 0; hq < c->Hq; ++hq)
      for (int i = 0; i < S_q; ++i) {
        const size_t row = (((size_t)b * c->Hq + hq) * S_q + i) * D;
        /* query i sits at position S - S_q + i and sees tokens up to it */
        orc_attend_prefix(c, b, hq, q + row, c->S[b] - S_q + i, scale, o);
        for (int ch = 0; ch < D; ++ch) out[row + ch] = (float)o[ch];
      }
  free(o);
  return 0;
}

/* All heads: q fp16 [B][Hq][D] -> out fp32 [B][Hq][D]. */
int orc_attend(const orc_cache *c, const uint16_t *q, double scale,
               float *out) {
  double *o = (double *)malloc(sizeof(double) * c->D);
  for (int b = 0; b < c->B; ++b)
    for (int hq = 0; hq < c->Hq; ++hq) {
      size_t off = ((size_t)b * c->Hq + hq) * c->D;
      orc_attend_one(c, b, hq, q + off, scale, o);
      for (int ch = 0; ch < c->D; ++ch) out[off + ch] = (float)o[ch];
    }
  free(o);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Accessors.                                                                 */
/* ------------------------------------------------------------------------ */

void orc_lengths(const orc_cache *c, int32_t *S, int32_t *Tq, int32_t *nres) {
  memcpy(S, c->S, 4 * (size_t)c->B);
  memcpy(Tq, c->Tq, 4 * (size_t)c->B);
  memcpy(nres, c->nres, 4 * (size_t)c->B);
}

void orc_dims(const orc_cache *c, int32_t *Tcap, int32_t *Rcap) {
  *Tcap = c->Tcap;
  *Rcap = c->Rcap;
}

/* which: 0 Kc, 1 Ks, 2 Kz, 3 Vc, 4 Vs, 5 Vz, 6 Kr, 7 Vr.  Copies the whole
 * plane into dst (size given by orc_plane_bytes). */
size_t orc_plane_bytes(const orc_cache *c, int which) {
  size_t bh = (size_t)c->B * c->Hkv;
  switch (which) {
    case 0: return bh * c->Tcap * (c->Kmask ? c->krow : c->row);
    case 3: return bh * c->Tcap * c->row;
    case 1: case 2: return bh * (c->Tcap / c->g) * c->D * 2;
    case 4: case 5: return bh * c->Tcap * (c->D / c->g) * 2;
    case 6: case 7: return bh * c->Rcap * c->D * 2;
    case 8: return bh * c->n_sink * 4;
    case 9: case 10: return bh * c->n_sink * c->D * 2;
    case 11: return c->Kmask ? bh * (c->Tcap / c->g) * (c->D / 32) * 4 : 0;
    case 13: return c->tier ? bh * (c->Tcap / c->g) : 0;
    case 12: return c->Vf ? bh * c->Tcap * c->D * 2 : 0;
    default: return 0;
  }
}

int orc_get_plane(const orc_cache *c, int which, void *dst) {
  const void *src = NULL;
  switch (which) {
    case 0: src = c->Kc; break;
    case 1: src = c->Ks; break;
    case 2: src = c->Kz; break;
    case 3: src = c->Vc; break;
    case 4: src = c->Vs; break;
    case 5: src = c->Vz; break;
    case 6: src = c->Kr; break;
    case 7: src = c->Vr; break;
    case 8: src = c->sink_pos; break;
    case 9: src = c->sink_k; break;
    case 10: src = c->sink_v; break;
    case 11: src = c->Kmask; break;
    case 12: src = c->Vf; break;
    case 13: src = c->tier; break;
    default: return -1;
  }
  if (!src) return orc_plane_bytes(c, which) == 0 ? 0 : -1;
  memcpy(dst, src, orc_plane_bytes(c, which));
  return 0;
}
