/*
 * oracle.c - plain, slow CPU oracle of the quantized small-batch matvec and
 * MoE decode path.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by
 * __graft_entry__.smoke() and by the CPU-baseline leg of bench.py, never by
 * the library.  It shares no code with the CUDA path.
 *
 * What it computes (plain definitions; no blocking, fusion or reordering):
 *   - the activation quantizer (per-32 int8 with an fp32 scale), in fp32 as
 *     the rule fixes it, so that integer codes are decided in the same
 *     precision as on the GPU;
 *   - the weight quantizers and dequantizers of Q8_0, Q4_K, IQ4_XS, Q5_K, Q6_K
 *     and Q8 with one scale per 64 or 128 weights, in
 *     fp64, following the byte layouts written out in include/qmv.h, and the
 *     conversions of the unquantized F16 / F32 rows;
 *   - the matvec y[t][m] = sum_k What[m][k] * Xhat[t][k] in fp64, plus the
 *     tolerance scale sum_k |What[m][k] * Xhat[t][k]| (Xhat = x, unquantized,
 *     for F16 / F32 weights);
 *   - the MoE decode layer (routing, gate/up, SwiGLU, requantization of h,
 *     down projection, gate-weighted combine in k order) in fp64 except the
 *     requantization, which uses the fp32 activation rule;
 *   - the router's top-k selection and gate normalization (softmax or
 *     sigmoid) on given logits, in fp64.
 * Sources: small-batch matvecs over Q8_0 / K-quant / IQ4_XS weights and the
 * MoE decode kernels: "Castagna Veloce", section "Kernels for the MI50";
 * gate/up + SwiGLU and Q8 activations shared across weight types: same page,
 * section "Fused operations".  The pages fix no formula or layout; the block
 * definitions are the library's, restated here from their text.
 *
 * Parity pins: every function here is checked in tests/test_oracle.py against
 * brute force, closed forms, library routines or invariants (see that file).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no FMA contraction, so the
 * fp32 and fp64 results are the same on x86-64 and aarch64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_Q8_0 0
#define OR_Q4_K 1
#define OR_IQ4_XS 2
#define OR_Q5_K 3
#define OR_Q6_K 4
#define OR_Q8_G64 5
#define OR_Q8_G128 6
#define OR_F16 7
#define OR_F32 8

/* Unquantized weight rows: activations are used as they are. */
static int is_float_fmt(int fmt) { return fmt == OR_F16 || fmt == OR_F32; }

static const int8_t OR_CB[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                 1,    13,   25,  38,  53,  69,  89,  113};

/* ------------------------------------------------------------------------ */
/* binary16 <-> double                                                       */
/* ------------------------------------------------------------------------ */

double oracle_f16_to_f64(uint16_t h) {
  int sgn = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25);
  return sgn ? -v : v;
}

/* Round to the nearest binary16, ties to even; overflow gives infinity. */
uint16_t oracle_f64_to_f16(double v) {
  uint16_t sgn = signbit(v) ? 0x8000 : 0;
  if (isnan(v)) return 0x7E00;
  double a = fabs(v);
  if (a == 0.0) return sgn;
  if (isinf(a)) return sgn | 0x7C00;
  int e2;
  frexp(a, &e2);      /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;     /* a in [2^E, 2^(E+1)) */
  if (E < -14) E = -14; /* subnormal binade: spacing 2^-24 */
  double spacing = ldexp(1.0, E - 10);
  double r = nearbyint(a / spacing); /* exact quotient; rounding mode RNE */
  double rv = r * spacing;
  if (rv == 0.0) return sgn;
  if (rv >= 65536.0) return sgn | 0x7C00;
  frexp(rv, &e2);
  int RE = e2 - 1;
  if (RE < -14) return sgn | (uint16_t)(rv / ldexp(1.0, -24));
  uint16_t mant = (uint16_t)(rv / ldexp(1.0, RE - 10) - 1024.0);
  return sgn | (uint16_t)((RE + 15) << 10) | mant;
}

/* ------------------------------------------------------------------------ */
/* layout helpers                                                            */
/* ------------------------------------------------------------------------ */

int64_t oracle_group_weights(int fmt) {
  switch (fmt) {
    case OR_Q8_0: return 256;
    case OR_Q4_K: return 256;
    case OR_IQ4_XS: return 512;
    case OR_Q5_K: return 256;
    case OR_Q6_K: return 256;
    case OR_Q8_G64: return 512;
    case OR_Q8_G128: return 1024;
    case OR_F16: return 32;
    case OR_F32: return 32;
  }
  return -1;
}

int64_t oracle_group_bytes(int fmt) {
  switch (fmt) {
    case OR_Q8_0: return 272;
    case OR_Q4_K: return 144;
    case OR_IQ4_XS: return 272;
    case OR_Q5_K: return 176;
    case OR_Q6_K: return 208;
    case OR_Q8_G64: return 528;
    case OR_Q8_G128: return 1040;
    case OR_F16: return 64;
    case OR_F32: return 128;
  }
  return -1;
}

int64_t oracle_row_bytes(int fmt, int64_t K) {
  int64_t gw = oracle_group_weights(fmt);
  if (gw <= 0 || K <= 0 || K % gw) return -1;
  return (K / gw) * oracle_group_bytes(fmt);
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFF);
  p[1] = (uint8_t)(v >> 8);
}

/* nbits-wide field starting at bit `bit` of a little-endian bit string. */
static unsigned get_bits(const uint8_t* s, int bit, int nbits) {
  unsigned v = 0;
  for (int i = 0; i < nbits; i++) {
    int b = bit + i;
    v |= (unsigned)((s[b >> 3] >> (b & 7)) & 1) << i;
  }
  return v;
}
static void put_bits(uint8_t* s, int bit, int nbits, unsigned v) {
  for (int i = 0; i < nbits; i++) {
    int b = bit + i;
    if ((v >> i) & 1)
      s[b >> 3] |= (uint8_t)(1 << (b & 7));
    else
      s[b >> 3] &= (uint8_t)~(1 << (b & 7));
  }
}

/* 4-bit code of weight i (0..31) of a 32-weight sub-block whose 16 payload
 * bytes start at p: byte i%16, low nibble for i < 16, high nibble otherwise. */
static unsigned get_nib(const uint8_t* p, int i) {
  return i < 16 ? (p[i] & 0xF) : (p[i - 16] >> 4);
}
static void put_nib(uint8_t* p, int i, unsigned c) {
  if (i < 16)
    p[i] = (uint8_t)((p[i] & 0xF0) | (c & 0xF));
  else
    p[i - 16] = (uint8_t)((p[i - 16] & 0x0F) | ((c & 0xF) << 4));
}

/* Payload byte of weight i (0..31) of Q8_0 block b (0..7) within a group:
 * the first 16 weights of the 8 blocks come first, then the last 16. */
static int q8_0_offset(int b, int i) { return i < 16 ? 16 * b + i : 128 + 16 * b + (i - 16); }

/* ------------------------------------------------------------------------ */
/* activation quantizer (fp32 rule)                                          */
/* ------------------------------------------------------------------------ */

void oracle_act_quant(const float* x, int64_t K, int64_t n, int8_t* q, float* d,
                      int32_t* s) {
  int64_t nb = K / 32;
  for (int64_t t = 0; t < n; t++) {
    for (int64_t j = 0; j < nb; j++) {
      const float* xb = x + t * K + j * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; i++) {
        float a = fabsf(xb[i]);
        if (a > amax) amax = a;
      }
      float dd = amax / 127.0f;
      float id = dd > 0.0f ? 1.0f / dd : 0.0f;
      int32_t sum = 0;
      for (int i = 0; i < 32; i++) {
        float p = xb[i] * id;
        float r = rintf(p); /* default rounding mode: half to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        /* a block whose largest magnitude is below about 3.7e-37 has a
         * subnormal d whose reciprocal overflows to infinity; its zero
         * elements then give 0 * inf, not a number: their code is 0 */
        if (p != p) r = 0.0f;
        q[t * K + j * 32 + i] = (int8_t)r;
        sum += (int32_t)r;
      }
      d[t * nb + j] = dd;
      s[t * nb + j] = sum;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* weight quantizers (fp64)                                                  */
/* ------------------------------------------------------------------------ */

static void quant_q8_0_group(const float* w, uint8_t* g) {
  memset(g, 0, 272);
  for (int b = 0; b < 8; b++) {
    const float* wb = w + b * 32;
    double amax = 0.0;
    for (int i = 0; i < 32; i++) {
      double a = fabs((double)wb[i]);
      if (a > amax) amax = a;
    }
    uint16_t d16 = oracle_f64_to_f16(amax / 127.0);
    double dv = oracle_f16_to_f64(d16);
    wr16(g + 2 * b, d16);
    for (int i = 0; i < 32; i++) {
      double r = 0.0;
      if (dv > 0.0) {
        r = nearbyint((double)wb[i] / dv);
        if (r > 127.0) r = 127.0;
        if (r < -127.0) r = -127.0;
      }
      g[16 + q8_0_offset(b, i)] = (uint8_t)(int8_t)r;
    }
  }
}

static void quant_q4_k_group(const float* w, uint8_t* g) {
  memset(g, 0, 144);
  double a[8], bmin[8];
  for (int j = 0; j < 8; j++) {
    double lo = 0.0, hi = -INFINITY;
    for (int i = 0; i < 32; i++) {
      double v = (double)w[32 * j + i];
      if (v < lo) lo = v;
      if (v > hi) hi = v;
    }
    a[j] = (hi - lo) / 15.0;
    bmin[j] = -lo;
  }
  double amax = 0.0, bmax = 0.0;
  for (int j = 0; j < 8; j++) {
    if (a[j] > amax) amax = a[j];
    if (bmin[j] > bmax) bmax = bmin[j];
  }
  uint16_t d16 = oracle_f64_to_f16(amax / 63.0);
  uint16_t dm16 = oracle_f64_to_f16(bmax / 63.0);
  double dv = oracle_f16_to_f64(d16), dmv = oracle_f16_to_f64(dm16);
  wr16(g, d16);
  wr16(g + 2, dm16);
  for (int j = 0; j < 8; j++) {
    double sc = 0.0, m = 0.0;
    if (dv > 0.0) {
      sc = nearbyint(a[j] / dv);
      if (sc > 63.0) sc = 63.0;
      if (sc < 0.0) sc = 0.0;
    }
    if (dmv > 0.0) {
      m = nearbyint(bmin[j] / dmv);
      if (m > 63.0) m = 63.0;
      if (m < 0.0) m = 0.0;
    }
    put_bits(g + 4, 12 * j, 6, (unsigned)sc);
    put_bits(g + 4, 12 * j + 6, 6, (unsigned)m);
    double S = dv * sc, O = dmv * m;
    for (int i = 0; i < 32; i++) {
      double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(v - (S * 0.0 - O));
      for (int q = 1; q < 16; q++) {
        double e = fabs(v - (S * (double)q - O));
        if (e < berr) {
          berr = e;
          best = q;
        }
      }
      put_nib(g + 16 + 16 * j, i, (unsigned)best);
    }
  }
}

/* Q5_K group (256 weights, 176 bytes): bytes 0-1 d, 2-3 dmin (fp16), 4-15
 * the 6-bit sc / m fields as in Q4_K, 16-47 the fifth bit of every weight
 * (4 bytes per 32-weight sub-block j, little-endian: bit i is weight i's),
 * 48-175 the low four bits (16 bytes per sub-block, byte i: weight i in the
 * low nibble, weight i + 16 in the high nibble).  w = d sc_j q - dmin m_j,
 * q in [0, 31].  The fit is Q4_K's with 31 steps. */
static void quant_q5_k_group(const float* w, uint8_t* g) {
  memset(g, 0, 176);
  double a[8], bmin[8];
  for (int j = 0; j < 8; j++) {
    double lo = 0.0, hi = -INFINITY;
    for (int i = 0; i < 32; i++) {
      double v = (double)w[32 * j + i];
      if (v < lo) lo = v;
      if (v > hi) hi = v;
    }
    a[j] = (hi - lo) / 31.0;
    bmin[j] = -lo;
  }
  double amax = 0.0, bmax = 0.0;
  for (int j = 0; j < 8; j++) {
    if (a[j] > amax) amax = a[j];
    if (bmin[j] > bmax) bmax = bmin[j];
  }
  uint16_t d16 = oracle_f64_to_f16(amax / 63.0);
  uint16_t dm16 = oracle_f64_to_f16(bmax / 63.0);
  double dv = oracle_f16_to_f64(d16), dmv = oracle_f16_to_f64(dm16);
  wr16(g, d16);
  wr16(g + 2, dm16);
  for (int j = 0; j < 8; j++) {
    double sc = 0.0, m = 0.0;
    if (dv > 0.0) {
      sc = nearbyint(a[j] / dv);
      if (sc > 63.0) sc = 63.0;
      if (sc < 0.0) sc = 0.0;
    }
    if (dmv > 0.0) {
      m = nearbyint(bmin[j] / dmv);
      if (m > 63.0) m = 63.0;
      if (m < 0.0) m = 0.0;
    }
    put_bits(g + 4, 12 * j, 6, (unsigned)sc);
    put_bits(g + 4, 12 * j + 6, 6, (unsigned)m);
    double S = dv * sc, O = dmv * m;
    for (int i = 0; i < 32; i++) {
      double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(v - (S * 0.0 - O));
      for (int q = 1; q < 32; q++) {
        double e = fabs(v - (S * (double)q - O));
        if (e < berr) {
          berr = e;
          best = q;
        }
      }
      put_nib(g + 48 + 16 * j, i, (unsigned)best & 15u);
      put_bits(g + 16 + 4 * j, i, 1, (unsigned)best >> 4);
    }
  }
}

/* Q6_K group (256 weights = 16 sub-blocks of 16, 208 bytes): bytes 0-1 d
 * (fp16), bytes 2-15 a 112-bit string of 7-bit sub-scales (bits [7i, 7i+7)
 * = sc_i), bytes 16-79 the top two bits and bytes 80-207 the low four bits
 * of each 6-bit code v = (q - 32) mod 64, q in [0, 63].  w = d sc_i (q - 32).
 * Per 32-weight block j (sub-blocks 2j and 2j+1): two 32-bit words at
 * 16 + 8j (weights 0..15, then 16..31 of the block), weight e of a word
 * (k = e / 4, b = e % 4) at bits [8b + 2k, 8b + 2k + 2); 16 nibble bytes at
 * 80 + 16j as in Q4_K (byte i: weight i low, weight i + 16 high).  The fit:
 * s_i = amax_i / 31, d = max s_i / 127 (fp16), sc_i = clamp(rne(s_i / d16),
 * 0, 127), q = argmin over 0..63 of |w - d16 sc_i (q - 32)|, ties to the
 * lower q. */
static void q6_k_put(uint8_t* g, int j, int i, unsigned v) {
  put_nib(g + 80 + 16 * j, i, v & 15u);
  const int e = i & 15, word = i >> 4;
  put_bits(g + 16 + 8 * j + 4 * word, 8 * (e & 3) + 2 * (e >> 2), 2, v >> 4);
}
static unsigned q6_k_get(const uint8_t* g, int j, int i) {
  const int e = i & 15, word = i >> 4;
  return get_nib(g + 80 + 16 * j, i) | (get_bits(g + 16 + 8 * j + 4 * word, 8 * (e & 3) + 2 * (e >> 2), 2) << 4);
}
static void quant_q6_k_group(const float* w, uint8_t* g) {
  memset(g, 0, 208);
  double s[16], smax = 0.0;
  for (int i = 0; i < 16; i++) {
    double amax = 0.0;
    for (int k = 0; k < 16; k++) {
      double v = fabs((double)w[16 * i + k]);
      if (v > amax) amax = v;
    }
    s[i] = amax / 31.0;
    if (s[i] > smax) smax = s[i];
  }
  uint16_t d16 = oracle_f64_to_f16(smax / 127.0);
  double dv = oracle_f16_to_f64(d16);
  wr16(g, d16);
  for (int i = 0; i < 16; i++) {
    double sc = 0.0;
    if (dv > 0.0) {
      sc = nearbyint(s[i] / dv);
      if (sc > 127.0) sc = 127.0;
      if (sc < 0.0) sc = 0.0;
    }
    put_bits(g + 2, 7 * i, 7, (unsigned)sc);
    double S = dv * sc;
    for (int k = 0; k < 16; k++) {
      double v = (double)w[16 * i + k];
      int best = 0;
      double berr = fabs(v - S * -32.0);
      for (int q = 1; q < 64; q++) {
        double e = fabs(v - S * (double)(q - 32));
        if (e < berr) {
          berr = e;
          best = q;
        }
      }
      const int el = 16 * i + k;  /* weight index in the group */
      q6_k_put(g, el >> 5, el & 31, (unsigned)(best - 32) & 63u);
    }
  }
}

/* Q8 with one scale per gs weights (gs = 64 or 128), groups of n256 x 256
 * weights (2 for gs = 64, 4 for gs = 128): bytes [2s, 2s+2) the fp16 d of
 * scale group s (8 per group), then n256 payloads of 256 bytes arranged as
 * Q8_0's.  d = amax / 127 over the gs weights (fp16), q = rne(w / d16)
 * clamped to +-127 (the Q8_0 rule over a larger block). */
static void quant_q8_g_group(const float* w, uint8_t* g, int gs, int n256) {
  memset(g, 0, 16 + 256 * (size_t)n256);
  for (int sidx = 0; sidx < 8; sidx++) {
    double amax = 0.0;
    for (int i = 0; i < gs; i++) {
      double a = fabs((double)w[gs * sidx + i]);
      if (a > amax) amax = a;
    }
    uint16_t d16 = oracle_f64_to_f16(amax / 127.0);
    double dv = oracle_f16_to_f64(d16);
    wr16(g + 2 * sidx, d16);
    for (int i = 0; i < gs; i++) {
      const int el = gs * sidx + i, half = el >> 8, b = (el >> 5) & 7, ii = el & 31;
      double r = 0.0;
      if (dv > 0.0) {
        r = nearbyint((double)w[el] / dv);
        if (r > 127.0) r = 127.0;
        if (r < -127.0) r = -127.0;
      }
      g[16 + 256 * half + q8_0_offset(b, ii)] = (uint8_t)(int8_t)r;
    }
  }
}

static void quant_iq4_xs_superblock(const float* w, uint8_t* meta, uint8_t* payload) {
  double s[8];
  double smax = 0.0;
  for (int j = 0; j < 8; j++) {
    double amax = 0.0;
    for (int i = 0; i < 32; i++) {
      double v = fabs((double)w[32 * j + i]);
      if (v > amax) amax = v;
    }
    s[j] = amax / 113.0;
    if (s[j] > smax) smax = s[j];
  }
  uint16_t d16 = oracle_f64_to_f16(smax / 31.0);
  double dv = oracle_f16_to_f64(d16);
  wr16(meta, d16);
  for (int j = 0; j < 8; j++) {
    double l = 0.0;
    if (dv > 0.0) {
      l = nearbyint(s[j] / dv);
      if (l > 31.0) l = 31.0;
      if (l < 0.0) l = 0.0;
    }
    int ls = 32 + (int)l;
    put_bits(meta + 2, 6 * j, 6, (unsigned)ls);
    double e = dv * (double)(ls - 32);
    for (int i = 0; i < 32; i++) {
      double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(v - e * (double)OR_CB[0]);
      for (int c = 1; c < 16; c++) {
        double err = fabs(v - e * (double)OR_CB[c]);
        if (err < berr) {
          berr = err;
          best = c;
        }
      }
      put_nib(payload + 16 * j, i, (unsigned)best);
    }
  }
}

static void quant_iq4_xs_group(const float* w, uint8_t* g) {
  memset(g, 0, 272);
  for (int sb = 0; sb < 2; sb++)
    quant_iq4_xs_superblock(w + 256 * sb, g + 8 * sb, g + 16 + 128 * sb);
}

int oracle_quantize(int fmt, const float* w, int64_t M, int64_t K, uint8_t* out) {
  int64_t rb = oracle_row_bytes(fmt, K);
  if (rb < 0 || M <= 0) return -1;
  int64_t gw = oracle_group_weights(fmt), gb = oracle_group_bytes(fmt);
  for (int64_t m = 0; m < M; m++) {
    for (int64_t gi = 0; gi < K / gw; gi++) {
      const float* wg = w + m * K + gi * gw;
      uint8_t* g = out + m * rb + gi * gb;
      if (fmt == OR_Q8_0)
        quant_q8_0_group(wg, g);
      else if (fmt == OR_Q4_K)
        quant_q4_k_group(wg, g);
      else if (fmt == OR_Q5_K)
        quant_q5_k_group(wg, g);
      else if (fmt == OR_Q6_K)
        quant_q6_k_group(wg, g);
      else if (fmt == OR_Q8_G64)
        quant_q8_g_group(wg, g, 64, 2);
      else if (fmt == OR_Q8_G128)
        quant_q8_g_group(wg, g, 128, 4);
      else if (fmt == OR_F16)
        for (int i = 0; i < 32; i++) wr16(g + 2 * i, oracle_f64_to_f16((double)wg[i]));
      else if (fmt == OR_F32)
        for (int i = 0; i < 32; i++) {
          uint32_t b;
          memcpy(&b, &wg[i], 4);
          for (int k = 0; k < 4; k++) g[4 * i + k] = (uint8_t)(b >> (8 * k));
        }
      else
        quant_iq4_xs_group(wg, g);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* dequantizers (fp64)                                                       */
/* ------------------------------------------------------------------------ */

/* Dequantize one row (K weights) into out[0..K). */
static void dequant_row(int fmt, const uint8_t* row, int64_t K, double* out) {
  int64_t gw = oracle_group_weights(fmt), gb = oracle_group_bytes(fmt);
  for (int64_t gi = 0; gi < K / gw; gi++) {
    const uint8_t* g = row + gi * gb;
    double* o = out + gi * gw;
    if (fmt == OR_Q8_0) {
      for (int b = 0; b < 8; b++) {
        double d = oracle_f16_to_f64(rd16(g + 2 * b));
        for (int i = 0; i < 32; i++) o[32 * b + i] = d * (double)(int8_t)g[16 + q8_0_offset(b, i)];
      }
    } else if (fmt == OR_Q4_K) {
      double d = oracle_f16_to_f64(rd16(g)), dmin = oracle_f16_to_f64(rd16(g + 2));
      for (int j = 0; j < 8; j++) {
        unsigned sc = get_bits(g + 4, 12 * j, 6), m = get_bits(g + 4, 12 * j + 6, 6);
        for (int i = 0; i < 32; i++) {
          unsigned q = get_nib(g + 16 + 16 * j, i);
          o[32 * j + i] = d * (double)sc * (double)q - dmin * (double)m;
        }
      }
    } else if (fmt == OR_Q5_K) {
      double d = oracle_f16_to_f64(rd16(g)), dmin = oracle_f16_to_f64(rd16(g + 2));
      for (int j = 0; j < 8; j++) {
        unsigned sc = get_bits(g + 4, 12 * j, 6), m = get_bits(g + 4, 12 * j + 6, 6);
        for (int i = 0; i < 32; i++) {
          unsigned q = get_nib(g + 48 + 16 * j, i) | (get_bits(g + 16 + 4 * j, i, 1) << 4);
          o[32 * j + i] = d * (double)sc * (double)q - dmin * (double)m;
        }
      }
    } else if (fmt == OR_F16) {
      for (int i = 0; i < 32; i++) o[i] = oracle_f16_to_f64(rd16(g + 2 * i));
    } else if (fmt == OR_F32) {
      for (int i = 0; i < 32; i++) {
        uint32_t b = (uint32_t)g[4 * i] | ((uint32_t)g[4 * i + 1] << 8) | ((uint32_t)g[4 * i + 2] << 16) |
                     ((uint32_t)g[4 * i + 3] << 24);
        float f;
        memcpy(&f, &b, 4);
        o[i] = (double)f;
      }
    } else if (fmt == OR_Q8_G64 || fmt == OR_Q8_G128) {
      const int gs = fmt == OR_Q8_G64 ? 64 : 128;
      for (int el = 0; el < (int)gw; el++) {
        double d = oracle_f16_to_f64(rd16(g + 2 * (el / gs)));
        o[el] = d * (double)(int8_t)g[16 + 256 * (el >> 8) + q8_0_offset((el >> 5) & 7, el & 31)];
      }
    } else if (fmt == OR_Q6_K) {
      double d = oracle_f16_to_f64(rd16(g));
      for (int el = 0; el < 256; el++) {
        unsigned sc = get_bits(g + 2, 7 * (el >> 4), 7);
        unsigned v = q6_k_get(g, el >> 5, el & 31);
        int q32 = (int)v - ((v & 32u) ? 64 : 0);  /* q - 32 */
        o[el] = d * (double)sc * (double)q32;
      }
    } else {
      for (int sb = 0; sb < 2; sb++) {
        const uint8_t* meta = g + 8 * sb;
        double d = oracle_f16_to_f64(rd16(meta));
        for (int j = 0; j < 8; j++) {
          int ls = (int)get_bits(meta + 2, 6 * j, 6);
          for (int i = 0; i < 32; i++) {
            unsigned c = get_nib(g + 16 + 128 * sb + 16 * j, i);
            o[256 * sb + 32 * j + i] = d * (double)(ls - 32) * (double)OR_CB[c];
          }
        }
      }
    }
  }
}

int oracle_dequant(int fmt, const uint8_t* W, int64_t M, int64_t K, double* out) {
  int64_t rb = oracle_row_bytes(fmt, K);
  if (rb < 0 || M <= 0) return -1;
  for (int64_t m = 0; m < M; m++) dequant_row(fmt, W + m * rb, K, out + m * K);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* matvec (fp64)                                                             */
/* ------------------------------------------------------------------------ */

typedef struct {
  int fmt;
  const uint8_t* W;
  int64_t M, K, n, rb;
  const double* xhat; /* [n][K] */
  double* y;          /* [n][M] */
  double* sabs;       /* [n][M] or NULL */
  int64_t m0, m1;
} qmv_job;

static void* qmv_worker(void* arg) {
  qmv_job* j = (qmv_job*)arg;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)j->K);
  if (!wrow) return NULL;
  for (int64_t m = j->m0; m < j->m1; m++) {
    dequant_row(j->fmt, j->W + m * j->rb, j->K, wrow);
    for (int64_t t = 0; t < j->n; t++) {
      const double* xr = j->xhat + t * j->K;
      double acc = 0.0, aabs = 0.0;
      for (int64_t k = 0; k < j->K; k++) {
        double p = wrow[k] * xr[k];
        acc += p;
        aabs += fabs(p);
      }
      j->y[t * j->M + m] = acc;
      if (j->sabs) j->sabs[t * j->M + m] = aabs;
    }
  }
  free(wrow);
  return NULL;
}

/* y[t][m] = sum_k What[m][k] * Xhat[t][k]; sabs[t][m] = sum_k |What Xhat|.
 * x is fp32 [n][K], quantized here with oracle_act_quant (F16 / F32 weights:
 * Xhat = x).  Rows are split across nthreads POSIX threads (1 = serial). */
int oracle_qmv(int fmt, const uint8_t* W, int64_t M, int64_t K, const float* x,
               int64_t n, double* y, double* sabs, int nthreads) {
  int64_t rb = oracle_row_bytes(fmt, K);
  if (rb < 0 || M <= 0 || n <= 0) return -1;
  int8_t* q = (int8_t*)malloc((size_t)(n * K));
  float* d = (float*)malloc(sizeof(float) * (size_t)(n * K / 32));
  int32_t* s = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n * K / 32));
  double* xhat = (double*)malloc(sizeof(double) * (size_t)(n * K));
  if (!q || !d || !s || !xhat) return -2;
  oracle_act_quant(x, K, n, q, d, s);
  for (int64_t t = 0; t < n; t++)
    for (int64_t k = 0; k < K; k++)
      xhat[t * K + k] = is_float_fmt(fmt) ? (double)x[t * K + k]
                                          : (double)d[t * (K / 32) + k / 32] * (double)q[t * K + k];
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  qmv_job jobs[256];
  pthread_t th[256];
  for (int i = 0; i < nthreads; i++) {
    jobs[i] = (qmv_job){fmt, W, M, K, n, rb, xhat, y, sabs, M * i / nthreads, M * (i + 1) / nthreads};
  }
  if (nthreads == 1) {
    qmv_worker(&jobs[0]);
  } else {
    for (int i = 0; i < nthreads; i++) pthread_create(&th[i], NULL, qmv_worker, &jobs[i]);
    for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
  }
  free(q);
  free(d);
  free(s);
  free(xhat);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* MoE decode layer                                                          */
/* ------------------------------------------------------------------------ */

/* A slot (t, k) is valid when its id lies in [0, E) and does not repeat an
 * earlier id of the same token. */
int oracle_moe_slot_valid(const int32_t* ids, int top_k, int E, int t, int k) {
  int32_t e = ids[t * top_k + k];
  if (e < 0 || e >= E) return 0;
  for (int kk = 0; kk < k; kk++)
    if (ids[t * top_k + kk] == e) return 0;
  return 1;
}

/* Work of one thread over slots [p0, p1) of one of the two per-slot phases
 * of the MoE layer (the slots are independent: each reads only the inputs and
 * writes only its own rows). */
typedef struct {
  int fmt_gu, fmt_d;
  const uint8_t *Wgu, *Wd;
  int64_t rb_gu, rb_d;
  int E, H, F, top_k;
  const int32_t* ids;
  const double* xhat;  /* [n][H] */
  const float* h_in;   /* [S][F] or NULL */
  double *g, *u, *gabs, *uabs;  /* phase 1 outputs (may be NULL) */
  float* hloc;                  /* phase 1: fp32 h [S][F] */
  const int8_t* hq;             /* phase 2 inputs: quantized h */
  const float* hd;
  double *oloc, *oaloc;         /* phase 2 outputs [S][H] */
  int p0, p1;
} moe_job;

/* gate / up / SwiGLU of slots [p0, p1) */
static void* moe_gate_up_worker(void* arg) {
  moe_job* j = (moe_job*)arg;
  const int H = j->H, F = j->F;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)H);
  if (!wrow) return NULL;
  for (int p = j->p0; p < j->p1; p++) {
    int t = p / j->top_k, k = p % j->top_k;
    int valid = oracle_moe_slot_valid(j->ids, j->top_k, j->E, t, k);
    int32_t e = j->ids[p];
    for (int r = 0; r < F; r++) {
      double gv = 0.0, uv = 0.0, ga = 0.0, ua = 0.0;
      if (valid) {
        const uint8_t* base = j->Wgu + (int64_t)e * 2 * F * j->rb_gu;
        dequant_row(j->fmt_gu, base + (int64_t)r * j->rb_gu, H, wrow);
        for (int i = 0; i < H; i++) {
          double pr = wrow[i] * j->xhat[(int64_t)t * H + i];
          gv += pr;
          ga += fabs(pr);
        }
        dequant_row(j->fmt_gu, base + (int64_t)(F + r) * j->rb_gu, H, wrow);
        for (int i = 0; i < H; i++) {
          double pr = wrow[i] * j->xhat[(int64_t)t * H + i];
          uv += pr;
          ua += fabs(pr);
        }
      }
      if (j->g) j->g[(int64_t)p * F + r] = gv;
      if (j->u) j->u[(int64_t)p * F + r] = uv;
      if (j->gabs) j->gabs[(int64_t)p * F + r] = ga;
      if (j->uabs) j->uabs[(int64_t)p * F + r] = ua;
      double hv = valid ? gv / (1.0 + exp(-gv)) * uv : 0.0;
      j->hloc[(int64_t)p * F + r] = j->h_in ? (valid ? j->h_in[(int64_t)p * F + r] : 0.0f) : (float)hv;
    }
  }
  free(wrow);
  return NULL;
}

/* down projection o = Wdown_e Hhat of slots [p0, p1) */
static void* moe_down_worker(void* arg) {
  moe_job* j = (moe_job*)arg;
  const int H = j->H, F = j->F;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)F);
  double* hhat = (double*)malloc(sizeof(double) * (size_t)F);
  if (!wrow || !hhat) {
    free(wrow);
    free(hhat);
    return NULL;
  }
  for (int p = j->p0; p < j->p1; p++) {
    int t = p / j->top_k, k = p % j->top_k;
    int valid = oracle_moe_slot_valid(j->ids, j->top_k, j->E, t, k);
    int32_t e = j->ids[p];
    for (int i = 0; i < F; i++)
      hhat[i] = (double)j->hd[(int64_t)p * (F / 32) + i / 32] * (double)j->hq[(int64_t)p * F + i];
    for (int m = 0; m < H; m++) {
      double ov = 0.0, oa = 0.0;
      if (valid) {
        dequant_row(j->fmt_d, j->Wd + ((int64_t)e * H + m) * j->rb_d, F, wrow);
        for (int i = 0; i < F; i++) {
          double pr = wrow[i] * hhat[i];
          ov += pr;
          oa += fabs(pr);
        }
      }
      j->oloc[(int64_t)p * H + m] = ov;
      j->oaloc[(int64_t)p * H + m] = oa;
    }
  }
  free(wrow);
  free(hhat);
  return NULL;
}

/* Runs fn over the slots [0, S) split into nthreads contiguous ranges. */
static void moe_parallel(void* (*fn)(void*), moe_job proto, int S, int nthreads) {
  moe_job jobs[256];
  pthread_t th[256];
  if (nthreads > S) nthreads = S;
  if (nthreads < 1) nthreads = 1;
  for (int i = 0; i < nthreads; i++) {
    jobs[i] = proto;
    jobs[i].p0 = (int)((int64_t)S * i / nthreads);
    jobs[i].p1 = (int)((int64_t)S * (i + 1) / nthreads);
  }
  if (nthreads == 1) {
    fn(&jobs[0]);
    return;
  }
  for (int i = 0; i < nthreads; i++) pthread_create(&th[i], NULL, fn, &jobs[i]);
  for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
}

/* Full MoE layer.  Optional outputs may be NULL.  If h_in is non-NULL it
 * supplies the fp32 h of every slot (for grading the down/combine stage on
 * given h); otherwise h is computed from x.
 *   y      [n][H]        sum_k gates[t][k] * o_{t,k}  (fp64)
 *   ybound [n][H]        sum_k |gates[t][k]| * sum_i |Wdown_e[m][i] Hhat_i|
 *   g, u   [n*top_k][F]  gate / up projections (fp64)
 *   gabs, uabs [n*top_k][F]  sum_i |What x Xhat| of those rows
 *   h32    [n*top_k][F]  fp32 h (as computed here, or h_in)
 *   hq, hd, hs           activation quantization of h32
 *   o      [n*top_k][H]  down projections (fp64)
 *   oabs   [n*top_k][H]  sum_i |Wdown_e[m][i] Hhat_i| of those rows
 * The slots' gate/up and down projections are computed by nthreads POSIX
 * threads (1 = serial); the combine then adds the slots of each token in k
 * order, so the result does not depend on the thread count. */
int oracle_moe(int fmt_gu, const uint8_t* Wgu, int fmt_d, const uint8_t* Wd, int E,
               int H, int F, const int32_t* ids, const float* gates, const float* x,
               int n, int top_k, const float* h_in, double* y, double* ybound,
               double* g, double* u, double* gabs, double* uabs, float* h32,
               int8_t* hq, float* hd, int32_t* hs, double* o, double* oabs, int nthreads) {
  int64_t rb_gu = oracle_row_bytes(fmt_gu, H), rb_d = oracle_row_bytes(fmt_d, F);
  if (rb_gu < 0 || rb_d < 0 || E <= 0 || n <= 0 || top_k <= 0) return -1;
  if (nthreads > 256) nthreads = 256;
  int S = n * top_k;
  int8_t* xq = (int8_t*)malloc((size_t)n * H);
  float* xd = (float*)malloc(sizeof(float) * (size_t)n * (H / 32));
  int32_t* xs = (int32_t*)malloc(sizeof(int32_t) * (size_t)n * (H / 32));
  double* xhat = (double*)malloc(sizeof(double) * (size_t)n * H);
  float* hloc = (float*)malloc(sizeof(float) * (size_t)S * F);
  int8_t* hql = (int8_t*)malloc((size_t)S * F);
  float* hdl = (float*)malloc(sizeof(float) * (size_t)S * (F / 32));
  int32_t* hsl = (int32_t*)malloc(sizeof(int32_t) * (size_t)S * (F / 32));
  double* oloc = (double*)malloc(sizeof(double) * (size_t)S * H);
  double* oaloc = (double*)malloc(sizeof(double) * (size_t)S * H);
  if (!xq || !xd || !xs || !xhat || !hloc || !hql || !hdl || !hsl || !oloc || !oaloc) return -2;
  oracle_act_quant(x, H, n, xq, xd, xs);
  for (int64_t i = 0; i < (int64_t)n * H; i++)
    xhat[i] = (double)xd[i / 32] * (double)xq[i];

  moe_job proto;
  memset(&proto, 0, sizeof(proto));
  proto.fmt_gu = fmt_gu;
  proto.fmt_d = fmt_d;
  proto.Wgu = Wgu;
  proto.Wd = Wd;
  proto.rb_gu = rb_gu;
  proto.rb_d = rb_d;
  proto.E = E;
  proto.H = H;
  proto.F = F;
  proto.top_k = top_k;
  proto.ids = ids;
  proto.xhat = xhat;
  proto.h_in = h_in;
  proto.g = g;
  proto.u = u;
  proto.gabs = gabs;
  proto.uabs = uabs;
  proto.hloc = hloc;
  proto.hq = hql;
  proto.hd = hdl;
  proto.oloc = oloc;
  proto.oaloc = oaloc;

  /* gate / up / SwiGLU per slot, then the requantization of h */
  moe_parallel(moe_gate_up_worker, proto, S, nthreads);
  oracle_act_quant(hloc, F, S, hql, hdl, hsl);
  if (h32) memcpy(h32, hloc, sizeof(float) * (size_t)S * F);
  if (hq) memcpy(hq, hql, (size_t)S * F);
  if (hd) memcpy(hd, hdl, sizeof(float) * (size_t)S * (F / 32));
  if (hs) memcpy(hs, hsl, sizeof(int32_t) * (size_t)S * (F / 32));

  /* down projection per slot, then the combine in slot (= k) order */
  moe_parallel(moe_down_worker, proto, S, nthreads);
  for (int64_t i = 0; i < (int64_t)n * H; i++) {
    if (y) y[i] = 0.0;
    if (ybound) ybound[i] = 0.0;
  }
  for (int p = 0; p < S; p++) {
    int t = p / top_k;
    double gt = (double)gates[p];
    for (int m = 0; m < H; m++) {
      double ov = oloc[(int64_t)p * H + m], oa = oaloc[(int64_t)p * H + m];
      if (y) y[(int64_t)t * H + m] += gt * ov;
      if (ybound) ybound[(int64_t)t * H + m] += fabs(gt) * oa;
    }
  }
  if (o) memcpy(o, oloc, sizeof(double) * (size_t)S * H);
  if (oabs) memcpy(oabs, oaloc, sizeof(double) * (size_t)S * H);
  free(xq);
  free(xd);
  free(xs);
  free(xhat);
  free(hloc);
  free(hql);
  free(hdl);
  free(hsl);
  free(oloc);
  free(oaloc);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Router gating and top-k                                                   */
/* ------------------------------------------------------------------------ */

/* Per token t of logits [n][E] (fp64): the top_k experts in decreasing
 * order of logit, a tie going to the lower expert index (each pick is the
 * first maximum among the experts not yet picked), and their gates:
 *   gating 0 (softmax): g_k = exp(l_k - l_0) / sum_j exp(l_j - l_0) over the
 *     picked experts (the full softmax renormalised over the picked ones);
 *   gating 1 (sigmoid): g_k = s_k / sum_j s_j, s = 1 / (1 + exp(-l)).
 * Source: "Castagna Veloce", section "Fused operations" (router and top-k:
 * matvec, gating, top-k and weight normalization).  Returns -1 on bad
 * arguments. */
int oracle_route_select(const double* logits, int n, int E, int top_k, int gating, int32_t* ids,
                        double* gates) {
  if (n <= 0 || E <= 0 || top_k <= 0 || top_k > E || (gating != 0 && gating != 1)) return -1;
  char* taken = (char*)malloc((size_t)E);
  if (!taken) return -2;
  for (int t = 0; t < n; t++) {
    const double* l = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int k = 0; k < top_k; k++) {
      int best = -1;
      for (int e = 0; e < E; e++)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[t * top_k + k] = best;
    }
    double sum = 0.0;
    for (int k = 0; k < top_k; k++) {
      double v = l[ids[t * top_k + k]];
      double w = gating == 0 ? exp(v - l[ids[t * top_k]]) : 1.0 / (1.0 + exp(-v));
      gates[t * top_k + k] = w;
      sum += w;
    }
    for (int k = 0; k < top_k; k++) gates[t * top_k + k] /= sum;
  }
  free(taken);
  return 0;
}
