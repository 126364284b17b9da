// Weight quantizers (a preparation step, not part of the decode hot path):
// fp32 weights -> the library's Q8_0 / Q4_K / IQ4_XS / Q5_K / Q6_K / Q8 group-64 /
// group-128 groups.  Each scale is
// chosen from its block's range and each code is the nearest grid point, in
// fp64 with every operation written as an explicitly rounded IEEE intrinsic
// (no contraction), so the bytes do not depend on the compiler.  One thread
// builds one group in registers / local memory and writes it out.
#include "common.cuh"
#include "launch.h"

namespace qmv {

namespace {

__device__ __forceinline__ uint16_t f16_bits(double v) { return __half_as_ushort(__double2half(v)); }
__device__ __forceinline__ double f16_val(uint16_t b) { return (double)__half2float(__ushort_as_half(b)); }

__device__ __forceinline__ void put_bits(uint8_t* s, int bit, int nbits, unsigned v) {
  for (int i = 0; i < nbits; i++) {
    const int b = bit + i;
    if ((v >> i) & 1u)
      s[b >> 3] |= (uint8_t)(1u << (b & 7));
    else
      s[b >> 3] &= (uint8_t)~(1u << (b & 7));
  }
}
__device__ __forceinline__ void put_nib(uint8_t* p, int i, unsigned c) {
  if (i < 16)
    p[i] = (uint8_t)((p[i] & 0xF0) | (c & 0xF));
  else
    p[i - 16] = (uint8_t)((p[i - 16] & 0x0F) | ((c & 0xF) << 4));
}

__device__ __forceinline__ double clampd(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }

__device__ void group_q8_0(const float* w, uint8_t* g) {
  for (int b = 0; b < 8; b++) {
    double amax = 0.0;
    for (int i = 0; i < 32; i++) amax = fmax(amax, fabs((double)w[32 * b + i]));
    const uint16_t d16 = f16_bits(__ddiv_rn(amax, 127.0));
    const double dv = f16_val(d16);
    g[2 * b] = (uint8_t)(d16 & 0xFF);
    g[2 * b + 1] = (uint8_t)(d16 >> 8);
    for (int i = 0; i < 32; i++) {
      double r = 0.0;
      if (dv > 0.0) r = clampd(rint(__ddiv_rn((double)w[32 * b + i], dv)), -127.0, 127.0);
      const int off = i < 16 ? 16 * b + i : 128 + 16 * b + (i - 16);
      g[16 + off] = (uint8_t)(int8_t)(int)r;
    }
  }
}

__device__ void group_q4_k(const float* w, uint8_t* g) {
  double a[8], bm[8], amax = 0.0, bmax = 0.0;
  for (int j = 0; j < 8; j++) {
    double lo = 0.0, hi = -INFINITY;
    for (int i = 0; i < 32; i++) {
      const double v = (double)w[32 * j + i];
      lo = fmin(lo, v);
      hi = fmax(hi, v);
    }
    a[j] = __ddiv_rn(__dsub_rn(hi, lo), 15.0);
    bm[j] = -lo;
    amax = fmax(amax, a[j]);
    bmax = fmax(bmax, bm[j]);
  }
  const uint16_t d16 = f16_bits(__ddiv_rn(amax, 63.0)), dm16 = f16_bits(__ddiv_rn(bmax, 63.0));
  const double dv = f16_val(d16), dmv = f16_val(dm16);
  g[0] = (uint8_t)(d16 & 0xFF);
  g[1] = (uint8_t)(d16 >> 8);
  g[2] = (uint8_t)(dm16 & 0xFF);
  g[3] = (uint8_t)(dm16 >> 8);
  for (int j = 0; j < 8; j++) {
    const double sc = dv > 0.0 ? clampd(rint(__ddiv_rn(a[j], dv)), 0.0, 63.0) : 0.0;
    const double m = dmv > 0.0 ? clampd(rint(__ddiv_rn(bm[j], dmv)), 0.0, 63.0) : 0.0;
    put_bits(g + 4, 12 * j, 6, (unsigned)sc);
    put_bits(g + 4, 12 * j + 6, 6, (unsigned)m);
    const double S = __dmul_rn(dv, sc), O = __dmul_rn(dmv, m);
    for (int i = 0; i < 32; i++) {
      const double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(__dsub_rn(v, __dsub_rn(__dmul_rn(S, 0.0), O)));
      for (int q = 1; q < 16; q++) {
        const double e = fabs(__dsub_rn(v, __dsub_rn(__dmul_rn(S, (double)q), O)));
        if (e < berr) {
          berr = e;
          best = q;
        }
      }
      put_nib(g + 16 + 16 * j, i, (unsigned)best);
    }
  }
}

// Q5_K: Q4_K's fit with 31 steps; the low four bits of each code go to the
// nibble area at byte 48, the fifth to the bit words at byte 16.
__device__ void group_q5_k(const float* w, uint8_t* g) {
  double a[8], bm[8], amax = 0.0, bmax = 0.0;
  for (int j = 0; j < 8; j++) {
    double lo = 0.0, hi = -INFINITY;
    for (int i = 0; i < 32; i++) {
      const double v = (double)w[32 * j + i];
      lo = fmin(lo, v);
      hi = fmax(hi, v);
    }
    a[j] = __ddiv_rn(__dsub_rn(hi, lo), 31.0);
    bm[j] = -lo;
    amax = fmax(amax, a[j]);
    bmax = fmax(bmax, bm[j]);
  }
  const uint16_t d16 = f16_bits(__ddiv_rn(amax, 63.0)), dm16 = f16_bits(__ddiv_rn(bmax, 63.0));
  const double dv = f16_val(d16), dmv = f16_val(dm16);
  g[0] = (uint8_t)(d16 & 0xFF);
  g[1] = (uint8_t)(d16 >> 8);
  g[2] = (uint8_t)(dm16 & 0xFF);
  g[3] = (uint8_t)(dm16 >> 8);
  for (int j = 0; j < 8; j++) {
    const double sc = dv > 0.0 ? clampd(rint(__ddiv_rn(a[j], dv)), 0.0, 63.0) : 0.0;
    const double m = dmv > 0.0 ? clampd(rint(__ddiv_rn(bm[j], dmv)), 0.0, 63.0) : 0.0;
    put_bits(g + 4, 12 * j, 6, (unsigned)sc);
    put_bits(g + 4, 12 * j + 6, 6, (unsigned)m);
    const double S = __dmul_rn(dv, sc), O = __dmul_rn(dmv, m);
    for (int i = 0; i < 32; i++) {
      const double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(__dsub_rn(v, __dsub_rn(__dmul_rn(S, 0.0), O)));
      for (int q = 1; q < 32; q++) {
        const double e = fabs(__dsub_rn(v, __dsub_rn(__dmul_rn(S, (double)q), O)));
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

// Q6_K: per 16 weights s_i = amax_i / 31, d = max s_i / 127, 7-bit sc_i;
// codes v = (q - 32) mod 64, low four bits in the nibble area at byte 80,
// the top two in the block's bit words at byte 16 (weight e of a word at
// bit 8 (e % 4) + 2 (e / 4)).
__device__ void group_q6_k(const float* w, uint8_t* g) {
  double s[16], smax = 0.0;
  for (int i = 0; i < 16; i++) {
    double amax = 0.0;
    for (int k = 0; k < 16; k++) amax = fmax(amax, fabs((double)w[16 * i + k]));
    s[i] = __ddiv_rn(amax, 31.0);
    smax = fmax(smax, s[i]);
  }
  const uint16_t d16 = f16_bits(__ddiv_rn(smax, 127.0));
  const double dv = f16_val(d16);
  g[0] = (uint8_t)(d16 & 0xFF);
  g[1] = (uint8_t)(d16 >> 8);
  for (int i = 0; i < 16; i++) {
    const double sc = dv > 0.0 ? clampd(rint(__ddiv_rn(s[i], dv)), 0.0, 127.0) : 0.0;
    put_bits(g + 2, 7 * i, 7, (unsigned)sc);
    const double S = __dmul_rn(dv, sc);
    for (int k = 0; k < 16; k++) {
      const double v = (double)w[16 * i + k];
      int best = 0;
      double berr = fabs(__dsub_rn(v, __dmul_rn(S, -32.0)));
      for (int q = 1; q < 64; q++) {
        const double e = fabs(__dsub_rn(v, __dmul_rn(S, (double)(q - 32))));
        if (e < berr) {
          berr = e;
          best = q;
        }
      }
      const int el = 16 * i + k, j = el >> 5, ii = el & 31, e = ii & 15;
      const unsigned code = (unsigned)(best - 32) & 63u;
      put_nib(g + 80 + 16 * j, ii, code & 15u);
      put_bits(g + 16 + 8 * j + 4 * (ii >> 4), 8 * (e & 3) + 2 * (e >> 2), 2, code >> 4);
    }
  }
}

// Q8 with one scale per GS weights over a group of 8 GS: the Q8_0 rule per
// scale group, codes in Q8_0's payload order per 256 weights.
template <int GS>
__device__ void group_q8_g(const float* w, uint8_t* g) {
  for (int sidx = 0; sidx < 8; sidx++) {
    double amax = 0.0;
    for (int i = 0; i < GS; i++) amax = fmax(amax, fabs((double)w[GS * sidx + i]));
    const uint16_t d16 = f16_bits(__ddiv_rn(amax, 127.0));
    const double dv = f16_val(d16);
    g[2 * sidx] = (uint8_t)(d16 & 0xFF);
    g[2 * sidx + 1] = (uint8_t)(d16 >> 8);
    for (int i = 0; i < GS; i++) {
      const int el = GS * sidx + i, half = el >> 8, b = (el >> 5) & 7, ii = el & 31;
      double r = 0.0;
      if (dv > 0.0) r = clampd(rint(__ddiv_rn((double)w[el], dv)), -127.0, 127.0);
      const int off = ii < 16 ? 16 * b + ii : 128 + 16 * b + (ii - 16);
      g[16 + 256 * half + off] = (uint8_t)(int8_t)(int)r;
    }
  }
}

__device__ void superblock_iq4_xs(const float* w, uint8_t* meta, uint8_t* payload) {
  const double cb[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};
  double s[8], smax = 0.0;
  for (int j = 0; j < 8; j++) {
    double amax = 0.0;
    for (int i = 0; i < 32; i++) amax = fmax(amax, fabs((double)w[32 * j + i]));
    s[j] = __ddiv_rn(amax, 113.0);
    smax = fmax(smax, s[j]);
  }
  const uint16_t d16 = f16_bits(__ddiv_rn(smax, 31.0));
  const double dv = f16_val(d16);
  meta[0] = (uint8_t)(d16 & 0xFF);
  meta[1] = (uint8_t)(d16 >> 8);
  for (int j = 0; j < 8; j++) {
    const double l = dv > 0.0 ? clampd(rint(__ddiv_rn(s[j], dv)), 0.0, 31.0) : 0.0;
    const int ls = 32 + (int)l;
    put_bits(meta + 2, 6 * j, 6, (unsigned)ls);
    const double e = __dmul_rn(dv, (double)(ls - 32));
    for (int i = 0; i < 32; i++) {
      const double v = (double)w[32 * j + i];
      int best = 0;
      double berr = fabs(__dsub_rn(v, __dmul_rn(e, cb[0])));
      for (int c = 1; c < 16; c++) {
        const double err = fabs(__dsub_rn(v, __dmul_rn(e, cb[c])));
        if (err < berr) {
          berr = err;
          best = c;
        }
      }
      put_nib(payload + 16 * j, i, (unsigned)best);
    }
  }
}

template <int F>
__global__ void __launch_bounds__(128) quantize_kernel(const float* __restrict__ w, long long n_groups, int K,
                                                       uint8_t* __restrict__ W
                                                           QMV_DEBUG_ONLY(, unsigned* err, long long w_len,
                                                                          long long W_len)) {
  constexpr int GW = Fmt<F>::GW, GB = Fmt<F>::GB;
  const long long gpr = K / GW;
  for (long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x; gi < n_groups;
       gi += (long long)gridDim.x * blockDim.x) {
    const long long row = gi / gpr, col = gi - row * gpr;
    // the group reads w[row K + col GW ..] (GW values) and writes GB bytes at W + gi GB
    if (!QMV_CHECK(in_range(row * K + col * GW, GW, w_len, err)) ||
        !QMV_CHECK(in_range(gi * GB, GB, W_len, err)))
      continue;
    const float* src = w + row * K + col * GW;
    __align__(16) uint8_t g[GB];
    for (int i = 0; i < GB; i++) g[i] = 0;
    if constexpr (F == QMV_Q8_0)
      group_q8_0(src, g);
    else if constexpr (F == QMV_Q4_K)
      group_q4_k(src, g);
    else if constexpr (F == QMV_Q5_K)
      group_q5_k(src, g);
    else if constexpr (F == QMV_Q6_K)
      group_q6_k(src, g);
    else if constexpr (F == QMV_Q8_G64)
      group_q8_g<64>(src, g);
    else if constexpr (F == QMV_Q8_G128)
      group_q8_g<128>(src, g);
    else {
      superblock_iq4_xs(src, g, g + 16);
      superblock_iq4_xs(src + 256, g + 8, g + 16 + 128);
    }
    uint4* dst = reinterpret_cast<uint4*>(W + gi * GB);
    const uint4* s4 = reinterpret_cast<const uint4*>(g);
    for (int i = 0; i < GB / 16; i++) dst[i] = s4[i];
  }
}

}  // namespace

// F16 / F32 rows: one conversion per weight (binary16 rounded to nearest
// even, or the fp32 value as it is); the rows are the flat [M][K] array.
template <int F>
__global__ void convert_rows_kernel(const float* __restrict__ w, long long n, uint8_t* __restrict__ out
                                        QMV_DEBUG_ONLY(, unsigned* err, long long out_len)) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    if (!QMV_CHECK(in_range(i, 1, out_len, err))) continue;  // (w holds the same n elements)
    if constexpr (F == QMV_F16)
      reinterpret_cast<__half*>(out)[i] = __float2half_rn(w[i]);
    else
      reinterpret_cast<float*>(out)[i] = w[i];
  }
}

// extents: w holds M K values, W the M (K / GW) groups of GB bytes
template <int F>
static void quantize_groups(const float* w, long long M, int K, uint8_t* W, long long ctas, cudaStream_t stream) {
  const long long groups = M * (K / Fmt<F>::GW);
  quantize_kernel<F><<<(unsigned)ctas, 128, 0, stream>>>(
      w, groups, K, W QMV_DEBUG_ONLY(, device_error_word(), M * K, output_extent(groups * Fmt<F>::GB)));
}

cudaError_t launch_quantize_weights(int fmt, const float* w, long long M, int K, void* W, cudaStream_t stream) {
  if (fmt == QMV_F16 || fmt == QMV_F32) {
    const long long n = M * K;
    long long ctas = (n + 255) / 256;
    const long long cap = 32ll * device_sm_count();
    if (ctas > cap) ctas = cap;
    if (fmt == QMV_F16)
      convert_rows_kernel<QMV_F16><<<(unsigned)ctas, 256, 0, stream>>>(
          w, n, static_cast<uint8_t*>(W) QMV_DEBUG_ONLY(, device_error_word(), output_extent(n)));
    else
      convert_rows_kernel<QMV_F32><<<(unsigned)ctas, 256, 0, stream>>>(
          w, n, static_cast<uint8_t*>(W) QMV_DEBUG_ONLY(, device_error_word(), output_extent(n)));
    return cudaGetLastError();
  }
  const int gw = fmt == QMV_IQ4_XS || fmt == QMV_Q8_G64 ? 512 : (fmt == QMV_Q8_G128 ? 1024 : 256);
  long long groups = M * (K / gw);
  long long ctas = (groups + 127) / 128;
  const long long cap = 32ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  uint8_t* out = static_cast<uint8_t*>(W);
  switch (fmt) {
    case QMV_Q8_0: quantize_groups<QMV_Q8_0>(w, M, K, out, ctas, stream); break;
    case QMV_Q4_K: quantize_groups<QMV_Q4_K>(w, M, K, out, ctas, stream); break;
    case QMV_Q5_K: quantize_groups<QMV_Q5_K>(w, M, K, out, ctas, stream); break;
    case QMV_Q6_K: quantize_groups<QMV_Q6_K>(w, M, K, out, ctas, stream); break;
    case QMV_Q8_G64: quantize_groups<QMV_Q8_G64>(w, M, K, out, ctas, stream); break;
    case QMV_Q8_G128: quantize_groups<QMV_Q8_G128>(w, M, K, out, ctas, stream); break;
    default: quantize_groups<QMV_IQ4_XS>(w, M, K, out, ctas, stream); break;
  }
  return cudaGetLastError();
}

}  // namespace qmv
