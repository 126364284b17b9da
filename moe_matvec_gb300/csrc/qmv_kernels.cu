// Small kernels of the path: the standalone activation quantizer and the
// deterministic second pass of the split-K matvec.
#include "launch.h"
#include "qmv_dense.cuh"

namespace qmv {

// Activation rule over x [n_tok][K] into the library's Q8 activation layout:
// the codes of each 256-element group in act_pos order, d and s per block in
// order.  A warp quantizes SU groups per step, four lanes per block.  The
// next kernel may launch at once (it streams weights); this one waits for its
// predecessor before it reads x or writes q / d / s.
__global__ void __launch_bounds__(256) act_quant_kernel(const float* __restrict__ x, int K, int n_tok,
                                                        int8_t* __restrict__ q, float* __restrict__ d,
                                                        int32_t* __restrict__ s
                                                            QMV_DEBUG_ONLY(, unsigned* err, long long x_len,
                                                                           long long q_len)) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int SU = 4;
  const int lane = threadIdx.x & 31, sub = lane >> 2, li = lane & 3;
  const long long groups = (long long)n_tok * (K / 256);
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long g0 = ((long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * SU; g0 < groups;
       g0 += nwarps * SU) {
    float4 v[SU][2];
    uint32_t w0[SU], w1[SU];
    float dd[SU];
    int ss[SU];
#pragma unroll
    for (int u = 0; u < SU; u++) {
      v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g0 + u < groups && QMV_CHECK(in_range((g0 + u) * 256 + sub * 32 + 8 * li, 8, x_len, err))) {
        const float4* p = reinterpret_cast<const float4*>(x + (g0 + u) * 256 + sub * 32) + 2 * li;
        v[u][0] = __ldg(p);
        v[u][1] = __ldg(p + 1);
      }
    }
    quant_units<SU>(v, w0, w1, dd, ss);
#pragma unroll
    for (int u = 0; u < SU; u++) {
      if (g0 + u < groups) {
        const long long g = g0 + u;
        if (QMV_CHECK(in_range(g * 256 + act_pos(sub, 8 * li), 8, q_len, err)))
          *reinterpret_cast<uint2*>(q + g * 256 + act_pos(sub, 8 * li)) = make_uint2(w0[u], w1[u]);
        if (li == 0 && QMV_CHECK(in_range(g * 8 + sub, 1, q_len / 32, err))) {
          d[g * 8 + sub] = dd[u];
          s[g * 8 + sub] = ss[u];
        }
      }
    }
  }
}

// y[t][m] = sum_{s=0..S-1} partial[s][t][m], added in the fixed order of s,
// then + add[t][m] when add is given (add may be y).  The partials of a
// group of splits are all loaded before the first is added, so their
// latencies overlap.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial, float* y,
                                                            const float* add, long long n, int n_split
                                                                QMV_DEBUG_ONLY(, unsigned* err, long long part_len,
                                                                               long long y_len, long long add_len)) {
  pdl_wait();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    // the checks cover partial[s n + i] for every s (i and the last split)
    if (!QMV_CHECK(in_range(i, 1, part_len, err)) || !QMV_CHECK(in_range((long long)(n_split - 1) * n + i, 1, part_len, err))) continue;
    float acc = partial[i];
    int s = 1;
    for (; s + 8 <= n_split; s += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; j++) v[j] = partial[(long long)(s + j) * n + i];
#pragma unroll
      for (int j = 0; j < 8; j++) acc += v[j];
    }
    for (; s < n_split; s++) acc += partial[(long long)s * n + i];
    if (!QMV_CHECK(in_range(i, 1, y_len, err))) continue;
    y[i] = add ? acc + (QMV_CHECK(in_range(i, 1, add_len, err)) ? add[i] : 0.f) : acc;
  }
  pdl_launch_dependents();
}

// MoE combine: y[t][m] = sum over routed slots k (in k order) of
// gates[t][k] * o[t * top_k + k][m]; a slot that does not route (id out of
// range, or repeating an earlier id of the token) adds nothing.  One thread
// per 4 consecutive outputs of a token; the ids, gates and slot outputs of
// the token are all loaded before the first is used (the outputs do not wait
// for the ids), so their latencies overlap.
__global__ void __launch_bounds__(256) moe_combine_kernel(const int32_t* __restrict__ ids,
                                                          const float* __restrict__ gates,
                                                          const float* __restrict__ o, float* __restrict__ y,
                                                          int n_tok, int top_k, int n_experts, int hidden
                                                              QMV_DEBUG_ONLY(, unsigned* err, long long ids_len,
                                                                             long long o_len, long long y_len)) {
  pdl_wait();
  const int q4 = hidden / 4;
  const long long total = (long long)n_tok * q4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / q4), m4 = (int)(i - (long long)t * q4);
    // the slot outputs' addresses do not depend on the ids: loaded at once,
    // beside the ids and gates (a slot that does not route is skipped below,
    // whatever its o holds)
    float4 v[QMV_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++)
      v[k] = k < top_k && QMV_CHECK(in_range(((long long)t * top_k + k) * hidden + 4 * m4, 4, o_len, err))
                 ? reinterpret_cast<const float4*>(o + ((long long)t * top_k + k) * hidden)[m4]
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    int e[QMV_MAX_TOPK];
    float g[QMV_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      const bool in = k < top_k && QMV_CHECK(in_range((long long)t * top_k + k, 1, ids_len, err));
      e[k] = in ? ids[t * top_k + k] : -1;
      g[k] = in ? gates[t * top_k + k] : 0.f;
    }
    bool ok[QMV_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      ok[k] = e[k] >= 0 && e[k] < n_experts;
#pragma unroll
      for (int kk = 0; kk < k; kk++) ok[k] = ok[k] && e[kk] != e[k];
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      if (!ok[k]) continue;
      acc.x = fmaf(g[k], v[k].x, acc.x);
      acc.y = fmaf(g[k], v[k].y, acc.y);
      acc.z = fmaf(g[k], v[k].z, acc.z);
      acc.w = fmaf(g[k], v[k].w, acc.w);
    }
    if (QMV_CHECK(in_range((long long)t * hidden + 4 * m4, 4, y_len, err))) reinterpret_cast<float4*>(y + (long long)t * hidden)[m4] = acc;
  }
  pdl_launch_dependents();
}

// Router gating and top-k: one warp per token over its logits [E] (E <=
// 512, held as up to 16 values per lane).  Each of the top_k picks is a warp
// arg-max over the experts not yet picked (larger logit first, the lower
// index on a tie), so the picks come out in decreasing order of logit; the
// gates are then normalised over the picked experts (softmax: exp(l_k - l_0)
// over their sum; sigmoid: s_k over the sum of s).
constexpr int ROUTE_MAX_PER_LANE = 16;
__global__ void __launch_bounds__(128) route_topk_kernel(const float* __restrict__ logits, int n_tok, int E,
                                                         int top_k, int gating, int32_t* __restrict__ ids,
                                                         float* __restrict__ gates
                                                             QMV_DEBUG_ONLY(, unsigned* err, long long logits_len,
                                                                            long long ids_len)) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t < n_tok) {
    float l[ROUTE_MAX_PER_LANE];
#pragma unroll
    for (int i = 0; i < ROUTE_MAX_PER_LANE; i++) {
      const int e = i * 32 + lane;  // expert of slot i of this lane
      l[i] = e < E && QMV_CHECK(in_range((long long)t * E + e, 1, logits_len, err)) ? logits[(long long)t * E + e] : 0.f;
    }
    unsigned taken = 0;  // bit i: slot i picked (or past E)
#pragma unroll
    for (int i = 0; i < ROUTE_MAX_PER_LANE; i++)
      if (i * 32 + lane >= E) taken |= 1u << i;
    float pick_l[QMV_MAX_TOPK];
    int pick_e[QMV_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      if (k >= top_k) break;
      // this lane's first maximum among its untaken slots (slots are in
      // increasing expert order, so the first one is the lowest index)
      int bi = -1;
      float bl = 0.f;
#pragma unroll
      for (int i = 0; i < ROUTE_MAX_PER_LANE; i++)
        if (!((taken >> i) & 1u) && (bi < 0 || l[i] > bl)) {
          bi = i;
          bl = l[i];
        }
      int be = bi < 0 ? 0x7fffffff : bi * 32 + lane;
      // warp arg-max: larger logit wins, an equal logit goes to the lower expert
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const bool other = oe != 0x7fffffff && (be == 0x7fffffff || ol > bl || (ol == bl && oe < be));
        if (other) {
          bl = ol;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      pick_l[k] = bl;
      pick_e[k] = be;
    }
    float w[QMV_MAX_TOPK], sum = 0.f;
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      if (k >= top_k) break;
      w[k] = gating == QMV_GATING_SOFTMAX ? expf(pick_l[k] - pick_l[0]) : 1.0f / (1.0f + expf(-pick_l[k]));
      sum += w[k];
    }
#pragma unroll
    for (int k = 0; k < QMV_MAX_TOPK; k++) {
      if (k < top_k && lane == k && QMV_CHECK(in_range((long long)t * top_k + k, 1, ids_len, err))) {
        ids[t * top_k + k] = pick_e[k];
        gates[t * top_k + k] = w[k] / sum;
      }
    }
  }
  pdl_launch_dependents();
}

cudaError_t launch_route_topk(const float* logits, int n_tok, int E, int top_k, int gating, int32_t* ids,
                              float* gates, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)((n_tok + 3) / 4)), dim3(128), 0, stream, pdl);
  return cudaLaunchKernelEx(&cfg, route_topk_kernel, logits, n_tok, E, top_k, gating, ids, gates
                            QMV_DEBUG_ONLY(, device_error_word(), (long long)n_tok * E,
                                           output_extent((long long)n_tok * top_k)));
}

cudaError_t launch_moe_combine(const int32_t* ids, const float* gates, const float* o, float* y, int n_tok,
                               int top_k, int n_experts, int hidden, cudaStream_t stream, bool pdl) {
  const long long total = (long long)n_tok * (hidden / 4);
  long long ctas = (total + 255) / 256;
  const long long cap = 4ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)ctas), dim3(256), 0, stream, pdl);
  const long long S = (long long)n_tok * top_k;
  (void)S;
  return cudaLaunchKernelEx(&cfg, moe_combine_kernel, ids, gates, o, y, n_tok, top_k, n_experts, hidden
                            QMV_DEBUG_ONLY(, device_error_word(), S, S * hidden,
                                           output_extent((long long)n_tok * hidden)));
}

// Every non-negative float against the IEEE operations: [0] counts inputs
// where div127_rn differs from __fdiv_rn(a, 127) (a == 0 or a / 127 normal),
// [1] inputs where rcp_rn differs from __frcp_rn (2^-126 <= d <= 2^126).
__global__ void __launch_bounds__(256) check_rounding_kernel(unsigned long long* bad) {
  unsigned long long nd = 0, nr = 0;
  const unsigned stride = gridDim.x * blockDim.x;
  for (unsigned u = blockIdx.x * blockDim.x + threadIdx.x; u <= 0x7F7FFFFFu; u += stride) {
    const float a = __uint_as_float(u);
    if (a == 0.0f || a >= 127.0f * 0x1p-126f)
      nd += __float_as_uint(div127_rn(a)) != __float_as_uint(__fdiv_rn(a, 127.0f));
    if (a >= 0x1p-126f && a <= 0x1p126f) nr += __float_as_uint(rcp_rn(a)) != __float_as_uint(__frcp_rn(a));
    if (u > 0x7F7FFFFFu - stride) break;  // the next step would wrap past FLT_MAX
  }
  if (nd) atomicAdd(&bad[0], nd);
  if (nr) atomicAdd(&bad[1], nr);
}

cudaError_t launch_check_rounding(unsigned long long* bad, cudaStream_t stream) {
  check_rounding_kernel<<<8 * device_sm_count(), 256, 0, stream>>>(bad);
  return cudaGetLastError();
}

void make_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                 cudaStream_t stream, bool pdl) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
}

cudaError_t launch_act_quant(const float* x, int K, int n_tok, int8_t* q, float* d, int32_t* s, long long q_len,
                             cudaStream_t stream, bool pdl) {
  const long long groups = (long long)K / 256 * n_tok;
  long long ctas = (groups + 31) / 32;  // 8 warps x 4 groups
  const long long cap = 8ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)ctas), dim3(256), 0, stream, pdl);
  (void)q_len;
  return cudaLaunchKernelEx(&cfg, act_quant_kernel, x, K, n_tok, q, d, s
                            QMV_DEBUG_ONLY(, device_error_word(), (long long)n_tok * K, q_len));
}

cudaError_t launch_splitk_reduce(const float* partial, float* y, const float* add, long long M, int n_tok, int n_split,
                                 cudaStream_t stream, bool pdl) {
  const long long n = M * n_tok;
  long long ctas = (n + 255) / 256;
  const long long cap = 8ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)ctas), dim3(256), 0, stream, pdl);
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, partial, y, add, n, n_split
                            QMV_DEBUG_ONLY(, device_error_word(), (long long)n_split * n, output_extent(n),
                                           add ? n : 0ll));
}

}  // namespace qmv
