// Small kernels of the path: the standalone activation quantizer and the
// deterministic second pass of the split-K matvec.
#include "launch.h"
#include "qmv_dense.cuh"

namespace qmv {

// Activation rule over x [n_tok][K]: codes in natural order, per-32 scale d
// and code sum s.  Each warp handles 4 blocks per step, 8 lanes per block,
// 4 elements per lane.
__global__ void __launch_bounds__(256) act_quant_kernel(const float* __restrict__ x, int K, int n_tok,
                                                        int8_t* __restrict__ q, float* __restrict__ d,
                                                        int32_t* __restrict__ s) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3, li = lane & 7;
  const long long nblk = (long long)K / 32;
  const long long total = nblk * n_tok;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long base = wid * 4; base < total; base += warps * 4) {
    const long long idx = base + sub;
    const bool ok = idx < total;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) v = __ldg(reinterpret_cast<const float4*>(x + idx * 32) + li);
    Quad qd = quant_quad(v);
    if (ok) {
      reinterpret_cast<uint32_t*>(q + idx * 32)[li] = qd.q;
      if (li == 0) {
        d[idx] = qd.d;
        s[idx] = qd.s;
      }
    }
  }
  pdl_launch_dependents();
}

// y[t][m] = sum_{s=0..S-1} partial[s][t][m], added in the fixed order of s.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial, float* __restrict__ y,
                                                            long long n, int n_split) {
  pdl_wait();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float acc = partial[i];
    for (int s = 1; s < n_split; s++) acc += partial[(long long)s * n + i];
    y[i] = acc;
  }
  pdl_launch_dependents();
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

cudaError_t launch_act_quant(const float* x, int K, int n_tok, int8_t* q, float* d, int32_t* s,
                             cudaStream_t stream, bool pdl) {
  const long long blocks = (long long)K / 32 * n_tok;
  long long ctas = (blocks + 31) / 32;  // 8 warps x 4 blocks per CTA step
  const long long cap = 4ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)ctas), dim3(256), 0, stream, pdl);
  return cudaLaunchKernelEx(&cfg, act_quant_kernel, x, K, n_tok, q, d, s);
}

cudaError_t launch_splitk_reduce(const float* partial, float* y, long long M, int n_tok, int n_split,
                                 cudaStream_t stream, bool pdl) {
  const long long n = M * n_tok;
  long long ctas = (n + 255) / 256;
  const long long cap = 8ll * device_sm_count();
  if (ctas > cap) ctas = cap;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3((unsigned)ctas), dim3(256), 0, stream, pdl);
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, partial, y, n, n_split);
}

}  // namespace qmv
