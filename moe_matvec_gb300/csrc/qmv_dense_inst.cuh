// Launcher of the dense matvec kernel for one format: picks the compiled
// token count and raises the dynamic shared-memory limit once per device.
#pragma once
#include <atomic>

#include "launch.h"
#include "qmv_dense.cuh"

namespace qmv {

template <int F, int NT, bool Q8IN, int CW, bool ADD>
static cudaError_t launch_dense_nt(const DenseLaunch& L) {
  using SH = Shape<CW>;
  auto kern = qmv_dense_kernel<F, NT, Q8IN, CW, ADD>;
  // bit per device ordinal; host threads racing on a first launch both
  // set the same attributes, which is harmless
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !((configured.load(std::memory_order_acquire) >> dev) & 1ull)) {
    if constexpr (SH::RESPLIT) {
      // the warpgroups' register shares must fit in what the CTA is launched
      // with, or the consumers' request for more would never be granted
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if ((long long)fa.numRegs * SH::THREADS <
          (long long)SH::PRODUCER_WARPS * 32 * SH::REG_PRODUCER + (long long)CW * 32 * SH::REG_CONSUMER)
        return cudaErrorInvalidConfiguration;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_smem_optin());
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared array as shared memory, so that two CTAs
    // (of this call or of the next one) can be resident together
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3(L.grid, L.passes), dim3(SH::THREADS), L.smem, L.stream, L.pdl);
  return cudaLaunchKernelEx(&cfg, kern, L.map_tile, L.map_unit, *L.p);
}

template <int F, bool Q8IN, bool ADD>
static cudaError_t launch_dense_src(const DenseLaunch& L) {
  if constexpr (is_float(F)) {
    // F16 / F32 rows: eight consumer warps at every token count
    switch (L.nt_tmpl) {
      case 1: return launch_dense_nt<F, 1, false, 8, ADD>(L);
      case 2: return launch_dense_nt<F, 2, false, 8, ADD>(L);
      case 4: return launch_dense_nt<F, 4, false, 8, ADD>(L);
      case 8: return launch_dense_nt<F, 8, false, 8, ADD>(L);
      case 16: return launch_dense_nt<F, 16, false, 8, ADD>(L);
    }
    return cudaErrorInvalidValue;
  } else {
    switch (L.nt_tmpl) {
      case 1: return launch_dense_nt<F, 1, Q8IN, 8, ADD>(L);
      case 2: return launch_dense_nt<F, 2, Q8IN, 8, ADD>(L);
      case 4: return L.cw == 12 ? launch_dense_nt<F, 4, Q8IN, 12, ADD>(L) : launch_dense_nt<F, 4, Q8IN, 8, ADD>(L);
      case 8: return L.cw == 12 ? launch_dense_nt<F, 8, Q8IN, 12, ADD>(L) : launch_dense_nt<F, 8, Q8IN, 8, ADD>(L);
      case 16:
        return L.cw == 12 ? launch_dense_nt<F, 16, Q8IN, 12, ADD>(L) : launch_dense_nt<F, 16, Q8IN, 8, ADD>(L);
    }
    return cudaErrorInvalidValue;
  }
}

template <int F>
static cudaError_t launch_dense_fmt(const DenseLaunch& L) {
  const bool q8 = L.p->x == nullptr, add = L.p->add != nullptr;
  if constexpr (is_float(F)) {
    if (q8) return cudaErrorInvalidValue;
    return add ? launch_dense_src<F, false, true>(L) : launch_dense_src<F, false, false>(L);
  } else {
    if (add) return q8 ? launch_dense_src<F, true, true>(L) : launch_dense_src<F, false, true>(L);
    return q8 ? launch_dense_src<F, true, false>(L) : launch_dense_src<F, false, false>(L);
  }
}

}  // namespace qmv
