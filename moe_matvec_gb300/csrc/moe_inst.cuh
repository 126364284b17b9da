// Launcher of the expert-grouped MoE kernels for one format and projection:
// picks the compiled token-group size and raises the dynamic shared-memory
// limit once per device.
#pragma once
#include <atomic>

#include "launch.h"
#include "moe_kernels.cuh"

namespace qmv {

template <int F, int NT, int MODE, int CW>
static cudaError_t launch_moe_nt(const MoeLaunch& L) {
  using SH = Shape<CW>;
  auto kern = moe_qmv_kernel<F, NT, MODE, CW>;
  // bit per device ordinal; host threads racing on a first launch both
  // set the same attributes, which is harmless
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !((configured.load(std::memory_order_acquire) >> dev) & 1ull)) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // the warpgroups' register shares must fit in what the CTA is launched
    // with, or the consumers' request for more would never be granted
    if (SH::RESPLIT && (long long)fa.numRegs * SH::THREADS <
                           (long long)SH::PRODUCER_WARPS * 32 * SH::REG_PRODUCER + (long long)CW * 32 * SH::REG_CONSUMER)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             device_smem_optin() - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3(L.grid), dim3(SH::THREADS), L.smem, L.stream, L.pdl);
  return cudaLaunchKernelEx(&cfg, kern, L.map_tile, L.map_unit, *L.p);
}

template <int F, int MODE>
static cudaError_t launch_moe_fmt(const MoeLaunch& L) {
  switch (L.nt_tmpl) {
    case 1: return launch_moe_nt<F, 1, MODE, 8>(L);
    case 2: return launch_moe_nt<F, 2, MODE, 8>(L);
    case 4: return launch_moe_nt<F, 4, MODE, 8>(L);
    case 8: return L.cw == 12 ? launch_moe_nt<F, 8, MODE, 12>(L) : launch_moe_nt<F, 8, MODE, 8>(L);
    case 16: return L.cw == 12 ? launch_moe_nt<F, 16, MODE, 12>(L) : launch_moe_nt<F, 16, MODE, 8>(L);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qmv
