// Launcher of the expert-grouped MoE kernels for one format and projection:
// picks the compiled token-group size and raises the dynamic shared-memory
// limit once per device.
#pragma once
#include "launch.h"
#include "moe_kernels.cuh"

namespace qmv {

template <int F, int NT, int MODE>
static cudaError_t launch_moe_nt(const MoeLaunch& L) {
  auto kern = moe_qmv_kernel<F, NT, MODE>;
  static unsigned long long configured = 0;  // bit per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             device_smem_optin() - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3(L.grid), dim3(THREADS), L.smem, L.stream, L.pdl);
  return cudaLaunchKernelEx(&cfg, kern, L.map_tile, L.map_unit, *L.p);
}

template <int F, int MODE>
static cudaError_t launch_moe_fmt(const MoeLaunch& L) {
  switch (L.nt_tmpl) {
    case 1: return launch_moe_nt<F, 1, MODE>(L);
    case 2: return launch_moe_nt<F, 2, MODE>(L);
    case 4: return launch_moe_nt<F, 4, MODE>(L);
    case 8: return launch_moe_nt<F, 8, MODE>(L);
    case 16: return launch_moe_nt<F, 16, MODE>(L);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qmv
