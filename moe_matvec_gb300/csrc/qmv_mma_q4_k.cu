// Tensor-core Q4_K matvec kernels (8 and 16 token slots) and their launcher.
#include <atomic>

#include "launch.h"
#include "qmv_mma.cuh"

namespace qmv {

static_assert(MMA_BOX_BYTES == MK_PITCH && MMA_TILE_ROWS == MK_ROWS, "tensor maps match the stage layout");

template <int NT>
static cudaError_t launch_mma_nt(const DenseLaunch& L) {
  auto kern = qmv_mma_q4k_kernel<NT>;
  // bit per device ordinal; host threads racing on a first launch both set
  // the same attribute, which is harmless
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !((configured.load(std::memory_order_acquire) >> dev) & 1ull)) {
    // the warpgroups' register shares must fit in what the CTA is launched
    // with, or the consumers' request for more would never be granted
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if ((long long)fa.numRegs * MK_THREADS < (long long)MK_PW * 32 * MK_REG_PRODUCER + (long long)MK_CW * 32 * MK_REG_CONSUMER)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_smem_optin());
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3(L.grid, L.passes), dim3(MK_THREADS), L.smem, L.stream, L.pdl);
  return cudaLaunchKernelEx(&cfg, kern, L.map_tile, L.map_unit, *L.p);
}

cudaError_t launch_mma_q4_k(const DenseLaunch& L) {
  switch (L.nt_tmpl) {
    case 8: return launch_mma_nt<8>(L);
    case 16: return launch_mma_nt<16>(L);
  }
  return cudaErrorInvalidValue;
}

size_t mma_smem_bytes(int nt, int stages, int nbmax) { return MmaLayout(nt, stages, nbmax).total; }

}  // namespace qmv
