// Split-K matvec whose partial sums live in a library-owned static device
// array, for callers that may not allocate device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is off limits, for example a
// plugin executed while its host framework captures a CUDA graph (allocation
// is not allowed during stream capture), or a host that owns every byte of
// device memory and gives libraries none.  Those callers can still pass
// their inputs and outputs; the scratch comes from here instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library holds its QMV_STATIC_SCRATCH_BYTES until the process exits.  In
// host code its name is only a stand-in: the device address is looked up
// once per device (cudaGetSymbolAddress, with that device current) on the
// first call made on that device, which is why that first call should come
// before any stream capture.  All calls share the array: calls that may run
// at the same time on the GPU (different streams, or graphs launched
// concurrently) race on it.  With a split above one and more than 4 tokens,
// the activations quantized once are placed in it too, after the partial
// sums, when both fit (the same arithmetic as the per-CTA quantization,
// bitwise equal results).  Nothing in it needs clearing: every call writes
// each value it reads.
#include <mutex>

#include "../../include/qmv.h"

namespace qmv {

static __device__ __align__(256) unsigned char g_static_scratch[QMV_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_mu;
void* g_addr[64];  // device address of g_static_scratch, per device ordinal

int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return QMV_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return QMV_OK;
}

}  // namespace
}  // namespace qmv

extern "C" int qmv_splitk_run_static(int fmt, const void* W, const float* x, float* y, int64_t M, int64_t K,
                                     int n_tok, int n_split, cudaStream_t stream) {
  if (n_split == 0) {
    n_split = qmv_splitk_choose(fmt, M, K, n_tok);
    if (n_split < 0) return n_split;
  }
  if (n_split < 0) return QMV_ERR_SHAPE;
  if (n_split > 1 && qmv_splitk_workspace_bytes(M, n_tok, n_split) > QMV_STATIC_SCRATCH_BYTES)
    return QMV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (n_split > 1) {
    int rc = qmv::static_scratch(&ws);
    if (rc) return rc;
  }
  return qmv_splitk_run(fmt, W, x, y, M, K, n_tok, n_split, ws, n_split > 1 ? QMV_STATIC_SCRATCH_BYTES : 0,
                        stream);
}
