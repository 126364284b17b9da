// Host-side launch descriptors shared between the C-ABI dispatcher and the
// per-format kernel instantiation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmv {

struct DenseParams;

struct DenseLaunch {
  const DenseParams* p;
  CUtensorMap map_tile;  // box: a tile's rows (4 per consumer warp) x one chunk
  CUtensorMap map_unit;  // box: UNIT_ROWS rows x one chunk
  int nt_tmpl;           // compiled token count (1, 2, 4, 8, 16)
  int cw;                // consumer warps (8, or 12 from 8 tokens on)
  int grid;              // CTAs per token pass
  int passes;            // token passes of NT tokens (grid y)
  size_t smem;
  cudaStream_t stream;
  bool pdl;
};

cudaError_t launch_dense_q8_0(const DenseLaunch& L);
cudaError_t launch_dense_q4_k(const DenseLaunch& L);
cudaError_t launch_dense_iq4_xs(const DenseLaunch& L);
cudaError_t launch_dense_q5_k(const DenseLaunch& L);
cudaError_t launch_dense_q6_k(const DenseLaunch& L);
cudaError_t launch_dense_q8_g64(const DenseLaunch& L);
cudaError_t launch_dense_q8_g128(const DenseLaunch& L);
cudaError_t launch_dense_f16(const DenseLaunch& L);
cudaError_t launch_dense_f32(const DenseLaunch& L);
// Tensor-core Q4_K matvec (nt_tmpl 8 or 16; map_tile: box MMA_TILE_ROWS rows
// x MMA_BOX_BYTES, map_unit: UNIT_ROWS rows x MMA_BOX_BYTES) and the shared
// memory it takes with `stages` weight stages and split ranges of at most
// nbmax blocks.
constexpr int MMA_BOX_BYTES = 432;
constexpr int MMA_TILE_ROWS = 64;
// Tensor-core F16 matvec (nt_tmpl 8 or 16; boxes of MMA_F16_BOX_BYTES x
// MMA_TILE_ROWS / UNIT_ROWS rows) and its shared memory for split ranges of at
// most kmax weights.
constexpr int MMA_F16_BOX_BYTES = 528;
cudaError_t launch_mma_f16(const DenseLaunch& L);
size_t mma_f16_smem_bytes(int nt, int stages, int kmax);
cudaError_t launch_mma_q4_k(const DenseLaunch& L);
size_t mma_smem_bytes(int nt, int stages, int nbmax);

struct MoeParams;

struct MoeLaunch {
  const MoeParams* p;
  CUtensorMap map_tile;
  CUtensorMap map_unit;
  int nt_tmpl;
  int cw;  // consumer warps: 8, or 12 beside a producer warpgroup
  int grid;
  size_t smem;
  cudaStream_t stream;
  bool pdl;
};

cudaError_t launch_moe_gate_up_q8_0(const MoeLaunch& L);
cudaError_t launch_moe_gate_up_q4_k(const MoeLaunch& L);
cudaError_t launch_moe_gate_up_iq4_xs(const MoeLaunch& L);
cudaError_t launch_moe_down_q8_0(const MoeLaunch& L);
cudaError_t launch_moe_down_q4_k(const MoeLaunch& L);
cudaError_t launch_moe_down_iq4_xs(const MoeLaunch& L);
cudaError_t launch_moe_combine(const int32_t* ids, const float* gates, const float* o, float* y, int n_tok,
                               int top_k, int n_experts, int hidden, cudaStream_t stream, bool pdl);

cudaError_t launch_route_topk(const float* logits, int n_tok, int E, int top_k, int gating, int32_t* ids,
                              float* gates, cudaStream_t stream, bool pdl);
// q_len: the extent (elements) of q for the range checks (d, s: q_len / 32)
cudaError_t launch_act_quant(const float* x, int K, int n_tok, int8_t* q, float* d, int32_t* s, long long q_len,
                             cudaStream_t stream, bool pdl);
cudaError_t launch_splitk_reduce(const float* partial, float* y, const float* add, long long M, int n_tok, int n_split,
                                 cudaStream_t stream, bool pdl);
cudaError_t launch_quantize_weights(int fmt, const float* w, long long M, int K, void* W, cudaStream_t stream);
cudaError_t launch_check_rounding(unsigned long long* bad, cudaStream_t stream);

// 2-D TMA map over `rows` rows of `row_bytes` bytes (8-byte elements), box
// box_rows x box_bytes; false if the driver's encoder is unavailable or
// rejects the arguments.
bool encode_rows(CUtensorMap* map, const void* W, long long rows, long long row_bytes, int box_bytes, int box_rows);

// Maximum dynamic shared memory a CTA may use on the current device.
int device_smem_optin();
unsigned* device_error_word();  // address of the device error word (current device)
// Extent (elements) that the range checks of QMV_DEBUG builds take for a
// result buffer of the caller (y, logits, ids, gates, quantizer outputs) of
// n elements: n, or n less the amount set by qmv_debug_shrink_outputs (never
// below 0).  Workspace buffers always take their full extents.
long long output_extent(long long n);
int device_sm_count();

// Fill a launch config with the optional programmatic-dependent-launch
// attribute (attr must outlive the launch call).
void make_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                 cudaStream_t stream, bool pdl);

}  // namespace qmv
