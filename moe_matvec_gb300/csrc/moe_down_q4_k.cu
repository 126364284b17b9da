// Expert-grouped MoE down kernels for the QMV_Q4_K weight format.
#include "moe_inst.cuh"

namespace qmv {
cudaError_t launch_moe_down_q4_k(const MoeLaunch& L) { return launch_moe_fmt<QMV_Q4_K, MOE_DOWN>(L); }
}  // namespace qmv
