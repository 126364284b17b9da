// Expert-grouped MoE gate/up kernels for the QMV_Q8_0 weight format.
#include "moe_inst.cuh"

namespace qmv {
cudaError_t launch_moe_gate_up_q8_0(const MoeLaunch& L) { return launch_moe_fmt<QMV_Q8_0, MOE_GATE_UP>(L); }
}  // namespace qmv
