// Expert-grouped MoE gate/up kernels for the QMV_IQ4_XS weight format.
#include "moe_inst.cuh"

namespace qmv {
cudaError_t launch_moe_gate_up_iq4_xs(const MoeLaunch& L) { return launch_moe_fmt<QMV_IQ4_XS, MOE_GATE_UP>(L); }
}  // namespace qmv
