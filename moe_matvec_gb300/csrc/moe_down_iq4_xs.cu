// Expert-grouped MoE down kernels for the QMV_IQ4_XS weight format.
#include "moe_inst.cuh"

namespace qmv {
cudaError_t launch_moe_down_iq4_xs(const MoeLaunch& L) { return launch_moe_fmt<QMV_IQ4_XS, MOE_DOWN>(L); }
}  // namespace qmv
