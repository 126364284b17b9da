// Dense matvec kernels for the QMV_Q8_G64 weight format (one unit per format so the
// instantiations compile in parallel).
#include "qmv_dense_inst.cuh"

namespace qmv {
cudaError_t launch_dense_q8_g64(const DenseLaunch& L) { return launch_dense_fmt<QMV_Q8_G64>(L); }
}  // namespace qmv
