// Dense matvec kernels for the QMV_F16 weight format (one unit per format so the
// instantiations compile in parallel).
#include "qmv_dense_inst.cuh"

namespace qmv {
cudaError_t launch_dense_f16(const DenseLaunch& L) { return launch_dense_fmt<QMV_F16>(L); }
}  // namespace qmv
