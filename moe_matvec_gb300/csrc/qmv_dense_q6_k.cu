// Dense matvec kernels for the QMV_Q6_K weight format (one unit per format so the
// instantiations compile in parallel).
#include "qmv_dense_inst.cuh"

namespace qmv {
cudaError_t launch_dense_q6_k(const DenseLaunch& L) { return launch_dense_fmt<QMV_Q6_K>(L); }
}  // namespace qmv
