// Dense matvec kernels for the QMV_Q5_K weight format (one unit per format so the
// instantiations compile in parallel).
#include "qmv_dense_inst.cuh"

namespace qmv {
cudaError_t launch_dense_q5_k(const DenseLaunch& L) { return launch_dense_fmt<QMV_Q5_K>(L); }
}  // namespace qmv
