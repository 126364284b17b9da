// Dense matvec kernels for the QMV_IQ4_XS weight format (one unit per format so the
// instantiations compile in parallel).
#include "qmv_dense_inst.cuh"

namespace qmv {
cudaError_t launch_dense_iq4_xs(const DenseLaunch& L) { return launch_dense_fmt<QMV_IQ4_XS>(L); }
}  // namespace qmv
