// tc_q4_0.cu -- tcgen05 projection kernels for Q4_0 weights.
#include "tc_launch.cuh"

namespace m4q {
cudaError_t launch_tc_q4_0(const ProjLaunch& L) { return launch_tc_impl<kQ4_0>(L); }
}  // namespace m4q
