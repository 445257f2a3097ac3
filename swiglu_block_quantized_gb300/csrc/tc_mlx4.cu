// tc_mlx4.cu -- tcgen05 projection kernels for MLX 4-bit affine weights.
#include "tc_launch.cuh"

namespace m4q {
cudaError_t launch_tc_mlx4(const ProjLaunch& L) { return launch_tc_impl<kMLX4>(L); }
}  // namespace m4q
