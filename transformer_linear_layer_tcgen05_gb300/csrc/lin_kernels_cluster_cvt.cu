// lin_kernels_cluster_cvt.cu -- instantiations of the clustered persistent
// GEMM for matmul_w16 and matmul_residual_w16 (cluster sizes 1, 2, 4).
#include "lin_gemm_cluster.cuh"

namespace lin {

cudaError_t launch_gemm_cluster_cvt(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream) {
  if (resid) {
    switch (cn) {
      case 1: return launch_cluster_instance<A_CVT_F16, true, 256, 1>(maps, args, stream);
      case 2: return launch_cluster_instance<A_CVT_F16, true, 256, 2>(maps, args, stream);
      case 4: return launch_cluster_instance<A_CVT_F16, true, 256, 4>(maps, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (cn) {
    case 1: return launch_cluster_instance<A_CVT_F16, false, 256, 1>(maps, args, stream);
    case 2: return launch_cluster_instance<A_CVT_F16, false, 256, 2>(maps, args, stream);
    case 4: return launch_cluster_instance<A_CVT_F16, false, 256, 4>(maps, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lin
