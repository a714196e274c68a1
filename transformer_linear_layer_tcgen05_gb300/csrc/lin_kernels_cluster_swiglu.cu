// lin_kernels_cluster_swiglu.cu -- instantiations of the clustered
// persistent GEMM for matmul_residual_swiglu_a_w16 (cluster sizes 1, 2, 4).
#include "lin_gemm_cluster.cuh"

namespace lin {

cudaError_t launch_gemm_cluster_swiglu(int cn, const TensorMaps& maps, const KernelArgs& args,
                                       cudaStream_t stream) {
  switch (cn) {
    case 1: return launch_cluster_instance<A_SWIGLU_F16, true, 256, 1>(maps, args, stream);
    case 2: return launch_cluster_instance<A_SWIGLU_F16, true, 256, 2>(maps, args, stream);
    case 4: return launch_cluster_instance<A_SWIGLU_F16, true, 256, 4>(maps, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lin
