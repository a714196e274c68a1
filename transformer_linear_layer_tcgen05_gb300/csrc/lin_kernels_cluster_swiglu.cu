// lin_kernels_cluster_swiglu.cu -- instantiations of the clustered
// persistent GEMM for matmul_residual_swiglu_a_w16 (cluster sizes 1, 2, 4).
#include "lin_gemm_cluster.cuh"

namespace lin {

template <int CN>
using SwigluLaunch = ClusterLaunch<A_SWIGLU_F16, true, 256, CN>;

cudaError_t launch_gemm_cluster_swiglu(int cn, const TensorMaps& maps, const KernelArgs& args,
                                       cudaStream_t stream) {
  switch (cn) {
    case 1: return SwigluLaunch<1>::launch(maps, args, stream);
    case 2: return SwigluLaunch<2>::launch(maps, args, stream);
    case 4: return SwigluLaunch<4>::launch(maps, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

int cluster_capacity_swiglu(int cn, cudaError_t* err) {
  switch (cn) {
    case 1: return SwigluLaunch<1>::capacity(err);
    case 2: return SwigluLaunch<2>::capacity(err);
    case 4: return SwigluLaunch<4>::capacity(err);
    default: *err = cudaErrorInvalidValue; return 0;
  }
}

}  // namespace lin
