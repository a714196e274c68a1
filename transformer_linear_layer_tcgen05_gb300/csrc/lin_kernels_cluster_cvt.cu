// lin_kernels_cluster_cvt.cu -- instantiations of the clustered persistent
// GEMM for matmul_w16 and matmul_residual_w16 (cluster sizes 1, 2, 4), and
// the split-tail sum shared by every clustered form.
#include "lin_gemm_cluster.cuh"

namespace lin {

template <bool RESID, int CN>
using CvtLaunch = ClusterLaunch<A_CVT_F16, RESID, 256, CN>;

cudaError_t launch_gemm_cluster_cvt(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream) {
  if (resid) {
    switch (cn) {
      case 1: return CvtLaunch<true, 1>::launch(maps, args, stream);
      case 2: return CvtLaunch<true, 2>::launch(maps, args, stream);
      case 4: return CvtLaunch<true, 4>::launch(maps, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (cn) {
    case 1: return CvtLaunch<false, 1>::launch(maps, args, stream);
    case 2: return CvtLaunch<false, 2>::launch(maps, args, stream);
    case 4: return CvtLaunch<false, 4>::launch(maps, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

int cluster_capacity_cvt(int cn, bool resid, cudaError_t* err) {
  if (resid) {
    switch (cn) {
      case 1: return CvtLaunch<true, 1>::capacity(err);
      case 2: return CvtLaunch<true, 2>::capacity(err);
      case 4: return CvtLaunch<true, 4>::capacity(err);
      default: *err = cudaErrorInvalidValue; return 0;
    }
  }
  switch (cn) {
    case 1: return CvtLaunch<false, 1>::capacity(err);
    case 2: return CvtLaunch<false, 2>::capacity(err);
    case 4: return CvtLaunch<false, 4>::capacity(err);
    default: *err = cudaErrorInvalidValue; return 0;
  }
}

cudaError_t launch_split_reduce(const KernelArgs& args, bool resid, int cn, int bn, int tile0,
                                int num_ng, cudaStream_t stream) {
  const long long threads = (long long)args.split_rem * cn * 128 * (bn / 4);
  // Programmatic dependent launch: the sum is scheduled while the GEMM still
  // runs and waits for it in griddepcontrol.wait, hiding the launch gap.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + 255) / 256), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float4* part = reinterpret_cast<const float4*>(args.part);
  if (resid)
    return cudaLaunchKernelEx(&cfg, lin_split_reduce_kernel<true>, part, args.R, args.Y, args.M,
                              args.N, cn, bn, tile0, num_ng, args.split_rem, args.split_s);
  return cudaLaunchKernelEx(&cfg, lin_split_reduce_kernel<false>, part, args.R, args.Y, args.M,
                            args.N, cn, bn, tile0, num_ng, args.split_rem, args.split_s);
}

}  // namespace lin
