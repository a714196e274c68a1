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

cudaError_t launch_split_reduce(const KernelArgs& args, bool resid, int cn, int clusters,
                                int num_ng, cudaStream_t stream) {
  const long long threads = (long long)args.split_rem * cn * 128 * (kClusterBN / 4);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  const int tile0 = args.split_r * clusters;
  const float4* part = reinterpret_cast<const float4*>(args.part);
  if (resid)
    lin_split_reduce_kernel<true><<<blocks, 256, 0, stream>>>(part, args.R, args.Y, args.M, args.N,
                                                             cn, kClusterBN, tile0, num_ng,
                                                             args.split_rem, args.split_s);
  else
    lin_split_reduce_kernel<false><<<blocks, 256, 0, stream>>>(part, args.R, args.Y, args.M,
                                                              args.N, cn, kClusterBN, tile0,
                                                              num_ng, args.split_rem,
                                                              args.split_s);
  return cudaGetLastError();
}

}  // namespace lin
