// lin_kernels_cluster_cvt.cu -- instantiations of the clustered persistent
// GEMM for matmul_w16 and matmul_residual_w16 (A rounded to binary16 by
// the transform warps in clusters of 1, 2 or 4 CTAs, or by a pre-pass and
// then copied by TMA into single CTAs or CTA pairs), the pre-pass, and the
// split-tail sum shared by every clustered form.
#include "lin_gemm_cluster.cuh"

namespace lin {

template <bool RESID, int CN>
using CvtLaunch = ClusterLaunch<A_CVT_F16, RESID, 256, CN>;

template <bool RESID, int CN>
using TmaLaunch = ClusterLaunch<A_TMA_F16, RESID, 256, CN>;

// cn: 1 (single CTAs) or 2 (CTA pairs along M)
cudaError_t launch_gemm_cluster_tma(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream) {
  switch (cn * 2 + (resid ? 1 : 0)) {
    case 2: return TmaLaunch<false, 1>::launch(maps, args, stream);
    case 3: return TmaLaunch<true, 1>::launch(maps, args, stream);
    case 4: return TmaLaunch<false, 2>::launch(maps, args, stream);
    case 5: return TmaLaunch<true, 2>::launch(maps, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

int cluster_capacity_tma(int cn, bool resid, cudaError_t* err) {
  switch (cn * 2 + (resid ? 1 : 0)) {
    case 2: return TmaLaunch<false, 1>::capacity(err);
    case 3: return TmaLaunch<true, 1>::capacity(err);
    case 4: return TmaLaunch<false, 2>::capacity(err);
    case 5: return TmaLaunch<true, 2>::capacity(err);
    default: *err = cudaErrorInvalidValue; return 0;
  }
}

// X -> binary16, four elements per thread and step (one 16-byte load, one
// 8-byte store), the same rounding as the transform warps (pack_half2).
__global__ void __launch_bounds__(256)
    lin_cvt_f16_kernel(const float4* __restrict__ x, uint2* __restrict__ y, long long n4) {
  // The GEMM that reads the result may be scheduled now; it waits for this
  // grid's completion itself before it touches memory.
  pdl_launch_dependents();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = ldg_stream_v4f(reinterpret_cast<const float*>(x + i));
    y[i] = make_uint2(pack_half2(v.x, v.y), pack_half2(v.z, v.w));
  }
}

cudaError_t launch_cvt_f16(const float* X, uint16_t* Xh, int64_t n, int sms, cudaStream_t stream) {
  const long long n4 = n / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, lin_cvt_f16_kernel, reinterpret_cast<const float4*>(X),
                            reinterpret_cast<uint2*>(Xh), n4);
}

__global__ void lin_selftest_check_kernel(int* status, long long value) {
  report_check(status, CHK_SELFTEST, value);
}

cudaError_t launch_selftest_check(int* status, long long value, cudaStream_t stream) {
  lin_selftest_check_kernel<<<1, 1, 0, stream>>>(status, value);
  return cudaGetLastError();
}

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

cudaError_t launch_split_reduce(const KernelArgs& args, bool resid, int cn, bool pair, int bn,
                                int tile0, int num_ng, cudaStream_t stream) {
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
  if (args.flags & KFLAG_SWIGLU_BWD)
    return cudaLaunchKernelEx(&cfg, lin_split_reduce_kernel<false, true>, part, args.R, args.Y,
                              args.M, args.N, cn, pair ? 1 : 0, bn, tile0, num_ng, args.band_ng,
                              args.split_rem, args.split_s,
                              args.G2, args.U2, args.Y2, (long long)args.part_f4,
                              args.status);
  if (resid)
    return cudaLaunchKernelEx(&cfg, lin_split_reduce_kernel<true, false>, part, args.R, args.Y,
                              args.M, args.N, cn, pair ? 1 : 0, bn, tile0, num_ng, args.band_ng,
                              args.split_rem, args.split_s,
                              args.G2, args.U2, args.Y2, (long long)args.part_f4,
                              args.status);
  return cudaLaunchKernelEx(&cfg, lin_split_reduce_kernel<false, false>, part, args.R, args.Y,
                            args.M, args.N, cn, pair ? 1 : 0, bn, tile0, num_ng, args.band_ng,
                              args.split_rem, args.split_s,
                            args.G2, args.U2, args.Y2, (long long)args.part_f4,
                              args.status);
}

}  // namespace lin
