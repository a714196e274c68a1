// lin_kernels_f16.cu -- instantiations of the tcgen05 GEMM for the binary16
// weight forms: matmul_w16, matmul_residual_w16 (A = X rounded to binary16 by
// the transform warps) and matmul_residual_swiglu_a_w16 (A = silu(GATE) * UP
// rounded to binary16).
#include "lin_gemm.cuh"

namespace lin {

cudaError_t launch_gemm_f16(int amode, bool resid, int bn, bool bt, const TensorMaps& maps,
                            const KernelArgs& args, cudaStream_t stream) {
  if (bt) {   // dY · W^T with binary16 W as [N][K]
    if (amode != A_CVT_F16 || bn != 128) return cudaErrorInvalidValue;
    return resid ? launch_instance<A_CVT_F16, true, 128, true>(maps, args, stream)
                 : launch_instance<A_CVT_F16, false, 128, true>(maps, args, stream);
  }
  if (bn != 128) return cudaErrorInvalidValue;
  if (amode == A_CVT_F16)
    return resid ? launch_instance<A_CVT_F16, true, 128>(maps, args, stream)
                 : launch_instance<A_CVT_F16, false, 128>(maps, args, stream);
  if (amode == A_SWIGLU_F16 && resid)
    return launch_instance<A_SWIGLU_F16, true, 128>(maps, args, stream);
  return cudaErrorInvalidValue;
}

}  // namespace lin
