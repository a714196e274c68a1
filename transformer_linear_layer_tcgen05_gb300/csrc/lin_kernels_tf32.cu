// lin_kernels_tf32.cu -- instantiations of the tcgen05 GEMM whose operands
// are f32 consumed as TF32: matmul, matmul_residual (A copied by TMA) and
// matmul_residual_swiglu_a (A = silu(GATE) * UP built by the transform warps).
#include "lin_gemm.cuh"

namespace lin {

cudaError_t launch_gemm_tf32(int amode, bool resid, int bn, bool bt, const TensorMaps& maps,
                             const KernelArgs& args, cudaStream_t stream) {
  if (bt) {   // dY · W^T: both operands copied by TMA, nothing to transform
    if (amode != A_TMA_F32 || (bn != 128 && bn != 96)) return cudaErrorInvalidValue;
    if (bn == 96)
      return resid ? launch_instance<A_TMA_F32, true, 96, true>(maps, args, stream)
                   : launch_instance<A_TMA_F32, false, 96, true>(maps, args, stream);
    return resid ? launch_instance<A_TMA_F32, true, 128, true>(maps, args, stream)
                 : launch_instance<A_TMA_F32, false, 128, true>(maps, args, stream);
  }
  // the forward SwiGLU form also in 256-column tiles (each row block's
  // SwiGLU A built half as often)
  if (amode == A_SWIGLU_F32 && resid && bn == 256)
    return launch_instance<A_SWIGLU_F32, true, 256>(maps, args, stream);
  // X copied as is, in 96-column tiles: 4/3 as many tiles as 128 columns
  // give, for shapes whose 128-column tiles leave SMs idle
  if (amode == A_TMA_F32 && bn == 96)
    return resid ? launch_instance<A_TMA_F32, true, 96>(maps, args, stream)
                 : launch_instance<A_TMA_F32, false, 96>(maps, args, stream);
  if (bn != 128) return cudaErrorInvalidValue;
  if (amode == A_TMA_F32)
    return resid ? launch_instance<A_TMA_F32, true, 128>(maps, args, stream)
                 : launch_instance<A_TMA_F32, false, 128>(maps, args, stream);
  if (amode == A_TRANS_F32)   // the weight gradient X^T dY (+ dW)
    return resid ? launch_instance<A_TRANS_F32, true, 128>(maps, args, stream)
                 : launch_instance<A_TRANS_F32, false, 128>(maps, args, stream);
  if (amode == A_TRANS_SWIGLU_F32)   // the weight gradient of W_down (+ dW)
    return resid ? launch_instance<A_TRANS_SWIGLU_F32, true, 128>(maps, args, stream)
                 : launch_instance<A_TRANS_SWIGLU_F32, false, 128>(maps, args, stream);
  if (amode == A_SWIGLU_F32 && resid)
    return launch_instance<A_SWIGLU_F32, true, 128>(maps, args, stream);
  return cudaErrorInvalidValue;
}

}  // namespace lin
