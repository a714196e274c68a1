// lin_kernels_cluster_dual.cu -- instantiations of the clustered persistent
// GEMM for the FFN's gate and up projections in one launch (lin_gate_up_w16):
// GATE = X @ W_gate and UP = X @ W_up from one read and one binary16
// rounding of X (by the transform warps, or by the pre-pass and then TMA).
#include "lin_gemm_cluster.cuh"

namespace lin {

template <int AMODE, int CN>
using DualLaunch = ClusterLaunch<AMODE, false, 256, CN, /*BT=*/false, /*DUAL=*/true>;

// The rounded-by-the-transform form in clusters of 1, 2 or 4 CTAs along N;
// the pre-converted form (TMA-loaded A) in single CTAs or CTA pairs (cn 2;
// the even CTA loads the W tile, the odd one the W2 tile).
template <int AMODE>
cudaError_t dual_launch(int cn, const TensorMaps& m, const KernelArgs& a, cudaStream_t s) {
  if (cn == 1) return DualLaunch<AMODE, 1>::launch(m, a, s);
  if constexpr (AMODE == A_TMA_F16) {
    return cn == 2 ? DualLaunch<AMODE, 2>::launch(m, a, s) : cudaErrorInvalidValue;
  } else {
    switch (cn) {
      case 2: return DualLaunch<AMODE, 2>::launch(m, a, s);
      case 4: return DualLaunch<AMODE, 4>::launch(m, a, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int AMODE>
int dual_capacity(int cn, cudaError_t* err) {
  if (cn == 1) return DualLaunch<AMODE, 1>::capacity(err);
  if constexpr (AMODE == A_TMA_F16) {
    if (cn == 2) return DualLaunch<AMODE, 2>::capacity(err);
    *err = cudaErrorInvalidValue;
    return 0;
  } else {
    switch (cn) {
      case 2: return DualLaunch<AMODE, 2>::capacity(err);
      case 4: return DualLaunch<AMODE, 4>::capacity(err);
      default: *err = cudaErrorInvalidValue; return 0;
    }
  }
}

cudaError_t launch_gemm_cluster_dual(bool tma_a, int cn, const TensorMaps& maps,
                                     const KernelArgs& args, cudaStream_t stream) {
  return tma_a ? dual_launch<A_TMA_F16>(cn, maps, args, stream)
               : dual_launch<A_CVT_F16>(cn, maps, args, stream);
}

int cluster_capacity_dual(bool tma_a, int cn, cudaError_t* err) {
  return tma_a ? dual_capacity<A_TMA_F16>(cn, err) : dual_capacity<A_CVT_F16>(cn, err);
}

}  // namespace lin
