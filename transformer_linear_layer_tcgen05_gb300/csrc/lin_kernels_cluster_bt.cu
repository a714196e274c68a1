// lin_kernels_cluster_bt.cu -- instantiations of the clustered persistent
// GEMM for the transposed product dY · W^T with binary16 W
// (lin_matmul_t_w16 and its accumulating form): W is read as [N][K], a
// K-major B operand; A = dY is rounded to binary16 by the transform warps or
// by the pre-pass and then copied by TMA (single CTAs or CTA pairs).
#include "lin_gemm_cluster.cuh"

namespace lin {

template <int AMODE, bool RESID, int CN>
using BtLaunch = ClusterLaunch<AMODE, RESID, 256, CN, /*BT=*/true>;

// The rounded-by-the-transform form in clusters of 1, 2 or 4 CTAs along N;
// the pre-converted form (TMA-loaded A) in single CTAs or CTA pairs (cn 2).
template <int AMODE>
cudaError_t bt_launch(int cn, bool resid, const TensorMaps& m, const KernelArgs& a,
                      cudaStream_t s) {
  if (cn == 1) return resid ? BtLaunch<AMODE, true, 1>::launch(m, a, s)
                            : BtLaunch<AMODE, false, 1>::launch(m, a, s);
  if constexpr (AMODE == A_TMA_F16) {
    if (cn != 2) return cudaErrorInvalidValue;
    return resid ? BtLaunch<AMODE, true, 2>::launch(m, a, s)
                 : BtLaunch<AMODE, false, 2>::launch(m, a, s);
  } else {
    switch (cn * 2 + (resid ? 1 : 0)) {
      case 4: return BtLaunch<AMODE, false, 2>::launch(m, a, s);
      case 5: return BtLaunch<AMODE, true, 2>::launch(m, a, s);
      case 8: return BtLaunch<AMODE, false, 4>::launch(m, a, s);
      case 9: return BtLaunch<AMODE, true, 4>::launch(m, a, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int AMODE>
int bt_capacity(int cn, bool resid, cudaError_t* err) {
  if (cn == 1) return resid ? BtLaunch<AMODE, true, 1>::capacity(err)
                            : BtLaunch<AMODE, false, 1>::capacity(err);
  if constexpr (AMODE == A_TMA_F16) {
    if (cn != 2) {
      *err = cudaErrorInvalidValue;
      return 0;
    }
    return resid ? BtLaunch<AMODE, true, 2>::capacity(err)
                 : BtLaunch<AMODE, false, 2>::capacity(err);
  } else {
    switch (cn * 2 + (resid ? 1 : 0)) {
      case 4: return BtLaunch<AMODE, false, 2>::capacity(err);
      case 5: return BtLaunch<AMODE, true, 2>::capacity(err);
      case 8: return BtLaunch<AMODE, false, 4>::capacity(err);
      case 9: return BtLaunch<AMODE, true, 4>::capacity(err);
      default: *err = cudaErrorInvalidValue; return 0;
    }
  }
}

cudaError_t launch_gemm_cluster_bt(bool tma_a, int cn, bool resid, const TensorMaps& maps,
                                   const KernelArgs& args, cudaStream_t stream) {
  return tma_a ? bt_launch<A_TMA_F16>(cn, resid, maps, args, stream)
               : bt_launch<A_CVT_F16>(cn, resid, maps, args, stream);
}

int cluster_capacity_bt(bool tma_a, int cn, bool resid, cudaError_t* err) {
  return tma_a ? bt_capacity<A_TMA_F16>(cn, resid, err) : bt_capacity<A_CVT_F16>(cn, resid, err);
}

}  // namespace lin
