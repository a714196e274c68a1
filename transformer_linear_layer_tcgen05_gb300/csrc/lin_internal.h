// lin_internal.h -- declarations shared by the host API and the kernel
// translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lin {

// How the A operand (the left factor, [M, K]) reaches shared memory.
enum AMode : int {
  A_TMA_F32 = 0,     // X f32 copied by TMA, consumed as TF32
  A_CVT_F16 = 1,     // X f32 staged by TMA, rounded to binary16 by transform warps
  A_SWIGLU_F32 = 2,  // GATE, UP staged by TMA; silu(GATE) * UP written as f32 (TF32 MMA)
  A_SWIGLU_F16 = 3,  // GATE, UP staged by TMA; silu(GATE) * UP rounded to binary16
};

enum : uint32_t {
  // Self-test only: the TMA producers issue nothing, so every consumer wait
  // must run out and the kernel must leave through its timeout path.
  KFLAG_WITHHOLD_PRODUCER = 1u << 0,
};

// Device status word values (mirror lin_status).
enum : int { KSTATUS_OK = 0, KSTATUS_TIMEOUT = 7 };

struct KernelArgs {
  int32_t M, N, K;
  uint32_t flags;
  uint64_t timeout_ns;  // limit for any single wait inside the kernel
  int* status;          // device status word (first failure wins)
  const float* A;       // X or GATE [M, K] (kernels that load it directly)
  const float* U;       // UP [M, K] (SwiGLU forms, kernels that load it directly)
  const float* R;       // residual [M, N] (kernels that read it directly)
  float* Y;             // output [M, N] (kernels that write it directly)
};

// Tensor maps of one call. `a` is X (A_TMA_F32 / A_CVT_F16) or GATE, `u` is
// UP (SwiGLU forms only), `w` the weights, `r` the residual, `y` the output.
struct TensorMaps {
  CUtensorMap a, u, w, r, y;
};

// Block-tile geometry shared by host and device.
constexpr int kBM = 128;           // rows of the output tile (UMMA M)
constexpr int kThreads = 256;      // 8 warps
constexpr int kEpiRows = 32;       // rows per epilogue warp (one TMEM lane quadrant)
constexpr int kEpiCols = 32;       // columns per epilogue chunk (128 bytes of f32)

// Launchers, one per translation unit family. `bn` is the tile width (128 or
// 256). They set the shared-memory attribute on first use and launch a grid
// of (ceil(N/bn), ceil(M/128)) CTAs.
cudaError_t launch_gemm_tf32(int amode, bool resid, int bn, const TensorMaps& maps,
                             const KernelArgs& args, cudaStream_t stream);
cudaError_t launch_gemm_f16(int amode, bool resid, int bn, const TensorMaps& maps,
                            const KernelArgs& args, cudaStream_t stream);

// Clustered persistent kernels for the binary16-weight forms: a cluster of
// `cn` CTAs along N shares the on-chip A operand (128/cn rows each). They
// read X (or GATE and UP) through KernelArgs::A/U and W through its tensor
// map; R and Y through KernelArgs.
constexpr int kClusterBN = 256;
cudaError_t launch_gemm_cluster_swiglu(int cn, const TensorMaps& maps, const KernelArgs& args,
                                       cudaStream_t stream);
cudaError_t launch_gemm_cluster_cvt(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream);

}  // namespace lin
