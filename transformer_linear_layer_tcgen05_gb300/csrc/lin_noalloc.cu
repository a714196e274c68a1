// lin_noalloc.cu -- lin_matmul_residual_swiglu_a_w16_noalloc: the binary16
// SwiGLU form with the workspace of its split tail in a static device array,
// so that the call allocates no device memory.
//
// The array lives in this translation unit's own module: a process that
// never calls this entry point never loads it (with CUDA's lazy module
// loading) and never pays for its memory.
#include <mutex>

#include "lin_internal.h"

namespace {

// One f32 partial tile of 128 x 256 per CTA of every cluster of the split
// round at most: 128 KiB per SM, for the 152 SMs of a GB300.
constexpr size_t kNoallocWorkspaceBytes = size_t{152} * 128 * 1024;
constexpr int kMaxDevices = 64;

struct NoallocDevice {
  std::once_flag once;
  cudaError_t error = cudaSuccess;
  void* base = nullptr;
};
NoallocDevice g_noalloc_devices[kMaxDevices];

}  // namespace

// Nothing in it needs to start at zero: a call writes every byte it reads
// before reading it.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoallocWorkspaceBytes];

namespace {

// Base and size of the array on device `dev`; its address is looked up
// once per device (the first call that passes validation).
lin_status noalloc_workspace(int dev, void** ptr, size_t* bytes) {
  if (dev < 0 || dev >= kMaxDevices) return LIN_ERROR_UNSUPPORTED_DEVICE;
  NoallocDevice& d = g_noalloc_devices[dev];
  std::call_once(d.once, [&] {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) {
      d.error = e;
      cudaGetLastError();
      return;
    }
    d.base = p;
  });
  if (d.error != cudaSuccess) return lin_detail::record_cuda_error(d.error);
  *ptr = d.base;
  *bytes = kNoallocWorkspaceBytes;
  return LIN_SUCCESS;
}

}  // namespace

extern "C" lin_status lin_matmul_residual_swiglu_a_w16_noalloc(
    const float* GATE, const float* UP, const uint16_t* W16, const float* R, float* Y, int64_t M,
    int64_t N, int64_t K, lin_stream_t stream) {
  return lin_detail::run_swiglu_w16_fixed(GATE, UP, W16, R, Y, M, N, K,
                                          reinterpret_cast<cudaStream_t>(stream),
                                          noalloc_workspace);
}
