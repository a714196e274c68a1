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

// The array's address on one device, and the context it belongs to: the
// address is valid only while that context lives (a cudaDeviceReset ends it;
// the next context loads the module again, possibly elsewhere).
struct NoallocDevice {
  std::mutex mu;
  unsigned long long ctx_id = 0;   // unique id of that context; 0: none yet
  void* base = nullptr;
};
NoallocDevice g_noalloc_devices[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id (cuCtxGetId: never reused within a process) of the calling
// thread's current context, or 0 when it cannot be told.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  CUcontext c = nullptr;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

}  // namespace

// Nothing in it needs to start at zero: a call writes every byte it reads
// before reading it.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoallocWorkspaceBytes];

namespace {

// Base and size of the array on device `dev` (current). The address is
// looked up on the first call that passes validation and again whenever the
// device's context has changed since (or cannot be identified); a failed
// look-up is not remembered, so the next call tries again.
lin_status noalloc_workspace(int dev, void** ptr, size_t* bytes) {
  if (dev < 0 || dev >= kMaxDevices) return LIN_ERROR_UNSUPPORTED_DEVICE;
  NoallocDevice& d = g_noalloc_devices[dev];
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(d.mu);
  if (!d.base || ctx == 0 || ctx != d.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) {
      cudaGetLastError();
      d.base = nullptr;
      d.ctx_id = 0;
      return lin_detail::record_cuda_error(e);
    }
    d.base = p;
    d.ctx_id = ctx;
  }
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
