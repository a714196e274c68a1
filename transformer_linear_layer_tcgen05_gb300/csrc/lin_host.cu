// lin_host.cu -- the forward forms with every operand in host memory
// (lin_*_host): the operands cross to the GPU and the result comes back
// inside the call, in blocks of rows, so that the copies of one block
// overlap the GEMM of another. Host code only; the arithmetic is the device
// entry points' (the same kernels, one call per block).
//
// Three streams, ordered by events:
//
//   copy in   W | in(0) | in(1) | in(2) | in(3) ...     in(c) waits gemm(c - S)
//   caller         gemm(0) | gemm(1) | gemm(2) ...      gemm(c) waits in(c), out(c - S)
//   copy out             out(0) | out(1) | out(2) ...   out(c) waits gemm(c)
//
// with S staging buffers of each kind on the device (one stream-ordered
// allocation from the library's pool, taken and given back on the caller's
// stream). The caller's stream finally waits for the last copy out, so the
// call has the device entry points' stream semantics: it returns once the
// work is enqueued, and Y is complete when the caller's stream gets there.
// With pinned host memory the copies run on the copy engines concurrently
// with the GEMMs; with pageable memory the runtime stages them itself (the
// call is then largely synchronous, with the same results).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "lin.h"
#include "lin_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kStages = 3;                               // staging buffers of each kind
constexpr uint64_t kDefaultBlockBytes = 64ull << 20;     // operand + result bytes per block
std::atomic<uint64_t> g_block_bytes{0};                  // 0: the default

struct CopyStreams {
  std::once_flag once;
  cudaError_t error = cudaSuccess;
  cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_copy_streams[kMaxDevices];

// The two copy streams of device `dev`, created on first use and kept.
cudaError_t copy_streams(int dev, cudaStream_t* in, cudaStream_t* out) {
  CopyStreams& s = g_copy_streams[dev];
  std::call_once(s.once, [&] {
    cudaError_t e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking);
    if (e != cudaSuccess) cudaGetLastError();
    s.error = e;
  });
  *in = s.in;
  *out = s.out;
  return s.error;
}

// Forms as numbered by lin_detail::run_forward_staged.
enum Kind : int { KIND_MATMUL = 0, KIND_RESID = 1, KIND_SWIGLU = 2 };

struct HostProblem {
  Kind kind;
  bool w16;
  const float* X;
  const float* G;
  const float* U;
  const void* W;
  const float* R;
  float* Y;
  int64_t M, N, K;
};

// Host memory: pinned or ordinary pageable, not device or managed memory.
bool is_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

bool overlap(const void* a, uint64_t an, const void* b, uint64_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// The events of one call; destroying a recorded event is safe (its
// resources go once the work it marks is done).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t record(cudaEvent_t* out, cudaStream_t s) {
    cudaEvent_t e = nullptr;
    cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) return r;
    ev.push_back(e);
    *out = e;
    return cudaEventRecord(e, s);
  }
};

uint64_t round_up(uint64_t b) { return (b + 255) & ~uint64_t{255}; }

lin_status run_host(const HostProblem& h, cudaStream_t stream) {
  lin_detail::set_last_launch_info(0, 0);
  // 1. dims, required pointers and shapes (the device entry points' rules)
  if (h.M < 0 || h.N < 0 || h.K < 0) return LIN_ERROR_INVALID_VALUE;
  if (h.M == 0 || h.N == 0) return LIN_SUCCESS;
  const bool resid = h.kind != KIND_MATMUL, swiglu = h.kind == KIND_SWIGLU;
  if (!h.Y || (resid && !h.R)) return LIN_ERROR_INVALID_VALUE;
  if (h.K > 0 && (!h.W || (swiglu ? (!h.G || !h.U) : !h.X))) return LIN_ERROR_INVALID_VALUE;
  lin_status st = lin_detail::forward_shape_status(h.w16, h.M, h.N, h.K);
  if (st != LIN_SUCCESS) return st;
  const uint64_t M = h.M, N = h.N, K = h.K;
  const uint64_t a_bytes = M * K * 4, w_bytes = K * N * (h.w16 ? 2 : 4), mn_bytes = M * N * 4;

  // 2. Y overlaps no input, and every operand is host memory
  if (resid && overlap(h.Y, mn_bytes, h.R, mn_bytes)) return LIN_ERROR_ALIASING;
  if (K > 0) {
    if (overlap(h.Y, mn_bytes, h.W, w_bytes)) return LIN_ERROR_ALIASING;
    if (swiglu ? (overlap(h.Y, mn_bytes, h.G, a_bytes) || overlap(h.Y, mn_bytes, h.U, a_bytes))
               : overlap(h.Y, mn_bytes, h.X, a_bytes))
      return LIN_ERROR_ALIASING;
  }
  const void* host_ops[] = {h.Y, resid ? h.R : nullptr, K ? h.W : nullptr,
                            K ? (swiglu ? h.G : h.X) : nullptr, (K && swiglu) ? h.U : nullptr};
  for (const void* p : host_ops)
    if (p && !is_host(p)) return LIN_ERROR_INVALID_VALUE;

  // 3. device and copy streams (not under stream capture: the call's own
  // copy streams and events would become part of the caller's graph)
  int dev = 0;
  if ((st = lin_detail::checked_device(&dev)) != LIN_SUCCESS) return st;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
  if (ce != cudaSuccess) return lin_detail::record_cuda_error(ce);
  if (cs != cudaStreamCaptureStatusNone) return LIN_ERROR_INVALID_VALUE;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaError_t e = copy_streams(dev, &s_in, &s_out);
  if (e != cudaSuccess) return lin_detail::record_cuda_error(e);

  // 4. blocks of whole 128-row tiles moving about kDefaultBlockBytes each
  const uint64_t row_bytes = (swiglu ? 2 : 1) * K * 4 + (resid ? N * 4 : 0) + N * 4;
  const uint64_t target = g_block_bytes.load(std::memory_order_relaxed);
  uint64_t rows = (target ? target : kDefaultBlockBytes) / row_bytes / 128 * 128;
  rows = std::min<uint64_t>(std::max<uint64_t>(rows, 128), M);
  const uint64_t nblk = (M + rows - 1) / rows;
  const int ns = static_cast<int>(std::min<uint64_t>(kStages, nblk));
  const uint64_t a_blk = round_up(rows * K * 4), r_blk = resid ? round_up(rows * N * 4) : 0,
                 y_blk = round_up(rows * N * 4);
  const uint64_t stage_bytes = a_blk * (swiglu ? 2 : 1) + r_blk + y_blk;
  const uint64_t total = round_up(w_bytes) + ns * stage_bytes;

  // 5. staging memory, in stream order on the caller's stream
  void* base = nullptr;
  cudaMemPool_t pool = lin_detail::device_pool(dev);
  e = pool ? cudaMallocFromPoolAsync(&base, total, pool, stream) : cudaMallocAsync(&base, total, stream);
  if (e != cudaSuccess) return lin_detail::record_cuda_error(e);
  char* const w_dev = static_cast<char*>(base);
  auto stage = [&](uint64_t c) { return w_dev + round_up(w_bytes) + (c % ns) * stage_bytes; };

  Events ev;
  std::vector<cudaEvent_t> in_done(nblk), gemm_done(nblk), out_done(nblk);
  int kernels = 0;
  uint64_t workspace = 0;
  cudaEvent_t start = nullptr;
  e = ev.record(&start, stream);   // the staging memory exists from here on
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, start, 0);
  if (e == cudaSuccess && K > 0)
    e = cudaMemcpyAsync(w_dev, h.W, w_bytes, cudaMemcpyHostToDevice, s_in);
  for (uint64_t c = 0; c < nblk && e == cudaSuccess && st == LIN_SUCCESS; ++c) {
    const uint64_t r0 = c * rows, rc = std::min(rows, M - r0);
    char* a_dev = stage(c);
    char* u_dev = a_dev + a_blk;
    char* r_dev = a_dev + a_blk * (swiglu ? 2 : 1);
    char* y_dev = r_dev + r_blk;
    // copy in: the block's rows of A (or GATE and UP) and R, once the GEMM
    // that last used this stage is done with it
    if (c >= (uint64_t)ns) e = cudaStreamWaitEvent(s_in, gemm_done[c - ns], 0);
    if (e == cudaSuccess && K > 0)
      e = cudaMemcpyAsync(a_dev, (swiglu ? h.G : h.X) + r0 * K, rc * K * 4,
                          cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess && K > 0 && swiglu)
      e = cudaMemcpyAsync(u_dev, h.U + r0 * K, rc * K * 4, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess && resid)
      e = cudaMemcpyAsync(r_dev, h.R + r0 * N, rc * N * 4, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess) e = ev.record(&in_done[c], s_in);
    // the GEMM of the block, once its inputs are in and the copy out of the
    // block that last used this stage's Y has read it
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, in_done[c], 0);
    if (e == cudaSuccess && c >= (uint64_t)ns) e = cudaStreamWaitEvent(stream, out_done[c - ns], 0);
    if (e != cudaSuccess) break;
    st = lin_detail::run_forward_staged(
        h.kind, h.w16, swiglu ? nullptr : reinterpret_cast<const float*>(a_dev),
        swiglu ? reinterpret_cast<const float*>(a_dev) : nullptr,
        swiglu ? reinterpret_cast<const float*>(u_dev) : nullptr, K > 0 ? w_dev : nullptr,
        resid ? reinterpret_cast<const float*>(r_dev) : nullptr, reinterpret_cast<float*>(y_dev),
        (int64_t)rc, h.N, h.K, stream);
    if (st != LIN_SUCCESS) break;
    int k = 0;
    uint64_t ws = 0;
    lin_last_launch_info(&k, &ws);
    kernels += k;
    workspace = std::max(workspace, ws);
    e = ev.record(&gemm_done[c], stream);
    // copy out: the block of Y
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, gemm_done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.Y + r0 * N, y_dev, rc * N * 4, cudaMemcpyDeviceToHost, s_out);
    if (e == cudaSuccess) e = ev.record(&out_done[c], s_out);
  }
  // 6. join both copy streams into the caller's stream (also after a
  // failure: the staging memory is given back only after every copy that
  // was enqueued), then give the memory back
  cudaEvent_t in_end = nullptr, out_end = nullptr;
  cudaError_t j = ev.record(&in_end, s_in);
  if (j == cudaSuccess) j = ev.record(&out_end, s_out);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, in_end, 0);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, out_end, 0);
  if (j == cudaSuccess) j = cudaFreeAsync(base, stream);
  if (st != LIN_SUCCESS) return st;
  if (e == cudaSuccess) e = j;
  if (e != cudaSuccess) return lin_detail::record_cuda_error(e);
  lin_detail::set_last_launch_info(kernels, total + workspace);
  return LIN_SUCCESS;
}

cudaStream_t as_cuda(lin_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

lin_status lin_matmul_host(const float* X, const float* W, float* Y, int64_t M, int64_t N,
                           int64_t K, lin_stream_t stream) {
  return run_host({KIND_MATMUL, false, X, nullptr, nullptr, W, nullptr, Y, M, N, K},
                  as_cuda(stream));
}

lin_status lin_matmul_residual_host(const float* X, const float* W, const float* R, float* Y,
                                    int64_t M, int64_t N, int64_t K, lin_stream_t stream) {
  return run_host({KIND_RESID, false, X, nullptr, nullptr, W, R, Y, M, N, K}, as_cuda(stream));
}

lin_status lin_matmul_residual_swiglu_a_host(const float* GATE, const float* UP, const float* W,
                                             const float* R, float* Y, int64_t M, int64_t N,
                                             int64_t K, lin_stream_t stream) {
  return run_host({KIND_SWIGLU, false, nullptr, GATE, UP, W, R, Y, M, N, K}, as_cuda(stream));
}

lin_status lin_matmul_w16_host(const float* X, const uint16_t* W16, float* Y, int64_t M,
                               int64_t N, int64_t K, lin_stream_t stream) {
  return run_host({KIND_MATMUL, true, X, nullptr, nullptr, W16, nullptr, Y, M, N, K},
                  as_cuda(stream));
}

lin_status lin_matmul_residual_w16_host(const float* X, const uint16_t* W16, const float* R,
                                        float* Y, int64_t M, int64_t N, int64_t K,
                                        lin_stream_t stream) {
  return run_host({KIND_RESID, true, X, nullptr, nullptr, W16, R, Y, M, N, K}, as_cuda(stream));
}

lin_status lin_matmul_residual_swiglu_a_w16_host(const float* GATE, const float* UP,
                                                 const uint16_t* W16, const float* R, float* Y,
                                                 int64_t M, int64_t N, int64_t K,
                                                 lin_stream_t stream) {
  return run_host({KIND_SWIGLU, true, nullptr, GATE, UP, W16, R, Y, M, N, K}, as_cuda(stream));
}

lin_status lin_set_host_block_bytes(uint64_t bytes) {
  if (bytes != 0 && bytes < (1ull << 16)) return LIN_ERROR_INVALID_VALUE;
  g_block_bytes.store(bytes, std::memory_order_relaxed);
  return LIN_SUCCESS;
}

}  // extern "C"
