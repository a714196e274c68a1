// lin_api.cu -- the C ABI of include/lin.h: argument validation, tensor-map
// encoding, the workspace of split launches and kernel launch. No host<->device
// copies on the compute path; every operation runs in the library's kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "lin.h"
#include "lin_internal.h"

namespace lin_detail {

// Per-device status record written by kernels whose bounded waits ran out
// or (checked build) whose device checks failed: [status, check site, check
// value as int64].
__device__ __align__(16) int g_status_word[4];

constexpr uint64_t kDefaultTimeoutNs = 1000ull * 1000ull * 1000ull;   // 1 s per wait
constexpr int kMaxDevices = 64;

thread_local int t_last_cuda_error = 0;
thread_local int t_last_check_site = 0;         // lin_last_device_check
thread_local int64_t t_last_check_value = 0;
thread_local int t_last_kernels = 0;            // lin_last_launch_info
thread_local uint64_t t_last_workspace = 0;

lin_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  cudaGetLastError();   // clear the sticky-free error so later calls start clean
  return LIN_ERROR_CUDA;
}

// Driver entry points, fetched through the runtime so the library does not
// link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

struct Driver {
  EncodeTiledFn encode = nullptr;
  AddressRangeFn range = nullptr;
};

const Driver& driver() {
  static Driver d;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.encode = reinterpret_cast<EncodeTiledFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.range = reinterpret_cast<AddressRangeFn>(p);
    cudaGetLastError();
  });
  return d;
}

struct DeviceState {
  std::once_flag once;
  lin_status status = LIN_SUCCESS;
  int cuda_error = 0;
  int* status_word = nullptr;
  std::once_flag pool_once;
  cudaMemPool_t pool = nullptr;   // workspace of split launches (stream-ordered)
};
DeviceState g_devices[kMaxDevices];

// The library's own memory pool on device `dev`, created on first use, that
// keeps freed workspace for reuse (it never trims itself); null if the pool
// cannot be created.
cudaMemPool_t workspace_pool(int dev) {
  DeviceState& s = g_devices[dev];
  std::call_once(s.pool_once, [&] {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    uint64_t keep = UINT64_MAX;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
      cudaGetLastError();
    s.pool = pool;
  });
  return s.pool;
}

// Checks the current device once (sm_103, driver entry points, status word).
// SMs of device `dev` (queried once per device).
int sm_count(int dev) {
  static std::atomic<int> counts[kMaxDevices];
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

lin_status current_device(int* dev_out, int** status_word) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return LIN_ERROR_UNSUPPORTED_DEVICE;
  DeviceState& s = g_devices[dev];
  std::call_once(s.once, [&] {
    int major = 0, minor = 0;
    cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      s.status = LIN_ERROR_CUDA;
      s.cuda_error = static_cast<int>(e1 != cudaSuccess ? e1 : e2);
      cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) {
      s.status = LIN_ERROR_UNSUPPORTED_DEVICE;
      return;
    }
    const Driver& d = driver();
    if (!d.encode || !d.range) {
      s.status = LIN_ERROR_CUDA;
      s.cuda_error = static_cast<int>(cudaErrorSymbolNotFound);
      return;
    }
    void* p = nullptr;
    cudaError_t e3 = cudaGetSymbolAddress(&p, g_status_word);
    if (e3 != cudaSuccess) {
      s.status = LIN_ERROR_CUDA;
      s.cuda_error = static_cast<int>(e3);
      cudaGetLastError();
      return;
    }
    s.status_word = static_cast<int*>(p);
  });
  if (s.status == LIN_ERROR_CUDA) t_last_cuda_error = s.cuda_error;
  if (s.status != LIN_SUCCESS) return s.status;
  *dev_out = dev;
  *status_word = s.status_word;
  return LIN_SUCCESS;
}

// The buffer [p, p + bytes) must be device (or managed) memory of `dev`
// lying inside one allocation.
lin_status check_buffer(const void* p, uint64_t bytes, int dev) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LIN_ERROR_INVALID_VALUE;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return LIN_ERROR_INVALID_VALUE;
  if (a.device != dev) return LIN_ERROR_INVALID_VALUE;
  CUdeviceptr base = 0;
  size_t size = 0;
  if (driver().range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
    return LIN_ERROR_INVALID_VALUE;
  const uint64_t off = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(p)) - base;
  if (off > size || bytes > size - off) return LIN_ERROR_INVALID_VALUE;
  return LIN_SUCCESS;
}

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  if (!a || !b || abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// 2-D row-major tensor map with the 128-byte swizzle (16-byte atoms, or
// 32-byte atoms for an MN-major TF32 operand); out-of-range elements of a
// load read as zero.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols,
               uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return driver().encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Cluster size of the binary16 kernels: enough CTAs along N to share the
// transformed A operand, within what N can use. LIN_F16_KERNEL overrides it
// for measurements: "tile" selects the per-tile kernel, "1", "2" or "4" a
// cluster size.
int f16_forced_kernel() {
  static const int forced = [] {
    const char* v = std::getenv("LIN_F16_KERNEL");
    if (!v) return -1;
    if (std::strcmp(v, "tile") == 0) return 0;
    const int c = std::atoi(v);
    return (c == 1 || c == 2 || c == 4) ? c : -1;
  }();
  return forced;
}

int f16_cluster_size(uint64_t N) {
  const int forced = f16_forced_kernel();
  if (forced >= 0) return forced;
  // Clusters of 4 leave 8 of 152 SMs idle but transform each A row half as
  // often as pairs; with the transform warps taking turns by k-block they
  // measured fastest on the 16k-token SwiGLU down projection (4 > 2 > 1) and
  // level with the others on the 512-token vocabulary projection.
  const uint64_t per = (uint64_t)lin::kClusterBN;
  return N >= 4 * per ? 4 : (N >= 2 * per ? 2 : 1);
}

// Whether matmul_w16 / matmul_residual_w16 round X to binary16 in a
// pre-pass and feed the clustered kernel by TMA: by default when a row block
// spans several cluster tiles along N (each would otherwise transform the
// same rows again). LIN_F16_PRECONVERT=0 / 1 forces it off / on
// (measurements).
bool f16_preconvert(int num_ng) {
  static const int forced = [] {
    const char* v = std::getenv("LIN_F16_PRECONVERT");
    if (!v) return -1;
    return std::strcmp(v, "0") == 0 ? 0 : (std::strcmp(v, "1") == 0 ? 1 : -1);
  }();
  if (forced >= 0) return forced == 1;
  return num_ng >= 2;
}

// Whether the pre-converted forms (binary16 A copied by TMA) run as CTA
// pairs along M -- one UMMA of M = 256 over two CTAs (tcgen05
// .cta_group::2), each CTA loading half of the tile's W columns -- rather
// than single CTAs: when the 256-row tiles make at least two rounds over the
// SMs' pairs. Measured (cold / warm us, single CTAs -> pairs): the 16k-token
// dX 405 / 396 -> 371 / 364, the 16k-token gate/up pair 821 -> 723; on the
// 512-token shapes (under two rounds) no gain: lm_head_w16 18.95 -> 19.14
// warm. LIN_F16_PAIR=0 / 1 forces it off / on (measurements).
bool f16_pair(long long pair_tiles, int sms) {
  static const int forced = [] {
    const char* v = std::getenv("LIN_F16_PAIR");
    if (!v) return -1;
    return std::strcmp(v, "0") == 0 ? 0 : (std::strcmp(v, "1") == 0 ? 1 : -1);
  }();
  if (forced >= 0) return forced == 1;
  return pair_tiles >= (long long)sms;
}

// Tile width of the per-tile kernel for the forward f32 SwiGLU form, whose
// transform warps build each row block's A once per column tile: 256
// columns (half the rebuilds) when N spans more than one such tile, else
// 128. Measured on 512 x 768 x 3072 (cold / warm us): 30.4 / 22.5 with 128,
// 25.3 / 17.2 with 256. LIN_F32_SWIGLU_BN=128 / 256 forces it
// (measurements).
int f32_swiglu_bn(uint64_t N) {
  static const int forced = [] {
    const char* v = std::getenv("LIN_F32_SWIGLU_BN");
    if (!v) return -1;
    return std::strcmp(v, "128") == 0 ? 128 : (std::strcmp(v, "256") == 0 ? 256 : -1);
  }();
  if (forced > 0) return forced;
  return N > 256 ? 256 : 128;
}

// Tile width of the per-tile kernel for the f32 forms that copy X (or dY) as
// is (matmul, matmul_residual, and matmul_t, whose W tile is K-major), for
// the 512-token shapes: where 128-column tiles leave the SMs to a K split,
// 96 columns (a smaller split, a smaller partial tile to sum) when the
// contraction is short (at most 32 k-blocks), else 128 (the longer K
// ranges of the smaller split cost more than the sum saves); where they do
// not split, 96 columns while the 96-column tiles fit one wave (more SMs
// busy). Measured on one GB300 (warm µs, 128 -> 96 columns):
// attn_proj_f32 7.46 -> 7.14 and attn_proj_dx_f32 7.44 -> 7.11 (contraction
// 768, split 6 -> 4), ffn_up_dx_f32 12.3 -> 12.85 (contraction 3072: kept at
// 128), ffn_up_residual_f32 12.8 -> 12.25 (no split; 96 -> 128 tiles).
// LIN_F32_BN=96 / 128 forces it (measurements).
int f32_x_bn(uint64_t M, uint64_t N, uint64_t K, int sms) {
  static const int forced = [] {
    const char* v = std::getenv("LIN_F32_BN");
    if (!v) return -1;
    return std::strcmp(v, "96") == 0 ? 96 : (std::strcmp(v, "128") == 0 ? 128 : -1);
  }();
  if (forced > 0) return forced;
  const uint64_t rows = (M + lin::kBM - 1) / lin::kBM;
  const uint64_t t96 = rows * ((N + 95) / 96), t128 = rows * ((N + 127) / 128);
  const uint64_t nkb = (K + 31) / 32;
  if (t96 > (uint64_t)sms) return 128;
  const uint64_t split128 = std::min<uint64_t>((uint64_t)sms / t128, nkb / 4);
  if (split128 >= 2) return nkb <= 32 ? 96 : 128;
  return 96;
}

enum Form : int { F_MATMUL = 0, F_RESID = 1, F_SWIGLU = 2 };

// In the kernels' terms: Y[M,N] = A[M,K] · B[K,N] (+ R), A = X or
// silu(G)·U. B = W [K,N], or, for the transposed product (bt), W given as
// [N][K] (the backward dX = dY · W^T: X = dY, N = the output columns).
struct Problem {
  Form form;
  bool w16;
  const float* X;      // matmul / residual forms
  const float* G;      // SwiGLU forms
  const float* U;
  const void* W;       // float or binary16 bits
  const float* R;
  float* Y;
  int64_t M, N, K;
  bool bt = false;     // W is [N][K]
  bool at = false;     // A = X^T: X is [K][M] (the weight gradient X^T · dY, W = dY)
  bool acc = false;    // R is Y itself (Y += A · B)
  // SwiGLU backward epilogue: Y = dGATE, Y2 = dUP of the product dA, from
  // G2 = GATE and U2 = UP, all [M,N]
  const float* G2 = nullptr;
  const float* U2 = nullptr;
  float* Y2 = nullptr;
  // online-softmax partials of every output row (clustered kernel, no split)
  float4* row_stats = nullptr;
  int stats_cols = 0;
  uint32_t* zero_word = nullptr;   // the clustered GEMM zeroes it (a dependent kernel's counter)
  // dual GEMM: Y2 = A · W2 beside Y = A · W (binary16 W2 [K,N]; Y2 [M,N])
  const void* W2 = nullptr;
  // every buffer is a piece of one of the library's own device allocations
  // (the host-operand entry points' staging): step 6 is skipped
  bool staged = false;
};

// `fixed`: where a split tail's workspace comes from instead of the library's
// pool (null for the ordinary entry points); it is resolved once validation
// has passed and reports its base address and size.
lin_status run(const Problem& p, cudaStream_t stream, lin::WorkspaceGetter fixed = nullptr) {
  t_last_kernels = 0;
  t_last_workspace = 0;
  // 1. dims and required pointers
  if (p.M < 0 || p.N < 0 || p.K < 0) return LIN_ERROR_INVALID_VALUE;
  if (p.M == 0 || p.N == 0) return LIN_SUCCESS;
  // an R operand: the forward residual forms, and every accumulating form
  const bool resid = p.acc || p.form == F_RESID || (p.form == F_SWIGLU && !p.at);
  const bool swiglu = p.form == F_SWIGLU;
  if (!p.Y || (resid && !p.R)) return LIN_ERROR_INVALID_VALUE;
  if (p.K > 0 && (!p.W || (swiglu ? (!p.G || !p.U) : !p.X))) return LIN_ERROR_INVALID_VALUE;

  // 2. shapes
  const int64_t kMax = 0x7fffffffLL;
  if (p.M > kMax || p.N > kMax || p.K > kMax) return LIN_ERROR_UNSUPPORTED_SHAPE;
  // row strides of the row-major operands: whole 16-byte units (A^T's rows
  // are M long; its contraction K then needs no rule)
  if ((p.at ? p.M : p.K) % 4 != 0 || p.N % 4 != 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
  // binary16 W rows must be whole 16-byte units for TMA
  if (p.w16 && (p.bt ? p.K : p.N) % 8 != 0) return LIN_ERROR_UNSUPPORTED_SHAPE;

  const uint64_t M = p.M, N = p.N, K = p.K;
  const uint64_t a_bytes = M * K * 4, w_bytes = K * N * (p.w16 ? 2 : 4), mn_bytes = M * N * 4;

  // 3. alignment (16 bytes: TMA base addresses and vector accesses)
  auto misaligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
  if (misaligned(p.Y) || (resid && misaligned(p.R))) return LIN_ERROR_MISALIGNED;
  if (K > 0 && (misaligned(p.W) || (swiglu ? (misaligned(p.G) || misaligned(p.U))
                                           : misaligned(p.X))))
    return LIN_ERROR_MISALIGNED;

  const bool dual = p.W2 != nullptr;
  if (dual) {   // a second binary16 weight matrix and a second output
    if (!p.w16 || !p.Y2 || resid || p.bt || p.at || swiglu) return LIN_ERROR_INVALID_VALUE;
    if (misaligned(p.Y2) || (K > 0 && misaligned(p.W2))) return LIN_ERROR_MISALIGNED;
    if (overlaps(p.Y2, mn_bytes, p.Y, mn_bytes) || overlaps(p.Y2, mn_bytes, p.X, a_bytes) ||
        overlaps(p.Y2, mn_bytes, p.W, w_bytes) || overlaps(p.Y2, mn_bytes, p.W2, w_bytes) ||
        overlaps(p.Y, mn_bytes, p.W2, w_bytes))
      return LIN_ERROR_ALIASING;
  }
  const bool swb = p.Y2 != nullptr && !dual;
  if (swb) {
    if (!p.G2 || !p.U2 || resid) return LIN_ERROR_INVALID_VALUE;
    if (misaligned(p.G2) || misaligned(p.U2) || misaligned(p.Y2)) return LIN_ERROR_MISALIGNED;
    // both outputs overlap nothing: each other, GATE, UP, or the inputs below
    const void* ins[] = {p.Y2, p.G2, p.U2};
    for (const void* q : ins)
      if (overlaps(p.Y, mn_bytes, q, mn_bytes)) return LIN_ERROR_ALIASING;
    if (overlaps(p.Y2, mn_bytes, p.G2, mn_bytes) || overlaps(p.Y2, mn_bytes, p.U2, mn_bytes))
      return LIN_ERROR_ALIASING;
    if (K > 0 && (overlaps(p.Y2, mn_bytes, p.W, w_bytes) || overlaps(p.Y2, mn_bytes, p.X, a_bytes)))
      return LIN_ERROR_ALIASING;
  }

  // 4. aliasing: Y may overlap no input (an accumulating call reads and
  // writes the same Y, element by element)
  if (resid && !p.acc && overlaps(p.Y, mn_bytes, p.R, mn_bytes)) return LIN_ERROR_ALIASING;
  if (K > 0) {
    if (overlaps(p.Y, mn_bytes, p.W, w_bytes)) return LIN_ERROR_ALIASING;
    if (swiglu) {
      if (overlaps(p.Y, mn_bytes, p.G, a_bytes) || overlaps(p.Y, mn_bytes, p.U, a_bytes))
        return LIN_ERROR_ALIASING;
    } else if (overlaps(p.Y, mn_bytes, p.X, a_bytes)) {
      return LIN_ERROR_ALIASING;
    }
  }

  // 5. device
  int dev = 0;
  int* status_word = nullptr;
  lin_status st = current_device(&dev, &status_word);
  if (st != LIN_SUCCESS) return st;

  // 6. every buffer is device memory of this device and large enough
  if (!p.staged && (st = check_buffer(p.Y, mn_bytes, dev)) != LIN_SUCCESS) return st;
  if (!p.staged && resid && (st = check_buffer(p.R, mn_bytes, dev)) != LIN_SUCCESS) return st;
  if (dual) {
    if ((st = check_buffer(p.Y2, mn_bytes, dev)) != LIN_SUCCESS) return st;
    if (K > 0 && (st = check_buffer(p.W2, w_bytes, dev)) != LIN_SUCCESS) return st;
  }
  if (swb) {
    if ((st = check_buffer(p.Y2, mn_bytes, dev)) != LIN_SUCCESS) return st;
    if ((st = check_buffer(p.G2, mn_bytes, dev)) != LIN_SUCCESS) return st;
    if ((st = check_buffer(p.U2, mn_bytes, dev)) != LIN_SUCCESS) return st;
  }
  if (K > 0 && !p.staged) {
    if ((st = check_buffer(p.W, w_bytes, dev)) != LIN_SUCCESS) return st;
    if (swiglu) {
      if ((st = check_buffer(p.G, a_bytes, dev)) != LIN_SUCCESS) return st;
      if ((st = check_buffer(p.U, a_bytes, dev)) != LIN_SUCCESS) return st;
    } else if ((st = check_buffer(p.X, a_bytes, dev)) != LIN_SUCCESS) {
      return st;
    }
  }

  // 6b. a caller-provided workspace (its set-up runs on the first valid call)
  void* fixed_ptr = nullptr;
  size_t fixed_bytes = 0;
  if (fixed && (st = fixed(dev, &fixed_ptr, &fixed_bytes)) != LIN_SUCCESS) return st;

  // 7. K == 0: nothing is accumulated, Y = R (or 0)
  if (K == 0) {   // nothing to accumulate: Y = R (already so when accumulating in place), or 0
    cudaError_t e = cudaSuccess;
    if (swb || dual) {   // both outputs 0 (for swb: nan_guard maps a NaN product to 0 too)
      e = cudaMemsetAsync(p.Y, 0, mn_bytes, stream);
      if (e == cudaSuccess) e = cudaMemsetAsync(p.Y2, 0, mn_bytes, stream);
    } else if (!resid)
      e = cudaMemsetAsync(p.Y, 0, mn_bytes, stream);
    else if (p.R != p.Y)
      e = cudaMemcpyAsync(p.Y, p.R, mn_bytes, cudaMemcpyDeviceToDevice, stream);
    return e == cudaSuccess ? LIN_SUCCESS : cuda_fail(e);
  }

  // 8. tensor maps and launch
  const int bn = (swiglu && !p.w16 && !p.at && !p.bt) ? f32_swiglu_bn(N)
                 : (!swiglu && !p.w16 && !p.at) ? f32_x_bn(M, N, K, sm_count(dev))
                                                         : 128;
  int cn = (p.w16 && !p.at) ? f16_cluster_size(N) : 0;   // 0: the per-tile kernel
  // the row partials and the dual product exist in the clustered kernel only
  if ((p.row_stats || p.W2) && cn == 0) cn = 1;
  lin::TensorMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  bool ok = true;
  const float* a_src = swiglu ? p.G : p.X;
  if (p.at) {   // X^T: X is [K rows][M] in [32 x 32] boxes
    if (swiglu) {   // GATE, UP: transformed and transposed on chip
      ok &= encode_2d(&maps.a, f32, a_src, M, K, M * 4, 32, 32);
      ok &= encode_2d(&maps.u, f32, p.U, M, K, M * 4, 32, 32);
    } else {        // X: an MN-major TF32 operand as it is (32-byte atoms)
      ok &= encode_2d(&maps.a, f32, a_src, M, K, M * 4, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
    }
  } else if (cn == 0) {   // the clustered kernels load X / GATE / UP without tensor maps
    ok &= encode_2d(&maps.a, f32, a_src, K, M, K * 4, 32, lin::kBM);
    if (swiglu) ok &= encode_2d(&maps.u, f32, p.U, K, M, K * 4, 32, lin::kBM);
  }
  if (p.bt) {   // W as [N][K]: boxes of one k-block by the tile's rows
    if (p.w16)
      ok &= encode_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W, K, N, K * 2, 64,
                      cn > 0 ? (uint32_t)lin::kClusterBN : (uint32_t)bn);
    else
      ok &= encode_2d(&maps.w, f32, p.W, K, N, K * 4, 32, (uint32_t)bn);
  } else if (p.w16) {
    ok &= encode_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W, N, K, N * 2, 64, 64);
    if (dual) {
      ok &= encode_2d(&maps.w2, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W2, N, K, N * 2, 64, 64);
      ok &= encode_2d(&maps.y2, f32, p.Y2, N, M, N * 4, lin::kEpiCols, lin::kEpiRows);
    }
  } else {   // W [K,N] f32: an MN-major TF32 operand, 128-byte swizzle with 32-byte atoms
    ok &= encode_2d(&maps.w, f32, p.W, N, K, N * 4, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
  }
  if (resid) ok &= encode_2d(&maps.r, f32, p.R, N, M, N * 4, lin::kEpiCols, lin::kEpiRows);
  ok &= encode_2d(&maps.y, f32, p.Y, N, M, N * 4, lin::kEpiCols, lin::kEpiRows);
  if (swb) {   // the SwiGLU-backward epilogue's GATE, UP in and dGATE, dUP out:
    // [32 x 32] boxes (per-tile kernel), or [32 rows x 16] with the 64-byte
    // swizzle (clustered kernel, four tiles per warp)
    const uint32_t sc = cn > 0 ? (uint32_t)lin::kSwbCols : (uint32_t)lin::kEpiCols;
    const CUtensorMapSwizzle sz = cn > 0 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    ok &= encode_2d(&maps.g2, f32, p.G2, N, M, N * 4, sc, lin::kEpiRows, sz);
    ok &= encode_2d(&maps.u2, f32, p.U2, N, M, N * 4, sc, lin::kEpiRows, sz);
    ok &= encode_2d(&maps.y2, f32, p.Y2, N, M, N * 4, sc, lin::kEpiRows, sz);
    ok &= encode_2d(&maps.y, f32, p.Y, N, M, N * 4, sc, lin::kEpiRows, sz);
  }
  if (!ok) return cuda_fail(cudaErrorInvalidValue);

  lin::KernelArgs args{};
  args.M = static_cast<int32_t>(M);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  args.flags = 0;
  args.timeout_ns = kDefaultTimeoutNs;
  args.status = status_word;
  args.A = a_src;
  args.U = swiglu ? p.U : nullptr;
  args.R = resid ? p.R : nullptr;
  args.Y = p.Y;
  args.split_r = 0;
  args.split_rem = 0;
  args.split_s = 1;
  // 32-byte loads of the A-side inputs when every row start allows them
  auto align32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
  if (cn > 0 && K % 8 == 0 && align32(a_src) && (!swiglu || align32(p.U)))
    args.flags |= lin::KFLAG_A_V8;
  if (p.row_stats) {
    args.flags |= lin::KFLAG_ROW_STATS;
    args.row_stats = p.row_stats;
    args.zero_word = p.zero_word;
    args.stats_cols = p.stats_cols;
  }
  if (swb) {
    args.flags |= lin::KFLAG_SWIGLU_BWD;
    args.G2 = p.G2;
    args.U2 = p.U2;
    args.Y2 = p.Y2;
  }

  // Workspace for f32 partial tiles of a split (either kernel): the caller's
  // fixed workspace, or a stream-ordered allocation freed on the same stream
  // after the launch -- from the library's pool, or, while the stream is
  // being captured into a graph, a graph memory node (cudaMallocAsync), so
  // that each graph owns its workspace. 1: got it; 0: run unsplit (no memory
  // to be had); -1: the fixed workspace is too small (the call is rejected).
  void* ws = nullptr;           // pool allocation to free
  uint64_t workspace = 0;       // pool bytes taken
  auto take_workspace = [&](size_t bytes) -> int {
    if (fixed) {
      if (bytes > fixed_bytes) return -1;
      args.part = static_cast<float*>(fixed_ptr);
      return 1;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (cs != cudaStreamCaptureStatusNone) {
      if (cs != cudaStreamCaptureStatusActive || cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        ws = nullptr;
        return 0;
      }
      args.part = static_cast<float*>(ws);
      workspace = bytes;
      return 1;
    }
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool || cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) {
      cudaGetLastError();
      ws = nullptr;
      return 0;
    }
    args.part = static_cast<float*>(ws);
    workspace = bytes;
    return 1;
  };

  cudaError_t e;
  int kernels = 1;
  if (cn > 0) {
    // Persistent launch: split the K range of the last partial round when
    // that keeps idle clusters busy.
    cudaError_t ce = cudaSuccess;
    const int num_ng = (int)((N + (uint64_t)lin::kClusterBN * cn - 1) / ((uint64_t)lin::kClusterBN * cn));
    const int nkb = (int)((K + 63) / 64);
    // binary16 X from a pre-pass, in the workspace after the partial tiles
    bool tma_a = !swiglu && !fixed && K % 8 == 0 && f16_preconvert(num_ng);
    // With A already binary16 in global memory a CTA copies its own A tiles
    // by TMA and has nothing to share along N: single CTAs on every SM (152
    // rather than 144 in clusters of four) measured faster at every shape
    // than clusters along N (the 16k-token dX 447 -> 417 us, the gate/up
    // pair 868 -> 821 us, the 512-token dX 39.1 -> 35.6 us), and CTA pairs
    // along M, sharing the W tile between two SMs, faster again. Clusters
    // along N stay for the forms whose A is built on chip; a forced cluster
    // size applies to those only.
    bool pair = false;
    if (tma_a) {
      const long long bno_p = dual ? lin::kClusterBN / 2 : lin::kClusterBN;
      const long long pair_tiles = (long long)((M + 2 * lin::kBM - 1) / (2 * lin::kBM)) *
                                   (long long)((N + bno_p - 1) / bno_p);
      pair = f16_pair(pair_tiles, sm_count(dev));
      cn = pair ? 2 : 1;
    }
    const int cn_n = pair ? 1 : cn;                           // CTAs along N
    const int tile_rows = pair ? 2 * lin::kBM : lin::kBM;     // rows of a cluster tile
    const int num_m = (int)((M + tile_rows - 1) / tile_rows);
    auto capacity = [&]() {
      if (dual) return lin::cluster_capacity_dual(tma_a, cn, &ce);
      if (p.bt) return lin::cluster_capacity_bt(tma_a, cn, resid, &ce);
      return swiglu ? lin::cluster_capacity_swiglu(cn, &ce)
                    : (tma_a ? lin::cluster_capacity_tma(cn, resid, &ce)
                             : lin::cluster_capacity_cvt(cn, resid, &ce));
    };
    int cap = capacity();
    if (cap < 1) return cuda_fail(ce);
    // (a split tail's rows are finished by the split sum, which has no partials)
    // (the dual product's tiles are split nowhere either: the split sum
    // writes one output)
    const int bno = dual ? lin::kClusterBN / 2 : lin::kClusterBN;
    const int num_ng_o = (int)((N + (uint64_t)bno * cn_n - 1) / ((uint64_t)bno * cn_n));
    lin::SplitPlan plan = (p.row_stats || dual) ? lin::SplitPlan{0, 0, 1}
                                                : lin::split_plan(num_m * num_ng_o, cap, nkb);
    // Bands of column groups whose weights stay in L2 (every cluster tile
    // reads K x cn x 256 binary16 weights, both halves of the dual form
    // included), when the whole W would not fit.
    {
      const long long per_ng = (long long)K * cn_n * lin::kClusterBN * 2;
      const long long band = per_ng > 0 ? lin::kBandWeightBytes / per_ng : 0;
      args.band_ng = band >= 1 && band < num_ng_o ? (int)band : 0;
    }
    const size_t part_bytes = lin::split_part_bytes(plan, cn, lin::kClusterBN);
    const size_t xh_off = (part_bytes + 255) & ~size_t(255);
    const size_t xh_bytes = tma_a ? (size_t)M * (size_t)K * 2 : 0;
    const size_t need = xh_bytes ? xh_off + xh_bytes : part_bytes;
    const int got = need ? take_workspace(need) : 0;
    args.part_f4 = got > 0 ? (int64_t)(part_bytes / 16) : 0;
    if (got < 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
    if (got == 0 && tma_a) {   // no memory for the pre-pass: transform X in the GEMM
      tma_a = false;
      pair = false;
      cn = 1;
      cap = capacity();
      if (cap < 1) return cuda_fail(ce);
    }
    if (got > 0 && plan.s >= 2) {
      args.split_r = plan.r;
      args.split_rem = plan.rem;
      args.split_s = plan.s;
    }
    if (tma_a) {
      uint16_t* xh = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(args.part) + xh_off);
      if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT16, xh, K, M, K * 2, 64,
                     (uint32_t)lin::kBM))
        e = cudaErrorInvalidValue;
      // a pair's CTA loads half of the tile's rows of W as [N][K]
      else if (pair && p.bt &&
               !encode_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W, K, N, K * 2, 64,
                          (uint32_t)lin::kClusterBN / 2))
        e = cudaErrorInvalidValue;
      else
        e = lin::launch_cvt_f16(p.X, xh, M * K, sm_count(dev), stream);
      kernels = 2;
      if (e == cudaSuccess && dual && pair) {
        // The gate and up products as CTA pairs: two launches of the
        // single-product kernel on the one binary16 X, each in its own tile
        // order (its W alone stays in L2), rather than the dual kernel,
        // whose tiles hold both products' columns and whose W and W2 need
        // two bands: at 16k tokens 794 against 883 us (one GB300, the two
        // ways alternating), and 2 x 100.7 against 226.8 us with 140
        // against 166 MB of DRAM reads at 4k tokens.
        lin::KernelArgs a = args;
        const long long per_ng = (long long)K * lin::kClusterBN * 2;
        const long long band = per_ng > 0 ? lin::kBandWeightBytes / per_ng : 0;
        const long long ng = (long long)((N + lin::kClusterBN - 1) / lin::kClusterBN);
        a.band_ng = band >= 1 && band < ng ? (int)band : 0;
        e = lin::launch_gemm_cluster_tma(cn, false, maps, a, stream);
        if (e == cudaSuccess) {
          lin::TensorMaps m2 = maps;
          m2.w = maps.w2;
          m2.y = maps.y2;
          a.Y = p.Y2;
          e = lin::launch_gemm_cluster_tma(cn, false, m2, a, stream);
        }
        kernels = 3;
      } else if (e == cudaSuccess) {
        e = dual   ? lin::launch_gemm_cluster_dual(true, cn, maps, args, stream)
            : p.bt ? lin::launch_gemm_cluster_bt(true, cn, resid, maps, args, stream)
                   : lin::launch_gemm_cluster_tma(cn, resid, maps, args, stream);
      }
    } else if (dual) {
      e = lin::launch_gemm_cluster_dual(false, cn, maps, args, stream);
    } else if (p.bt) {
      e = lin::launch_gemm_cluster_bt(false, cn, resid, maps, args, stream);
    } else {
      e = swiglu ? lin::launch_gemm_cluster_swiglu(cn, maps, args, stream)
                 : lin::launch_gemm_cluster_cvt(cn, resid, maps, args, stream);
    }
    if (e == cudaSuccess && args.split_s >= 2) {
      const int clusters = args.split_r > 0 ? cap : args.split_rem * args.split_s;
      e = lin::launch_split_reduce(args, resid, cn, pair, lin::kClusterBN,
                                   args.split_r * clusters, num_ng_o, stream);
      kernels += 1;
    }
  } else {
    // One CTA per 128 x bn tile; when the tiles leave most SMs idle, split K
    // into S ranges (grid.z) of at least 4 k-blocks each. Where A is X (or
    // X^T, or dY) the S CTAs of a tile form a cluster and sum their partial
    // tiles through distributed shared memory (S at most 8, and lowered at
    // launch until every tile's cluster is resident at once); the SwiGLU
    // forms, whose A is built by the transform warps, gain more from every
    // SM than from one kernel, and keep the workspace and the split sum
    // (measured on the 512-token shapes).
    const int tiles_n = (int)((N + bn - 1) / bn);
    const int tiles = tiles_n * (int)((M + lin::kBM - 1) / lin::kBM);
    const int nkb = (int)((K + (p.w16 ? 63 : 31)) / (p.w16 ? 64 : 32));
    int split = sm_count(dev) / tiles;
    if (split > nkb / 4) split = nkb / 4;
    const bool cl = !(swiglu && !p.at);
    if (cl && split > lin::kMaxClusterSplit) split = lin::kMaxClusterSplit;
    if (split >= 2 && cl) {
      args.split_r = 0;
      args.split_rem = tiles;
      args.split_s = split;
      args.flags |= lin::KFLAG_CLUSTER_SPLIT;
    } else if (split >= 2) {
      const size_t bytes = (size_t)tiles * split * lin::kBM * bn * sizeof(float);
      const int got = take_workspace(bytes);
      args.part_f4 = got > 0 ? (int64_t)(bytes / 16) : 0;
      if (got < 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
      if (got > 0) {
        args.split_r = 0;
        args.split_rem = tiles;
        args.split_s = split;
      }
    }
    if (p.w16)
      e = lin::launch_gemm_f16(swiglu ? lin::A_SWIGLU_F16 : lin::A_CVT_F16, resid, bn, p.bt, maps,
                               args, stream);
    else
      e = lin::launch_gemm_tf32(swiglu ? (p.at ? lin::A_TRANS_SWIGLU_F32 : lin::A_SWIGLU_F32)
                                       : (p.at ? lin::A_TRANS_F32 : lin::A_TMA_F32),
                                resid, bn, p.bt, maps, args, stream);
    if (e == cudaSuccess && args.split_s >= 2 && !(args.flags & lin::KFLAG_CLUSTER_SPLIT)) {
      e = lin::launch_split_reduce(args, resid, 1, false, bn, 0, tiles_n, stream);
      kernels = 2;
    }
  }
  if (ws) {
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_kernels = kernels;
  t_last_workspace = workspace;
  return LIN_SUCCESS;
}

// lm_head (logits = X @ W16 into DLOGITS) and the fused cross-entropy of
// page 07_loss on them: the GEMM's epilogue leaves per-row partials, the
// loss kernel turns the logits into dLogits in place, writes the per-row
// losses, and its last CTA their sum.
lin_status lm_head_cross_entropy(const float* X, const uint16_t* W16, const int32_t* targets,
                                 float* dlogits, float* losses, float* loss_sum, int64_t M,
                                 int64_t V, int64_t K, float alpha, float beta, float inv_norm,
                                 cudaStream_t stream) {
  t_last_kernels = 0;
  t_last_workspace = 0;
  if (M < 0 || V < 0 || K < 0 || !loss_sum) return LIN_ERROR_INVALID_VALUE;
  if (M > 0 && (!targets || !dlogits || !losses)) return LIN_ERROR_INVALID_VALUE;
  if (M > 0 && V > 0 && K > 0 && (!X || !W16)) return LIN_ERROR_INVALID_VALUE;
  const int64_t kMax = 0x7fffffffLL;
  if (M > kMax || V > kMax || K > kMax) return LIN_ERROR_UNSUPPORTED_SHAPE;
  if (V % 8 != 0 || K % 4 != 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
  auto misaligned16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
  auto misaligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) != 0; };
  if (misaligned4(loss_sum)) return LIN_ERROR_MISALIGNED;
  if (M > 0 && (misaligned16(dlogits) || misaligned4(targets) || misaligned4(losses) ||
                (K > 0 && (misaligned16(X) || misaligned16(W16)))))
    return LIN_ERROR_MISALIGNED;
  const uint64_t mv = (uint64_t)M * (uint64_t)V * 4, mk = (uint64_t)M * (uint64_t)K * 4,
                 kv = (uint64_t)K * (uint64_t)V * 2, m4 = (uint64_t)M * 4;
  if (M > 0) {
    const struct { const void* p; uint64_t n; } ins[] = {{X, K > 0 ? mk : 0},
                                                         {W16, K > 0 ? kv : 0}, {targets, m4}};
    for (const auto& in : ins)
      if (overlaps(dlogits, mv, in.p, in.n) || overlaps(losses, m4, in.p, in.n) ||
          overlaps(loss_sum, 4, in.p, in.n))
        return LIN_ERROR_ALIASING;
    if (overlaps(dlogits, mv, losses, m4) || overlaps(dlogits, mv, loss_sum, 4) ||
        overlaps(losses, m4, loss_sum, 4))
      return LIN_ERROR_ALIASING;
  }
  int dev = 0;
  int* word = nullptr;
  lin_status st = current_device(&dev, &word);
  if (st != LIN_SUCCESS) return st;
  if ((st = check_buffer(loss_sum, 4, dev)) != LIN_SUCCESS) return st;
  if (M == 0) {   // no rows: the sum of no losses
    const cudaError_t e = cudaMemsetAsync(loss_sum, 0, 4, stream);
    return e == cudaSuccess ? LIN_SUCCESS : cuda_fail(e);
  }
  if ((st = check_buffer(targets, m4, dev)) != LIN_SUCCESS) return st;
  if ((st = check_buffer(losses, m4, dev)) != LIN_SUCCESS) return st;
  if (V == 0) {   // every target is outside the (empty) vocabulary
    cudaError_t e = cudaMemsetAsync(losses, 0, m4, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(loss_sum, 0, 4, stream);
    return e == cudaSuccess ? LIN_SUCCESS : cuda_fail(e);
  }
  // the row partials: stream-ordered workspace (a graph memory node under
  // capture), freed after the loss kernel; without it the loss kernel reads
  // each row three times instead of once
  const int cols = (int)((V + lin::kClusterBN - 1) / lin::kClusterBN);
  const size_t stats_bytes = (size_t)M * cols * sizeof(float4);
  // after the partials: the loss kernel's count of finished rows (zeroed by
  // the GEMM, or by a memset when there is no GEMM)
  const size_t ws_bytes = stats_bytes + 16;
  void* ws = nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) cudaGetLastError();
  if (cs == cudaStreamCaptureStatusActive) {
    if (cudaMallocAsync(&ws, ws_bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      ws = nullptr;
    }
  } else if (cs == cudaStreamCaptureStatusNone) {
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool || cudaMallocFromPoolAsync(&ws, ws_bytes, pool, stream) != cudaSuccess) {
      cudaGetLastError();
      ws = nullptr;
    }
  }
  Problem p{F_MATMUL, true, X, nullptr, nullptr, W16, nullptr, dlogits, M, V, K};
  // (with K == 0 the GEMM only zeroes the logits and leaves no partials)
  p.row_stats = K > 0 ? static_cast<float4*>(ws) : nullptr;
  p.stats_cols = cols;
  unsigned* done =
      ws ? reinterpret_cast<unsigned*>(static_cast<char*>(ws) + stats_bytes) : nullptr;
  p.zero_word = K > 0 ? done : nullptr;
  st = run(p, stream);
  const int gemm_kernels = t_last_kernels;
  const uint64_t gemm_ws = t_last_workspace;
  cudaError_t e = cudaSuccess;
  if (st == LIN_SUCCESS && done && K == 0) e = cudaMemsetAsync(done, 0, 4, stream);
  if (st == LIN_SUCCESS && e == cudaSuccess)
    e = lin::launch_cross_entropy(dlogits, p.row_stats, cols, targets, losses, loss_sum,
                                  (int)M, (int)V, alpha, beta, inv_norm, done, word, stream);
  if (ws) {
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
  }
  if (st != LIN_SUCCESS) return st;
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_kernels = gemm_kernels + (done ? 1 : 2);
  t_last_workspace = gemm_ws + (ws ? ws_bytes : 0);
  return LIN_SUCCESS;
}

lin_status record_cuda_error(cudaError_t e) { return cuda_fail(e); }

lin_status forward_shape_status(bool w16, int64_t M, int64_t N, int64_t K) {
  const int64_t kMax = 0x7fffffffLL;
  if (M > kMax || N > kMax || K > kMax) return LIN_ERROR_UNSUPPORTED_SHAPE;
  if (K % 4 != 0 || N % 4 != 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
  if (w16 && N % 8 != 0) return LIN_ERROR_UNSUPPORTED_SHAPE;
  return LIN_SUCCESS;
}

lin_status checked_device(int* dev) {
  int* word = nullptr;
  return current_device(dev, &word);
}

cudaMemPool_t device_pool(int dev) { return workspace_pool(dev); }

void set_last_launch_info(int kernels, uint64_t workspace_bytes) {
  t_last_kernels = kernels;
  t_last_workspace = workspace_bytes;
}

lin_status run_forward_staged(int form, bool w16, const float* X, const float* G, const float* U,
                              const void* W, const float* R, float* Y, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
  Problem p{static_cast<Form>(form), w16, X, G, U, W, R, Y, M, N, K};
  p.staged = true;
  return run(p, stream);
}

lin_status run_swiglu_w16_fixed(const float* GATE, const float* UP, const uint16_t* W16,
                                const float* R, float* Y, int64_t M, int64_t N, int64_t K,
                                cudaStream_t stream, lin::WorkspaceGetter get) {
  return run({F_SWIGLU, true, nullptr, GATE, UP, W16, R, Y, M, N, K}, stream, get);
}

lin_status read_and_clear_status(cudaStream_t stream) {
  int dev = 0;
  int* word = nullptr;
  lin_status st = current_device(&dev, &word);
  if (st != LIN_SUCCESS) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int v[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(v, g_status_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e);
  const int zero[4] = {0, 0, 0, 0};
  e = cudaMemcpyToSymbol(g_status_word, zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e);
  if (v[0] == lin::KSTATUS_CHECK) {
    t_last_check_site = v[1];
    int64_t value = 0;
    std::memcpy(&value, v + 2, sizeof(value));
    t_last_check_value = value;
    return LIN_ERROR_DEVICE_CHECK;
  }
  return v[0] == lin::KSTATUS_TIMEOUT ? LIN_ERROR_TIMEOUT : LIN_SUCCESS;
}

}  // namespace lin_detail

using namespace lin_detail;

extern "C" {

lin_status lin_matmul(const float* X, const float* W, float* Y, int64_t M, int64_t N, int64_t K,
                      lin_stream_t stream) {
  return run({F_MATMUL, false, X, nullptr, nullptr, W, nullptr, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_residual(const float* X, const float* W, const float* R, float* Y,
                               int64_t M, int64_t N, int64_t K, lin_stream_t stream) {
  return run({F_RESID, false, X, nullptr, nullptr, W, R, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_residual_swiglu_a(const float* GATE, const float* UP, const float* W,
                                        const float* R, float* Y, int64_t M, int64_t N, int64_t K,
                                        lin_stream_t stream) {
  return run({F_SWIGLU, false, nullptr, GATE, UP, W, R, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_w16(const float* X, const uint16_t* W16, float* Y, int64_t M, int64_t N,
                          int64_t K, lin_stream_t stream) {
  return run({F_MATMUL, true, X, nullptr, nullptr, W16, nullptr, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_residual_w16(const float* X, const uint16_t* W16, const float* R, float* Y,
                                   int64_t M, int64_t N, int64_t K, lin_stream_t stream) {
  return run({F_RESID, true, X, nullptr, nullptr, W16, R, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_residual_swiglu_a_w16(const float* GATE, const float* UP,
                                            const uint16_t* W16, const float* R, float* Y,
                                            int64_t M, int64_t N, int64_t K,
                                            lin_stream_t stream) {
  return run({F_SWIGLU, true, nullptr, GATE, UP, W16, R, Y, M, N, K},
             reinterpret_cast<cudaStream_t>(stream));
}

// Backward of the linear layer: dX[M,K] = dY[M,N] · W[K,N]^T (+ dX).
// In the kernels' terms the output has K columns and the contraction runs
// over N, with W read as [K rows][N] = B^T.
lin_status lin_matmul_t(const float* DY, const float* W, float* DX, int64_t M, int64_t N,
                        int64_t K, lin_stream_t stream) {
  Problem p{F_MATMUL, false, DY, nullptr, nullptr, W, nullptr, DX, M, K, N};
  p.bt = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_t_acc(const float* DY, const float* W, float* DX, int64_t M, int64_t N,
                            int64_t K, lin_stream_t stream) {
  Problem p{F_RESID, false, DY, nullptr, nullptr, W, DX, DX, M, K, N};
  p.bt = true;
  p.acc = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_t_w16(const float* DY, const uint16_t* W16, float* DX, int64_t M, int64_t N,
                            int64_t K, lin_stream_t stream) {
  Problem p{F_MATMUL, true, DY, nullptr, nullptr, W16, nullptr, DX, M, K, N};
  p.bt = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_t_acc_w16(const float* DY, const uint16_t* W16, float* DX, int64_t M,
                                int64_t N, int64_t K, lin_stream_t stream) {
  Problem p{F_RESID, true, DY, nullptr, nullptr, W16, DX, DX, M, K, N};
  p.bt = true;
  p.acc = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

// Weight gradient of the linear layer: dW[K,N] = X[M,K]^T · dY[M,N] (+ dW).
// In the kernels' terms the output has K rows and the contraction runs over
// the M tokens, with A = X^T.
lin_status lin_matmul_at(const float* X, const float* DY, float* DW, int64_t M, int64_t N,
                         int64_t K, lin_stream_t stream) {
  Problem p{F_MATMUL, false, X, nullptr, nullptr, DY, nullptr, DW, K, N, M};
  p.at = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_at_acc(const float* X, const float* DY, float* DW, int64_t M, int64_t N,
                             int64_t K, lin_stream_t stream) {
  Problem p{F_RESID, false, X, nullptr, nullptr, DY, DW, DW, K, N, M};
  p.at = true;
  p.acc = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

// Weight gradient of the SwiGLU down projection: dW[K,N] =
// (silu(GATE) * UP)[M,K]^T · dY[M,N] (+ dW), the product recomputed on chip.
lin_status lin_matmul_at_swiglu_a(const float* GATE, const float* UP, const float* DY, float* DW,
                                  int64_t M, int64_t N, int64_t K, lin_stream_t stream) {
  Problem p{F_SWIGLU, false, nullptr, GATE, UP, DY, nullptr, DW, K, N, M};
  p.at = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_at_swiglu_a_acc(const float* GATE, const float* UP, const float* DY,
                                      float* DW, int64_t M, int64_t N, int64_t K,
                                      lin_stream_t stream) {
  Problem p{F_SWIGLU, false, nullptr, GATE, UP, DY, DW, DW, K, N, M};
  p.at = true;
  p.acc = true;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

// Backward of the FFN down projection and its SwiGLU in one call: dA =
// dY · W^T stays on chip, and the epilogue writes dGATE and dUP of
// A = silu(GATE) * UP (page 09_backward_ffn, ffn_swiglu_backward).
lin_status lin_matmul_t_swiglu_backward(const float* DY, const float* W, const float* GATE,
                                        const float* UP, float* DGATE, float* DUP, int64_t M,
                                        int64_t N, int64_t K, lin_stream_t stream) {
  Problem p{F_MATMUL, false, DY, nullptr, nullptr, W, nullptr, DGATE, M, K, N};
  p.bt = true;
  p.G2 = GATE;
  p.U2 = UP;
  p.Y2 = DUP;
  if (!DUP) return LIN_ERROR_INVALID_VALUE;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_matmul_t_swiglu_backward_w16(const float* DY, const uint16_t* W16,
                                            const float* GATE, const float* UP, float* DGATE,
                                            float* DUP, int64_t M, int64_t N, int64_t K,
                                            lin_stream_t stream) {
  Problem p{F_MATMUL, true, DY, nullptr, nullptr, W16, nullptr, DGATE, M, K, N};
  p.bt = true;
  p.G2 = GATE;
  p.U2 = UP;
  p.Y2 = DUP;
  if (!DUP) return LIN_ERROR_INVALID_VALUE;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

lin_status lin_lm_head_cross_entropy_w16(const float* X, const uint16_t* W16,
                                         const int32_t* targets, float* DLOGITS, float* losses,
                                         float* loss_sum, int64_t M, int64_t V, int64_t K,
                                         float alpha, float beta, float inv_norm,
                                         lin_stream_t stream) {
  return lm_head_cross_entropy(X, W16, targets, DLOGITS, losses, loss_sum, M, V, K, alpha, beta,
                               inv_norm, reinterpret_cast<cudaStream_t>(stream));
}

// The FFN's gate and up projections in one launch: GATE = X @ W_gate and
// UP = X @ W_up (binary16 weights) from one read of X.
lin_status lin_gate_up_w16(const float* X, const uint16_t* WG16, const uint16_t* WU16,
                           float* GATE, float* UP, int64_t M, int64_t N, int64_t K,
                           lin_stream_t stream) {
  Problem p{F_MATMUL, true, X, nullptr, nullptr, WG16, nullptr, GATE, M, N, K};
  p.W2 = WU16;
  p.Y2 = UP;
  if (!UP || (K > 0 && !WU16)) return LIN_ERROR_INVALID_VALUE;
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

const char* lin_status_string(lin_status status) {
  switch (status) {
    case LIN_SUCCESS: return "LIN_SUCCESS";
    case LIN_ERROR_INVALID_VALUE: return "LIN_ERROR_INVALID_VALUE";
    case LIN_ERROR_UNSUPPORTED_SHAPE: return "LIN_ERROR_UNSUPPORTED_SHAPE";
    case LIN_ERROR_MISALIGNED: return "LIN_ERROR_MISALIGNED";
    case LIN_ERROR_ALIASING: return "LIN_ERROR_ALIASING";
    case LIN_ERROR_UNSUPPORTED_DEVICE: return "LIN_ERROR_UNSUPPORTED_DEVICE";
    case LIN_ERROR_CUDA: return "LIN_ERROR_CUDA";
    case LIN_ERROR_TIMEOUT: return "LIN_ERROR_TIMEOUT";
    case LIN_ERROR_DEVICE_CHECK: return "LIN_ERROR_DEVICE_CHECK";
  }
  return "LIN_ERROR_UNKNOWN";
}

int lin_last_cuda_error(void) { return t_last_cuda_error; }

void lin_last_launch_info(int* kernels, uint64_t* workspace_bytes) {
  if (kernels) *kernels = t_last_kernels;
  if (workspace_bytes) *workspace_bytes = t_last_workspace;
}

lin_status lin_get_device_status(lin_stream_t stream) {
  return read_and_clear_status(reinterpret_cast<cudaStream_t>(stream));
}

void lin_last_device_check(int* site, int64_t* value) {
  if (site) *site = t_last_check_site;
  if (value) *value = t_last_check_value;
}

lin_status lin_selftest_device_check(int64_t value, lin_stream_t stream) {
  int dev = 0;
  int* word = nullptr;
  lin_status st = current_device(&dev, &word);
  if (st != LIN_SUCCESS) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = lin::launch_selftest_check(word, (long long)value, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return read_and_clear_status(s);
}

lin_status lin_selftest_wait_timeout(int64_t timeout_us, lin_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return LIN_ERROR_INVALID_VALUE;
  int dev = 0;
  int* word = nullptr;
  lin_status st = current_device(&dev, &word);
  if (st != LIN_SUCCESS) return st;
  // The producers issue nothing, so the tensor maps are never dereferenced.
  lin::TensorMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  lin::KernelArgs args{};
  args.M = 128;
  args.N = 128;
  args.K = 128;
  args.flags = lin::KFLAG_WITHHOLD_PRODUCER;
  args.timeout_ns = static_cast<uint64_t>(timeout_us) * 1000ull;
  args.status = word;
  args.R = nullptr;
  args.Y = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = lin::launch_gemm_tf32(lin::A_TMA_F32, false, 128, false, maps, args, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return read_and_clear_status(s);
}

int lin_version(void) { return 200; }   // 0.2.0: backward, loss, gate/up and host-operand entry points

}  // extern "C"
