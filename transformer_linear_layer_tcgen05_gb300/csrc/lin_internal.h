// lin_internal.h -- declarations shared by the host API and the kernel
// translation units (not part of the public C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "lin.h"

namespace lin {

// How the A operand (the left factor, [M, K]) reaches shared memory.
enum AMode : int {
  A_TMA_F32 = 0,     // X f32 copied by TMA, consumed as TF32
  A_CVT_F16 = 1,     // X f32 staged by TMA, rounded to binary16 by transform warps
  A_SWIGLU_F32 = 2,  // GATE, UP staged by TMA; silu(GATE) * UP written as f32 (TF32 MMA)
  A_SWIGLU_F16 = 3,  // GATE, UP staged by TMA; silu(GATE) * UP rounded to binary16
  A_TMA_F16 = 4,     // X rounded to binary16 by a pre-pass, copied by TMA (clustered kernels)
  A_TRANS_F32 = 5,   // A = X^T (the weight gradient X^T dY): MN-major TF32 operand by TMA
                     // of X transposed on chip into the K-major TF32 operand
  A_TRANS_SWIGLU_F32 = 6,  // A = (silu(GATE) * UP)^T, recomputed from staged GATE/UP tiles
                           // and transposed on chip (the weight gradient of W_down)
};

enum : uint32_t {
  // Self-test only: the TMA producers issue nothing, so every consumer wait
  // must run out and the kernel must leave through its timeout path.
  KFLAG_WITHHOLD_PRODUCER = 1u << 0,
  // The A-side inputs (X, or GATE and UP) allow 32-byte loads: K % 8 == 0
  // and every base 32-byte aligned (clustered kernels).
  KFLAG_A_V8 = 1u << 1,
  // Epilogue: the SwiGLU backward of the product dA (page 09_backward_ffn,
  // ffn_swiglu_backward) instead of a store of it: dGATE -> Y, dUP -> Y2,
  // from GATE (G2) and UP (U2) at the same [M,N] coordinates.
  KFLAG_SWIGLU_BWD = 1u << 2,
  // Epilogue (clustered kernels): also the online-softmax partials of each
  // output row over this CTA's columns of a tile -- (max, sum of exp(y -
  // max), sum of y, 0) -- into row_stats[row][n0 / BN] (cross-entropy of
  // the lm_head: the row's log-sum-exp and, for label smoothing, its sum).
  KFLAG_ROW_STATS = 1u << 3,
  // Split K of the per-tile kernel within a cluster (gridDim.z CTAs of one
  // tile, cluster dims (1, 1, split_s)): each CTA leaves its partial tile in
  // its shared memory, and after a cluster barrier each sums a share of the
  // tile over the cluster's partials in K order (+ R) and writes Y; no
  // workspace and no second kernel.
  KFLAG_CLUSTER_SPLIT = 1u << 4,
};
// Largest split of the per-tile kernel: the portable cluster size.
constexpr int kMaxClusterSplit = 8;

// Device status word values (mirror lin_status). The status word is the
// first int of a 16-byte record: [status, check site, check value (int64)].
enum : int { KSTATUS_OK = 0, KSTATUS_TIMEOUT = 7, KSTATUS_CHECK = 8 };

// Sites of the checked build's device checks (lin_last_device_check).
enum CheckSite : int {
  CHK_TMA_X = 1,         // a TMA copy's innermost coordinate not 16-byte aligned
  CHK_STAGE = 2,         // an operand stage outside the ring
  CHK_BUFFER = 3,        // an epilogue or staging buffer outside its region
  CHK_TMEM = 4,          // a TMEM column range outside the allocation
  CHK_PART = 5,          // a partial-tile index outside the workspace
  CHK_STATS = 6,         // a row-partial index outside the workspace
  CHK_GLOBAL = 7,        // another global index outside its tensor
  CHK_PEER = 8,          // a cluster peer rank outside the cluster
  CHK_BARRIER = 9,       // a barrier slot outside the barrier region
  CHK_SELFTEST = 99,
};

struct KernelArgs {
  int32_t M, N, K;
  uint32_t flags;
  uint64_t timeout_ns;  // limit for any single wait inside the kernel
  int* status;          // device status word (first failure wins)
  const float* A;       // X or GATE [M, K] (kernels that load it directly)
  const float* U;       // UP [M, K] (SwiGLU forms, kernels that load it directly)
  const float* R;       // residual [M, N] (kernels that read it directly)
  float* Y;             // output [M, N] (kernels that write it directly)
  // Split tail of the clustered kernels (see SplitPlan); unused when split_s < 2.
  int32_t split_r, split_rem, split_s;
  float* part;          // partial tiles [unit][cta][BN/4 float4 columns][128 rows] (float4)
  const float* G2;      // GATE [M,N] of the SwiGLU-backward epilogue
  const float* U2;      // UP [M,N] of the SwiGLU-backward epilogue
  float* Y2;            // dUP [M,N] of the SwiGLU-backward epilogue (dGATE goes to Y)
  float4* row_stats;    // [M][stats_cols] (max, sum exp, sum, 0) partials (KFLAG_ROW_STATS)
  int32_t stats_cols;
  int32_t band_ng;      // column groups per band of the clustered tile order (0: one band)
  uint32_t* zero_word;  // (clustered kernels) set to 0 once the kernel may touch memory: the
                        // counter of a dependent kernel (null: none)
  int64_t part_f4;      // float4s of args.part (checked build: partial-tile indices)
};

// Order of the clustered kernels' tiles: tile t of a grid of num_m row
// blocks x num_ng column groups. The column groups are taken in bands of
// `band` (the last one narrower); the bands run one after another, and within
// a band the column group varies fastest. While a band runs, the clusters
// share its slice of the weights, which stays resident in L2 when the whole
// W would not. band <= 0 or >= num_ng: one band, plain row-major order.
struct TileRC {
  int m, ng;
};
__host__ __device__ inline TileRC tile_coords(int t, int num_m, int num_ng, int band) {
  if (band <= 0 || band >= num_ng) return TileRC{t / num_ng, t % num_ng};
  const int per_band = num_m * band;
  const int b = t / per_band;
  const int w = num_ng - b * band < band ? num_ng - b * band : band;
  const int i = t - b * per_band;
  return TileRC{i / w, b * band + i % w};
}
// Weight bytes a band may span (the L2 holds 126 MB; the streamed operands
// and outputs need the rest).
constexpr long long kBandWeightBytes = 32ll << 20;

// Work plan of a persistent launch over `tiles` cluster tiles on `clusters`
// clusters: `r` whole rounds (every cluster runs tiles cid + i*clusters), then
// the `rem` tiles left over are each cut into `s` K ranges (s >= 2), one per
// cluster, so that the last round keeps every cluster busy. The ranges' f32
// partial tiles go to a workspace, and a second kernel adds them up in K
// order (bitwise reproducible). s < 2: no split, whole tiles round robin.
struct SplitPlan {
  int r, rem, s;
};
constexpr int kSplitMinKb = 8;   // k-blocks per K range at least (else no split)

__host__ __device__ inline SplitPlan split_plan(int tiles, int clusters, int nkb) {
  SplitPlan p{0, 0, 1};
  if (clusters < 1 || tiles < 1) return p;
  const int r = tiles / clusters, rem = tiles % clusters;
  if (rem == 0) return p;
  int s = clusters / rem;
  if (s > nkb / kSplitMinKb) s = nkb / kSplitMinKb;
  if (s < 2) return p;
  return SplitPlan{r, rem, s};
}

// Workspace bytes of a split plan (partial tiles) for clusters of `cn` CTAs
// with tiles of 128 x `bn`.
inline size_t split_part_bytes(const SplitPlan& p, int cn, int bn) {
  return p.s >= 2 ? (size_t)p.rem * p.s * cn * 128 * bn * sizeof(float) : 0;
}

// Tensor maps of one call. `a` is X (A_TMA_F32 / A_CVT_F16) or GATE, `u` is
// UP (SwiGLU forms only), `w` the weights, `r` the residual, `y` the output.
struct TensorMaps {
  CUtensorMap a, u, w, r, y;
  CUtensorMap g2, u2, y2;   // GATE, UP, dUP of the SwiGLU-backward epilogue ([32 x 32] boxes);
                            // y2 is also the second output of the dual GEMM
  CUtensorMap w2;           // the second weight matrix of the dual GEMM
};

// Block-tile geometry shared by host and device.
constexpr int kBM = 128;           // rows of the output tile (UMMA M)
constexpr int kThreads = 256;      // 8 warps
constexpr int kEpiRows = 32;       // rows per epilogue warp (one TMEM lane quadrant)
constexpr int kEpiCols = 32;       // columns per epilogue chunk (128 bytes of f32)

// Launchers, one per translation unit family. `bn` is the tile width (128 or
// 256). They set the shared-memory attribute on first use and launch a grid
// of (ceil(N/bn), ceil(M/128)) CTAs.
cudaError_t launch_gemm_tf32(int amode, bool resid, int bn, bool bt, const TensorMaps& maps,
                             const KernelArgs& args, cudaStream_t stream);
cudaError_t launch_gemm_f16(int amode, bool resid, int bn, bool bt, const TensorMaps& maps,
                            const KernelArgs& args, cudaStream_t stream);

// Clustered persistent kernels for the binary16-weight forms: a cluster of
// `cn` CTAs along N shares the on-chip A operand (128/cn rows each). They
// read X (or GATE and UP) through KernelArgs::A/U and W through its tensor
// map; R and Y through KernelArgs.
constexpr int kClusterBN = 256;
// Columns per chunk of the clustered kernel's SwiGLU-backward epilogue
// ([32 rows][16 f32] tiles, 64-byte swizzle: GATE, UP in and dGATE, dUP out
// in four 2 KB buffers per warp).
constexpr int kSwbCols = 16;
cudaError_t launch_gemm_cluster_swiglu(int cn, const TensorMaps& maps, const KernelArgs& args,
                                       cudaStream_t stream);
cudaError_t launch_gemm_cluster_cvt(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream);
// Clusters of `cn` CTAs that can be resident at once (sets the kernel's
// shared-memory attribute on first use); > 0, or 0 with *err set.
int cluster_capacity_swiglu(int cn, cudaError_t* err);
int cluster_capacity_cvt(int cn, bool resid, cudaError_t* err);
// matmul_w16 / matmul_residual_w16 with A = binary16 X already in global
// memory (tensor map `a`, boxes of 64 x 128): each CTA copies every A
// k-block of its tile by TMA. cn 1: single CTAs (tiles of 128 rows); cn 2:
// CTA pairs (tiles of 256 rows, UMMAs of M = 256 over the two CTAs, each
// CTA loading half of the tile's W columns).
cudaError_t launch_gemm_cluster_tma(int cn, bool resid, const TensorMaps& maps,
                                    const KernelArgs& args, cudaStream_t stream);
int cluster_capacity_tma(int cn, bool resid, cudaError_t* err);
// The transposed product dY · W^T (binary16 W given as [N][K]): A rounded by
// the transform warps, or (tma_a) copied by TMA from the pre-pass's output
// (then cn 2 means CTA pairs, as above; the W box is then 128 rows).
cudaError_t launch_gemm_cluster_bt(bool tma_a, int cn, bool resid, const TensorMaps& maps,
                                   const KernelArgs& args, cudaStream_t stream);
int cluster_capacity_bt(bool tma_a, int cn, bool resid, cudaError_t* err);
// Two products of one A (Y = A @ W, Y2 = A @ W2; tensor maps w, w2, y, y2):
// each CTA covers 128 output columns of both.
cudaError_t launch_gemm_cluster_dual(bool tma_a, int cn, const TensorMaps& maps,
                                     const KernelArgs& args, cudaStream_t stream);
int cluster_capacity_dual(bool tma_a, int cn, cudaError_t* err);
// Xh[i] = binary16(X[i]) (round to nearest even) for i < n, n % 4 == 0,
// both bases 16-byte aligned.
cudaError_t launch_cvt_f16(const float* X, uint16_t* Xh, int64_t n, int sms, cudaStream_t stream);
// Cross-entropy of page 07_loss on logits [M,V] in place (dLogits), one CTA
// per row; with row_stats (stats_cols partials per row from the GEMM) the
// row max, the sum of exponentials and the row sum come from them, else from
// two passes over the row. Then the deterministic sum of the M losses into
// *loss_sum: by the loss kernel's last CTA when `done` (a counter that is
// zero when the loss kernel starts) is given, else by a second kernel.
cudaError_t launch_cross_entropy(float* logits, const float4* row_stats, int stats_cols,
                                 const int32_t* targets, float* losses, float* loss_sum, int M,
                                 int V, float alpha, float beta, float inv_norm, unsigned* done,
                                 int* status, cudaStream_t stream);
// Y (+ R) from the partial tiles of a split: tiles tile0 .. tile0 +
// split_rem - 1 of width `bn` (cluster tiles of `cn` CTAs along N, `num_ng`
// of them per row block; or, `pair`, tiles of 256 rows whose two CTAs hold
// 128 rows each), each summed over its split_s K ranges.
cudaError_t launch_split_reduce(const KernelArgs& args, bool resid, int cn, bool pair, int bn,
                                int tile0, int num_ng, cudaStream_t stream);

// One single-thread kernel that reports a failed check (site CHK_SELFTEST,
// `value`) into the status record `status`; it touches no other memory.
cudaError_t launch_selftest_check(int* status, long long value, cudaStream_t stream);

// A caller-provided split-tail workspace: returns its base and size on
// device `dev`, or an error status.
typedef lin_status (*WorkspaceGetter)(int dev, void** ptr, size_t* bytes);

}  // namespace lin

namespace lin_detail {
// lin_matmul_residual_swiglu_a_w16 with the split-tail workspace from `get`
// instead of the library's pool (lin_api.cu).
lin_status run_swiglu_w16_fixed(const float* GATE, const float* UP, const uint16_t* W16,
                                const float* R, float* Y, int64_t M, int64_t N, int64_t K,
                                cudaStream_t stream, lin::WorkspaceGetter get);
// Records `e` as the calling thread's last CUDA error; returns LIN_ERROR_CUDA.
lin_status record_cuda_error(cudaError_t e);
// The shape rules of the forward forms (dims below 2^31, K and N multiples
// of 4, N a multiple of 8 with binary16 W).
lin_status forward_shape_status(bool w16, int64_t M, int64_t N, int64_t K);
// The current device after the library's checks (sm_103, driver entry points).
lin_status checked_device(int* dev);
// The library's stream-ordered memory pool on `dev` (null if none).
cudaMemPool_t device_pool(int dev);
// What lin_last_launch_info() reports for the calling thread.
void set_last_launch_info(int kernels, uint64_t workspace_bytes);
// A forward form (0 matmul, 1 residual, 2 SwiGLU) on buffers that are pieces
// of the library's own device allocations (no allocation-range checks).
lin_status run_forward_staged(int form, bool w16, const float* X, const float* G, const float* U,
                              const void* W, const float* R, float* Y, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream);
}  // namespace lin_detail
