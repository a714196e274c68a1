// lin_loss.cu -- the fused cross-entropy of page "cross_entropy ve
// sum_losses -- Fused Loss + dLogits" (07_loss) applied to the logits the
// lm_head GEMM has just written, and the sum of the losses.
//
// One CTA per row, as on the page. The page's phases 1 and 2a (row max, sum
// of exponentials) read the row twice, and label smoothing needs the row's
// sum; when the GEMM's epilogue has left partials per row (max, sum of
// exp(l - max) and sum of l over each CTA's 256 columns), they are combined
// here instead, and the row is read once, for phase 4, which writes dLogits
// in place.
#include "lin_ce.cuh"

namespace lin {

namespace {

constexpr int kLossThreads = 256;

// Block-wide reductions in a fixed order (warp shuffles, then the warps'
// results by warp 0): the same inputs give the same bits.
template <bool MAX>
__device__ __forceinline__ float block_reduce(float v, float* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? fmaxf(v, w) : v + w;
  }
  __syncthreads();   // sh may still be read from the previous reduction
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kLossThreads / 32 ? sh[lane] : (MAX ? -INFINITY : 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float w = __shfl_xor_sync(0xffffffffu, v, o);
      v = MAX ? fmaxf(v, w) : v + w;
    }
    if (lane == 0) sh[0] = v;
  }
  __syncthreads();
  return sh[0];
}

}  // namespace

// A CTA's first kRegF4 float4s of its row are loaded into registers
// (kChunk per thread) and the next kSmemF4 (kSmemChunk per thread) copied
// into shared memory by cp.async, all requested together with the target
// index before anything else, so that the whole row (V <= 16384) is in
// flight at once; the rest of a longer row is read in further register
// chunks during phase 4. (Six register float4s a thread keep the kernel
// within the 64 registers of four CTAs per SM.)
constexpr int kChunk = 6;
constexpr int kSmemChunk = 10;
constexpr int kRegF4 = kChunk * kLossThreads;           // 1536 float4s: 24 KB
constexpr int kSmemF4 = kSmemChunk * kLossThreads;      // the next 40 KB
constexpr size_t kLossSmemBytes = (size_t)kSmemF4 * 16;

__global__ void __launch_bounds__(kLossThreads, 4)
    lin_cross_entropy_kernel(float* __restrict__ logits, const float4* __restrict__ stats,
                             int stats_cols, const int32_t* __restrict__ targets,
                             float* __restrict__ losses, int V, float alpha, float beta,
                             float inv_norm, unsigned* __restrict__ done,
                             float* __restrict__ loss_sum, int* status) {
  extern __shared__ float4 staged[];   // kSmemF4 float4s of the row
  __shared__ float sh[kLossThreads / 32];
  const int s = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // Launched as a programmatic dependent of the GEMM: wait for its logits.
  pdl_wait();
  float* row = logits + (size_t)s * (size_t)V;
  float4* row4 = reinterpret_cast<float4*>(row);
  const int V4 = V / 4;   // V % 4 == 0
  const int tgt = targets[s];
  float4 l[kChunk];
  auto load_chunk = [&](int v0) {
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int v = v0 + u * kLossThreads;
      if (v < V4) l[u] = row4[v];
    }
  };
  load_chunk(tid);
  // thread t's shared-memory float4s are t + u * kLossThreads, which it
  // alone copies and later reads: its own cp_async_wait_all suffices
  const uint32_t st0 = smem_u32(staged);
#pragma unroll
  for (int u = 0; u < kSmemChunk; ++u) {
    const int v = kRegF4 + tid + u * kLossThreads;
    if (v < V4 &&
        dcheck(tid + u * kLossThreads < kSmemF4, status, CHK_BUFFER, tid + u * kLossThreads))
      cp_async_16(st0 + 16u * (uint32_t)(tid + u * kLossThreads), row4 + v);
  }
  if (tgt < 0 || tgt >= V) {   // ignored row (padding): loss 0, dLogits 0
    cp_async_wait_all();       // no copy may still write our shared memory
    for (int v = tid; v < V4; v += kLossThreads) row4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == 0) {
      if (lane == 0) losses[s] = 0.0f;
      count_and_sum_warp(losses, gridDim.x, done, loss_sum, lane);
    }
    return;
  }
  const float l_t = tid == 0 ? row[tgt] : 0.0f;   // phase 3 needs it before phase 4 overwrites it
  // phases 1 and 2a (row max and sum of exp(l - max)) and the row sum that
  // label smoothing needs
  float row_max, denom, total;
  if (stats) {
    // Every warp merges the GEMM's partials of the row by itself, so no
    // warp waits for another.
    const float4* st = stats + (size_t)s * stats_cols;
    const bool row_ok = dcheck(s < (int)gridDim.x, status, CHK_STATS, s);
    const float3 rs = warp_merge_partials([&](int i) { return st[i]; }, row_ok ? stats_cols : 0,
                                          lane);
    row_max = rs.x;
    denom = rs.y;
    total = rs.z;
  } else {   // no partials: read the row from global memory for them
    float m = -INFINITY;
    for (int v = tid; v < V4; v += kLossThreads) {
      const float4 x = row4[v];
      m = fmaxf(m, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    }
    row_max = block_reduce<true>(m, sh);
    float d = 0.0f, sum = 0.0f;
    for (int v = tid; v < V4; v += kLossThreads) {
      const float4 x = row4[v];
      d += __expf(x.x - row_max) + __expf(x.y - row_max) + __expf(x.z - row_max) +
           __expf(x.w - row_max);
      sum += (x.x + x.y) + (x.z + x.w);
    }
    denom = block_reduce<false>(d, sh);
    total = block_reduce<false>(sum, sh);
  }
  const CeRow cr = ce_row(row_max, denom, V, alpha, beta, inv_norm);
  const int tv = tgt >> 2, tj = tgt & 3;   // the float4 holding the target, and its lane
  // phase 3: the loss, and the count of sum_losses (warp 0; before its
  // phase 4, so that the count's fence has only the loss to wait for)
  if (warp == 0) {
    if (lane == 0) losses[s] = ce_loss(cr, l_t, total, V, alpha, beta);
    count_and_sum_warp(losses, gridDim.x, done, loss_sum, lane);
  }
  // phase 4: dLogits in place, from registers, then from shared memory, then
  // (longer rows) register chunk by chunk
  auto grad = [&](const float4 x, int v) -> float4 { return ce_grad4(cr, x, v, tv, tj); };
#pragma unroll
  for (int u = 0; u < kChunk; ++u) {
    const int v = tid + u * kLossThreads;
    if (v < V4) row4[v] = grad(l[u], v);
  }
  cp_async_wait_all();
#pragma unroll
  for (int u = 0; u < kSmemChunk; ++u) {
    const int v = kRegF4 + tid + u * kLossThreads;
    if (v < V4) row4[v] = grad(staged[tid + u * kLossThreads], v);
  }
  for (int v0 = kRegF4 + kSmemF4 + tid; v0 < V4; v0 += kChunk * kLossThreads) {
    load_chunk(v0);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int v = v0 + u * kLossThreads;
      if (v < V4) row4[v] = grad(l[u], v);
    }
  }
}

// sum_losses: one CTA, a strided sum then the fixed-order block reduction.
__global__ void __launch_bounds__(kLossThreads)
    lin_sum_losses_kernel(const float* __restrict__ losses, int M, float* __restrict__ out) {
  __shared__ float sh[kLossThreads / 32];
  pdl_wait();
  float v = 0.0f;
  for (int i = threadIdx.x; i < M; i += kLossThreads) v += losses[i];
  v = block_reduce<false>(v, sh);
  if (threadIdx.x == 0) *out = v;
}

cudaError_t launch_cross_entropy(float* logits, const float4* row_stats, int stats_cols,
                                 const int32_t* targets, float* losses, float* loss_sum, int M,
                                 int V, float alpha, float beta, float inv_norm, unsigned* done,
                                 int* status, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(kLossThreads, 1, 1);
  cfg.dynamicSmemBytes = kLossSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lin_cross_entropy_kernel, logits, row_stats,
                                     stats_cols, targets, losses, V, alpha, beta, inv_norm, done,
                                     loss_sum, status);
  if (e != cudaSuccess || done) return e;
  cfg.gridDim = dim3(1, 1, 1);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, lin_sum_losses_kernel, (const float*)losses, M, loss_sum);
}

}  // namespace lin
