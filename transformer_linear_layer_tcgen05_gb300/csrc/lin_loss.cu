// lin_loss.cu -- the fused cross-entropy of page "cross_entropy ve
// sum_losses -- Fused Loss + dLogits" (07_loss) applied to the logits the
// lm_head GEMM has just written, and the sum of the losses.
//
// One CTA per row, as on the page. The page's phases 1 and 2a (row max, sum
// of exponentials) read the row twice; when the GEMM's epilogue has left
// online-softmax partials per row (max and sum of exp(l - max) over each
// CTA's 256 columns), they are combined here instead and the row is read
// once, in phase 4, which also forms the sum of the logits that label
// smoothing needs and writes dLogits in place.
#include "lin_common.cuh"

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

__global__ void __launch_bounds__(kLossThreads, 4)
    lin_cross_entropy_kernel(float* __restrict__ logits, const float2* __restrict__ stats,
                             int stats_cols, const int32_t* __restrict__ targets,
                             float* __restrict__ losses, int V, float alpha, float beta,
                             float inv_norm) {
  __shared__ float sh[kLossThreads / 32];
  const int s = blockIdx.x;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent of the GEMM: wait for its logits.
  pdl_wait();
  float* row = logits + (size_t)s * (size_t)V;
  float4* row4 = reinterpret_cast<float4*>(row);
  const int V4 = V / 4;   // V % 4 == 0
  // The thread's float4s of the row, kChunk at a time, in registers. The
  // first chunk is requested with the target index, before anything else,
  // so that its loads are in flight while the target logit and the row's
  // statistics are fetched and combined. (kChunk = 8 keeps four of these
  // CTAs resident per SM, so every row's CTA runs at once at M = 512.)
  constexpr int kChunk = 8;
  float4 l[kChunk];
  auto load_chunk = [&](int v0) {
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int v = v0 + u * kLossThreads;
      if (v < V4) l[u] = row4[v];
    }
  };
  const int tgt = targets[s];
  load_chunk(tid);
  if (tgt < 0 || tgt >= V) {   // ignored row (padding): loss 0, dLogits 0
    for (int v = tid; v < V4; v += kLossThreads) row4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) losses[s] = 0.0f;
    return;
  }
  const float l_t = row[tgt];
  // phases 1 and 2a: row max and sum of exp(l - max)
  float row_max, denom;
  if (stats) {
    const float2* st = stats + (size_t)s * stats_cols;
    float m = -INFINITY;
    for (int i = tid; i < stats_cols; i += kLossThreads) m = fmaxf(m, st[i].x);
    row_max = block_reduce<true>(m, sh);
    float d = 0.0f;
    if (row_max != -INFINITY)
      for (int i = tid; i < stats_cols; i += kLossThreads)
        if (st[i].x != -INFINITY) d += st[i].y * __expf(st[i].x - row_max);
    denom = block_reduce<false>(d, sh);
  } else {
    float m = -INFINITY;
    for (int v = tid; v < V4; v += kLossThreads) {
      const float4 l = row4[v];
      m = fmaxf(fmaxf(m, fmaxf(l.x, l.y)), fmaxf(l.z, l.w));
    }
    row_max = block_reduce<true>(m, sh);
    float d = 0.0f;
    for (int v = tid; v < V4; v += kLossThreads) {
      const float4 l = row4[v];
      d += __expf(l.x - row_max) + __expf(l.y - row_max) + __expf(l.z - row_max) +
           __expf(l.w - row_max);
    }
    denom = block_reduce<false>(d, sh);
  }
  // phase 3 needs the target logit before phase 4 overwrites the row
  // (requested before the statistics were combined, above)
  __syncthreads();
  const float dg = fmaxf(denom, 1e-30f);
  const float inv_denom = 1.0f / dg;
  const float lse = row_max + logf(dg);
  const float inv_V = 1.0f / (float)V;
  const float zl = 2.0f * beta * lse;
  const float smooth = alpha * inv_V;
  // phase 4: dLogits in place (and the sum of the logits for smoothing),
  // chunk by chunk from registers (every load of a chunk in flight at once)
  float sum_l = 0.0f;
  for (int v0 = tid; v0 < V4; v0 += kChunk * kLossThreads) {
    if (v0 != tid) load_chunk(v0);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int v = v0 + u * kLossThreads;
      if (v >= V4) break;
      sum_l += (l[u].x + l[u].y) + (l[u].z + l[u].w);
      float* e = &l[u].x;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __expf(e[i] - row_max) * inv_denom;
        const float tgt_dist = (4 * v + i == tgt ? 1.0f - alpha : 0.0f) + smooth;
        e[i] = ((p - tgt_dist) + zl * p) * inv_norm;
      }
      row4[v] = l[u];
    }
  }
  if (alpha > 0.0f) sum_l = block_reduce<false>(sum_l, sh);
  if (tid == 0) {
    const float ce = lse - (1.0f - alpha) * l_t - (alpha > 0.0f ? alpha * (sum_l * inv_V) : 0.0f);
    losses[s] = ce + beta * lse * lse;
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

cudaError_t launch_cross_entropy(float* logits, const float2* row_stats, int stats_cols,
                                 const int32_t* targets, float* losses, float* loss_sum, int M,
                                 int V, float alpha, float beta, float inv_norm,
                                 cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(kLossThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lin_cross_entropy_kernel, logits, row_stats,
                                     stats_cols, targets, losses, V, alpha, beta, inv_norm);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1, 1, 1);
  return cudaLaunchKernelEx(&cfg, lin_sum_losses_kernel, (const float*)losses, M, loss_sum);
}

}  // namespace lin
