// lin_ce.cuh -- the arithmetic of the fused cross-entropy of page
// "cross_entropy ve sum_losses -- Fused Loss + dLogits" (07_loss) that the
// loss kernel (lin_loss.cu) applies to the lm_head GEMM's logits: merging
// online-softmax partials, the loss of a row (phase 3), dLogits (phase 4)
// and sum_losses.
#pragma once

#include "lin_common.cuh"

namespace lin {

// Online-softmax partials (max m, sum s of exp(l - m)) merged: the pair for
// the union of both column sets. -inf maxima (no columns) merge as no-ops.
__device__ __forceinline__ void merge_softmax(float& m, float& s, float m2, float s2) {
  const float mx = fmaxf(m, m2);
  if (mx == -INFINITY) return;
  s = (m == -INFINITY ? 0.0f : s * __expf(m - mx)) + (m2 == -INFINITY ? 0.0f : s2 * __expf(m2 - mx));
  m = mx;
}

// A warp's merge of a row's partials (max, sum of exp(l - max), sum of l, 0)
// over `cols` column groups: lane i takes partials i, i + 32, ..., then a
// shuffle tree whose every lane ends with the same value, so that every warp
// merging the same partials gets the same bits.
template <typename Load>
__device__ __forceinline__ float3 warp_merge_partials(Load load, int cols, int lane) {
  float m = -INFINITY, e = 0.0f, sum = 0.0f;
  for (int i = lane; i < cols; i += 32) {
    const float4 p = load(i);
    merge_softmax(m, e, p.x, p.y);
    sum += p.z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float e2 = __shfl_xor_sync(0xffffffffu, e, o);
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    merge_softmax(m, e, m2, e2);
  }
  return make_float3(m, e, sum);
}

// The constants of a row once its max, sum of exponentials and sum are
// known: LSE, and phase 4 per logit l as p = exp(l - lse) =
// 2^(l log2(e) - lse log2(e)), dLogit = ((p - target share) + zl p) * inv_norm
// = p c_scale - c_off, less (1 - alpha) inv_norm at the target: two FMAs and
// one ex2 a logit.
struct CeRow {
  float lse, c_shift, c_scale, c_off, c_hit;
};

__device__ __forceinline__ CeRow ce_row(float row_max, float denom, int V, float alpha, float beta,
                                        float inv_norm) {
  constexpr float kLog2e = 1.4426950408889634f;
  CeRow r;
  r.lse = row_max + logf(fmaxf(denom, 1e-30f));
  const float zl = 2.0f * beta * r.lse;
  r.c_shift = r.lse * kLog2e;
  r.c_scale = (1.0f + zl) * inv_norm;
  r.c_off = alpha * (1.0f / (float)V) * inv_norm;
  r.c_hit = (1.0f - alpha) * inv_norm;
  return r;
}

// Phase 3: the row's loss from its LSE, the target's logit and the row sum
// (label smoothing's mean is sum / V; z-loss beta * LSE^2).
__device__ __forceinline__ float ce_loss(const CeRow& r, float l_t, float row_sum, int V,
                                         float alpha, float beta) {
  const float ce =
      r.lse - (1.0f - alpha) * l_t - (alpha > 0.0f ? alpha * (row_sum * (1.0f / (float)V)) : 0.0f);
  return ce + beta * r.lse * r.lse;
}

// Phase 4 for the float4 of logits at index v (tv: the float4 holding the
// target, j: its lane within it).
__device__ __forceinline__ float4 ce_grad4(const CeRow& r, float4 x, int v, int tv, int j) {
  constexpr float kLog2e = 1.4426950408889634f;
  auto g1 = [&](float l) {
    return fmaf(ex2_approx(fmaf(l, kLog2e, -r.c_shift)), r.c_scale, -r.c_off);
  };
  float4 y = make_float4(g1(x.x), g1(x.y), g1(x.z), g1(x.w));
  if (v == tv) {
    y.x -= j == 0 ? r.c_hit : 0.0f;
    y.y -= j == 1 ? r.c_hit : 0.0f;
    y.z -= j == 2 ? r.c_hit : 0.0f;
    y.w -= j == 3 ? r.c_hit : 0.0f;
  }
  return y;
}

// sum_losses, by the CTA that counts its row last: one warp, whose lane 0
// has written the row's loss, fences it and counts the row done; the warp
// whose count reaches M adds the M losses in a fixed order (a strided sum
// per lane, then a shuffle tree), so the total has the same bits whichever
// CTA that is. `done` is zero before the first count; null: no count (a
// separate kernel adds the losses).
__device__ __forceinline__ void count_and_sum_warp(const float* losses, int M, unsigned* done,
                                                   float* loss_sum, int lane) {
  if (!done) return;
  unsigned last = 0;
  if (lane == 0) {
    __threadfence();   // this row's loss, visible before its count
    last = atomicAdd(done, 1u) == (unsigned)(M - 1) ? 1u : 0u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();   // the other losses, visible before their counts
  float v = 0.0f;
  for (int i = lane; i < M; i += 32) v += __ldcg(losses + i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) *loss_sum = v;
}

}  // namespace lin
