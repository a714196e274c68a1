// lin_gemm.cuh -- the warp-specialised tcgen05 GEMM behind every forward
// form of the linear-layer family (page "matmul ve matmul_residual -- Tiled
// Matrix Multiply (Forward)", 03_linear_forward):
//
//   Y[M,N] = A[M,K] @ W[K,N] (+ R[M,N])
//
// with A = X (matmul, matmul_residual and their _w16 forms) or
// A = silu(GATE) * UP (matmul_residual_swiglu_a and its _w16 form).
//
// One CTA computes one 128 x BN output tile with the accumulator in TMEM.
// Eight warps:
//   warp 0      TMA producer of the W tiles (and of X for the TF32 path)
//   warp 1      single-thread UMMA issuer (tcgen05.mma + tcgen05.commit)
//   warp 2      TMEM allocator
//   warp 3      TMA producer of the raw f32 inputs the transform warps read
//   warps 4-7   transform warps (build the A operand in shared memory), then
//               the epilogue (TMEM -> registers, + R, TMA store of Y)
//
// The pages' design (64x64 tiles, 4x4 FMA sub-tiles per thread, TK = 16,
// double-buffered workgroup memory, "Algoritma" and "Önemli Optimizasyonlar")
// maps here to: a 128 x BN UMMA tile, a k-block of one 128-byte swizzle row
// (32 f32 or 64 f16), an NS-deep mbarrier ring instead of two buffers, and TMA
// out-of-bounds zero fill instead of `select` masking ("Code Review",
// Bulgu 1). The SwiGLU prologue fusion ("Önemli Optimizasyonlar" 3) becomes
// the transform warps: they compute silu(GATE) * UP from TMA-staged f32 tiles
// and write the swizzled UMMA operand straight into shared memory.
#pragma once

#include <cuda_fp16.h>

#include <atomic>

#include "lin_common.cuh"

namespace lin {

// BT: W is given as [N][K] (K contiguous; the transposed product dY · W^T
// of the backward pass, with N the output columns), so its tiles are a
// K-major B operand that TMA copies as they are.
template <int AMODE, bool RESID, int BN_, bool BT = false>
struct GemmTraits {
  static constexpr bool kF16 = (AMODE == A_CVT_F16 || AMODE == A_SWIGLU_F16);
  static_assert(AMODE != A_TMA_F16, "the per-tile kernel rounds A itself");
  static constexpr bool kSwiglu =
      (AMODE == A_SWIGLU_F32 || AMODE == A_SWIGLU_F16 || AMODE == A_TRANS_SWIGLU_F32);
  static constexpr bool kResid = RESID;
  // The A operand is built by the transform warps unless X is copied as is:
  // K-major (X), or MN-major for the weight gradient's X^T (X [M][K] read as
  // [contraction][tile rows], a TF32 operand in the 128-byte swizzle with
  // 32-byte atoms).
  static constexpr bool kXformA = (AMODE != A_TMA_F32 && AMODE != A_TRANS_F32);
  static constexpr bool kTransA = (AMODE == A_TRANS_F32 || AMODE == A_TRANS_SWIGLU_F32);  // A = X^T
  static constexpr bool kAmn = (AMODE == A_TRANS_F32);   // A copied MN-major
  // W [K,N] (N contiguous) is consumed MN-major straight from TMA: binary16
  // in the 128-byte swizzle, f32 (TF32) in the 128-byte swizzle with 32-byte
  // atoms (the layout an MN-major TF32 operand needs).
  static constexpr bool kBT = BT;
  static constexpr bool kXform = kXformA;
  // Transform warps: warps 4-7 (then the epilogue), and for the forward f32
  // SwiGLU form, whose transform (two MUFU operations an element) paces its
  // k-loop, warps 8-11 as well (transform only).
  static constexpr int XF_WARPS = (AMODE == A_SWIGLU_F32) ? 8 : 4;
  static constexpr int kThreadsT = (4 + XF_WARPS) * 32;

  static constexpr int BM = kBM;
  static constexpr int BN = BN_;
  static constexpr int ESZ = kF16 ? 2 : 4;      // operand element bytes
  static constexpr int BK = 128 / ESZ;          // k-block: one 128-byte swizzle row
  static constexpr int KSTEP = 32 / ESZ;        // UMMA K per instruction (32 bytes)
  static constexpr int NMMA = BK / KSTEP;       // UMMAs per k-block
  static constexpr int W_ATOM = 128 / ESZ;      // W columns per 128-byte run
  static constexpr int W_BOXES = BT ? 1 : BN / W_ATOM;   // TMA boxes per W tile

  static constexpr uint32_t A_BYTES = BM * 128;
  // one 128-byte run of BK rows (MN-major), or the whole [BN rows][128 B]
  // K-major tile (BT)
  static constexpr uint32_t B_ATOM_BYTES = BT ? BN * 128 : BK * 128;
  static constexpr uint32_t B_BYTES = W_BOXES * B_ATOM_BYTES;   // = BK * BN * ESZ
  static constexpr uint32_t OP_STAGE_BYTES = A_BYTES + B_BYTES;
  // bytes the TMA delivers straight into an operand stage
  static constexpr uint32_t OP_TMA_BYTES = (kXformA ? 0u : A_BYTES) + B_BYTES;

  // Raw stage: what the transform warps read for 32 f32 columns of K: the A
  // inputs (X, or GATE and UP).
  static constexpr int RAW_A_INPUTS = kXformA ? (kSwiglu ? 2 : 1) : 0;
  static constexpr uint32_t RAW_BOX_BYTES = BM * 128;           // [128 rows][32 f32]
  static constexpr uint32_t RAW_A_BYTES = RAW_A_INPUTS * RAW_BOX_BYTES;
  static constexpr uint32_t RAW_STAGE_BYTES = RAW_A_BYTES;
  static constexpr int RAW_PER_KB = kF16 ? BK / 32 : 1;         // raw stages per k-block
  // Raw stages carry the memory latency of the transformed inputs, operand
  // stages that of W and the local hand-off: three raw stages and what is
  // left for operand stages.
  static constexpr int NR = 3;

  static constexpr uint32_t EPI_BUF_BYTES = kEpiRows * kEpiCols * 4;   // 4 KB
  static constexpr uint32_t EPI_BYTES = 4 * 2 * EPI_BUF_BYTES;        // 2 per epilogue warp

  static constexpr uint32_t SMEM_CAP = 232448;
  static constexpr uint32_t BAR_REGION = 1024;
  static constexpr uint32_t ALIGN_SLACK = 1024;
  // The epilogue buffers alias the raw ring: it is idle once the last
  // k-block has been transformed (with nothing to transform, they stand
  // alone).
  static constexpr uint32_t FIXED_BYTES = kXform ? NR * RAW_STAGE_BYTES : EPI_BYTES;
  static constexpr int NS_FIT =
      (int)((SMEM_CAP - BAR_REGION - ALIGN_SLACK - FIXED_BYTES) / OP_STAGE_BYTES);
  static constexpr int NS = NS_FIT > 8 ? 8 : NS_FIT;

  static constexpr uint32_t OFF_OP = 0;
  static constexpr uint32_t OFF_RAW = NS * OP_STAGE_BYTES;
  static constexpr uint32_t OFF_EPI = OFF_RAW;
  static constexpr uint32_t OFF_BAR = NS * OP_STAGE_BYTES + FIXED_BYTES;
  static constexpr uint32_t SMEM_BYTES = ALIGN_SLACK + OFF_BAR + BAR_REGION;

  // Barrier slots (8 bytes each) at OFF_BAR, then the TMEM address and the
  // abort flag.
  static constexpr int BAR_OP_TMA = 0;       // TMA bytes of an operand stage landed
  static constexpr int BAR_OP_XF = BAR_OP_TMA + 8;    // transform warps filled the stage
  static constexpr int BAR_OP_EMPTY = BAR_OP_XF + 8;  // UMMAs reading the stage are done
  static constexpr int BAR_RAW_FULL = BAR_OP_EMPTY + 8;
  static constexpr int BAR_RAW_EMPTY = BAR_RAW_FULL + 4;
  static constexpr int BAR_ACC_FULL = BAR_RAW_EMPTY + 4;
  static constexpr int BAR_EPI = BAR_ACC_FULL + 1;   // 2 per epilogue warp
  static constexpr int BAR_COUNT = BAR_EPI + 8;
  static constexpr uint32_t OFF_TMEM_SLOT = BAR_COUNT * 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;

  // (TMEM is allocated in powers of two of at least 32 columns)
  static constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr uint32_t IDESC =
      umma_idesc(kF16 ? 0u : 2u, /*a_mn_major=*/kAmn, /*b_mn_major=*/!BT, BM, BN);

  // A cluster split keeps the partial tile in the operand ring; the forward
  // SwiGLU form (a workspace split only) may have a smaller ring.
  static constexpr bool kClusterSplitOK = NS * OP_STAGE_BYTES >= BM * BN * 4;
  static_assert(NS >= 2, "operand ring needs two stages");
  static_assert(kClusterSplitOK || (kSwiglu && !kTransA), "a cluster split's partial tile in the ring");
  static_assert(NR <= 4 && NS <= 8, "barrier slots");
  static_assert(!kXform || NR * RAW_STAGE_BYTES >= EPI_BYTES, "epilogue aliasing");
  static_assert(OFF_ABORT + 4 <= BAR_REGION, "barrier region");
  static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
  static_assert((BN / 4) % 8 == 0, "a cluster split's swizzle groups of eight 16-byte columns");
  static_assert(BN % W_ATOM == 0, "W runs per tile");
};

// Build part of one A k-block from one raw stage (32 f32 columns of X or of
// GATE and UP). `half` selects which 32 columns of the k-block this raw stage
// holds (always 0 for the f32 operand). tid in [0, 128).
template <int AMODE, int NT>
__device__ __forceinline__ void transform_raw_stage(uint32_t a_stage, uint32_t raw, int half,
                                                    int tid) {
  constexpr uint32_t BOX = kBM * 128;
  if constexpr (AMODE == A_SWIGLU_F32) {
    // f32 operand: chunk c of row r <- silu(G) * U of the same chunk; the
    // stage's 1024 chunks over the transform warps' NT threads.
#pragma unroll
    for (int i = 0; i < 1024 / NT; ++i) {
      const uint32_t idx = i * NT + tid;
      const uint32_t r = (idx >> 6) * 8 + (idx & 7);
      const uint32_t c = (idx >> 3) & 7;
      const uint32_t off = sw128(r, c);
      const float4 g = ld_shared_v4f(raw + off);
      const float4 u = ld_shared_v4f(raw + BOX + off);
      st_shared_v4(a_stage + off, __float_as_uint(silu_stable(g.x) * u.x),
                   __float_as_uint(silu_stable(g.y) * u.y), __float_as_uint(silu_stable(g.z) * u.z),
                   __float_as_uint(silu_stable(g.w) * u.w));
    }
  } else {
    // binary16 operand: chunk (4*half + cc) of row r holds 8 halves made from
    // f32 chunks 2cc and 2cc+1 of the raw stage.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t idx = i * 128 + tid;
      const uint32_t r = (idx >> 5) * 8 + (idx & 7);
      const uint32_t cc = (idx >> 3) & 3;
      const uint32_t o0 = sw128(r, 2 * cc);
      const uint32_t o1 = sw128(r, 2 * cc + 1);
      float4 a0 = ld_shared_v4f(raw + o0);
      float4 a1 = ld_shared_v4f(raw + o1);
      if constexpr (AMODE == A_SWIGLU_F16) {
        const float4 u0 = ld_shared_v4f(raw + BOX + o0);
        const float4 u1 = ld_shared_v4f(raw + BOX + o1);
        a0.x = silu_stable(a0.x) * u0.x;
        a0.y = silu_stable(a0.y) * u0.y;
        a0.z = silu_stable(a0.z) * u0.z;
        a0.w = silu_stable(a0.w) * u0.w;
        a1.x = silu_stable(a1.x) * u1.x;
        a1.y = silu_stable(a1.y) * u1.y;
        a1.z = silu_stable(a1.z) * u1.z;
        a1.w = silu_stable(a1.w) * u1.w;
      }
      st_shared_v4(a_stage + sw128(r, 4 * half + cc), pack_half2(a0.x, a0.y),
                   pack_half2(a0.z, a0.w), pack_half2(a1.x, a1.y), pack_half2(a1.z, a1.w));
    }
  }
}

// TF32 A operand of a weight gradient, X^T: transpose one staged tile (BN/32
// runs of [32 rows of the contraction][32 f32 of the tile's rows], 128-byte
// swizzle) into the K-major operand [BN rows][32 f32 along K] with the same
// swizzle. Warp q handles runs q, q+4, ...; lane = column inside the run.
// For a fixed k the 32 lanes read 32 distinct words of one 128-byte row, and
// each group of 8 lanes writes 8 distinct 16-byte bank groups, so neither
// side has bank conflicts.
template <int BN>
__device__ __forceinline__ void transpose_tile(uint32_t b_stage, uint32_t raw_w, int q,
                                               int lane) {
#pragma unroll 1
  for (int j = q; j < BN / 32; j += 4) {
    const uint32_t n = (uint32_t)(j * 32 + lane);
    const uint32_t src = raw_w + (uint32_t)j * 4096u;
    const uint32_t col = ((uint32_t)lane >> 2), word = ((uint32_t)lane & 3u) * 4u;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
      uint32_t v[4];
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e) {
        const uint32_t k = 4 * c + e;
        v[e] = ld_shared_u32(src + k * 128u + ((col ^ (k & 7u)) << 4) + word);
      }
      st_shared_v4(b_stage + sw128(n, c), v[0], v[1], v[2], v[3]);
    }
  }
}

// TF32 A operand of a weight gradient: (silu(GATE) * UP)^T. The raw stage
// holds [32 rows of the contraction][32 columns] boxes of GATE and of UP
// (BM/32 of each, UP at `raw_u`); warp q forms silu(g) * u of runs q, q+4,
// ... and writes them transposed, exactly as transpose_tile moves X^T.
template <int BM>
__device__ __forceinline__ void transpose_swiglu_tile(uint32_t a_stage, uint32_t raw_g,
                                                      uint32_t raw_u, int q, int lane) {
#pragma unroll 1
  for (int j = q; j < BM / 32; j += 4) {
    const uint32_t n = (uint32_t)(j * 32 + lane);
    const uint32_t sg = raw_g + (uint32_t)j * 4096u;
    const uint32_t su = raw_u + (uint32_t)j * 4096u;
    const uint32_t col = ((uint32_t)lane >> 2), word = ((uint32_t)lane & 3u) * 4u;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
      uint32_t v[4];
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e) {
        const uint32_t k = 4 * c + e;
        const uint32_t off = k * 128u + ((col ^ (k & 7u)) << 4) + word;
        const float g = __uint_as_float(ld_shared_u32(sg + off));
        const float u = __uint_as_float(ld_shared_u32(su + off));
        v[e] = __float_as_uint(silu_stable(g) * u);
      }
      st_shared_v4(a_stage + sw128(n, c), v[0], v[1], v[2], v[3]);
    }
  }
}

// ---------------------------------------------------------------- cluster split K

// Partial tile of a cluster split in shared memory (at the start of the
// operand ring, idle once the accumulator is complete): [128 rows][BN f32],
// the 16-byte column c of row r at ((c ^ (r & 7)) * 16) within the row, so
// that the 32 lanes of a warp (32 rows) store one column without bank
// conflicts and consecutive threads of the sum read consecutive columns.
template <typename T>
__device__ __forceinline__ uint32_t csplit_off(int r, int c4) {
  return (uint32_t)(r * T::BN * 4 + ((c4 ^ (r & 7)) * 16));
}

// The sum of a cluster split: CTA `rank` of the S takes its share of the
// tile's 128 x BN/4 float4s (row-major, so that consecutive threads touch
// consecutive columns of a row) and adds the S partials in K order (rank 0
// first, as the split sum kernel does), then the residual or the SwiGLU
// backward, and writes Y (and Y2) with 16-byte global stores. Every warp of
// the CTA takes part (the roles are done by now), and each thread has two
// outputs' partials and residual rows in flight before the first add: the
// sum is a chain of distributed-shared-memory and global round trips, and
// with four warps and one output at a time it took longer than the main
// loop on the 512-token shapes.
template <typename T>
__device__ __forceinline__ void cluster_split_sum(uint32_t part, int S, int rank, int tid,
                                                  int nthreads, int m0, int n0,
                                                  const KernelArgs& args) {
  constexpr int C4 = T::BN / 4;
  constexpr int TOTAL = T::BM * C4;
  const int beg = rank * TOTAL / S, end = (rank + 1) * TOTAL / S;
  const bool swb = (args.flags & KFLAG_SWIGLU_BWD) != 0;
  for (int idx0 = beg + tid; idx0 < end; idx0 += 2 * nthreads) {
    float4 v[2][kMaxClusterSplit];
    float4 rv[2], gt[2], up[2];
    bool live[2];
    size_t o[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = idx0 + j * nthreads;
      const int r = idx / C4, c4 = idx % C4;
      const int row = m0 + r, col = n0 + 4 * c4;
      live[j] = idx < end && row < args.M && col < args.N;
      o[j] = live[j] ? (size_t)row * (size_t)args.N + (size_t)col : 0;
      if (!live[j]) continue;
      const uint32_t off = part + csplit_off<T>(r, c4);
      if (!dcheck(csplit_off<T>(r, c4) + 16 <= T::NS * T::OP_STAGE_BYTES && S <= kMaxClusterSplit,
                  args.status, CHK_BUFFER, csplit_off<T>(r, c4))) {
        live[j] = false;
        continue;
      }
#pragma unroll
      for (int p = 0; p < kMaxClusterSplit; ++p)
        if (p < S) v[j][p] = ld_cluster_v4f(mapa_shared(off, (uint32_t)p));
      if (swb) {
        gt[j] = *reinterpret_cast<const float4*>(args.G2 + o[j]);
        up[j] = *reinterpret_cast<const float4*>(args.U2 + o[j]);
      } else if constexpr (T::kResid) {
        rv[j] = *reinterpret_cast<const float4*>(args.R + o[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (!live[j]) continue;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int p = 0; p < kMaxClusterSplit; ++p) {
        if (p < S) {
          sum.x += v[j][p].x;
          sum.y += v[j][p].y;
          sum.z += v[j][p].z;
          sum.w += v[j][p].w;
        }
      }
      if (swb) {   // the SwiGLU backward of the summed dA
        float4 dg, du;
        swiglu_backward(sum.x, gt[j].x, up[j].x, dg.x, du.x);
        swiglu_backward(sum.y, gt[j].y, up[j].y, dg.y, du.y);
        swiglu_backward(sum.z, gt[j].z, up[j].z, dg.z, du.z);
        swiglu_backward(sum.w, gt[j].w, up[j].w, dg.w, du.w);
        *reinterpret_cast<float4*>(args.Y + o[j]) = dg;
        *reinterpret_cast<float4*>(args.Y2 + o[j]) = du;
        continue;
      }
      if constexpr (T::kResid) {
        sum.x += rv[j].x;
        sum.y += rv[j].y;
        sum.z += rv[j].z;
        sum.w += rv[j].w;
      }
      *reinterpret_cast<float4*>(args.Y + o[j]) = sum;
    }
  }
}

// ---------------------------------------------------------------- kernel

template <int AMODE, bool RESID, int BN, bool BT>
__global__ void __launch_bounds__(GemmTraits<AMODE, RESID, BN, BT>::kThreadsT, 1)
    lin_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_r,
                    const __grid_constant__ CUtensorMap tm_y,
                    const __grid_constant__ CUtensorMap tm_g2,
                    const __grid_constant__ CUtensorMap tm_u2,
                    const __grid_constant__ CUtensorMap tm_y2, const KernelArgs args) {
  using T = GemmTraits<AMODE, RESID, BN, BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + T::OFF_BAR;
  auto bar = [&](int slot) -> uint32_t { return bar0 + 8u * (uint32_t)slot; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::OFF_BAR + T::OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_BAR + T::OFF_ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * T::BM;
  const int nkb_all = (args.K + T::BK - 1) / T::BK;
  // Split K (gridDim.z = split_s > 1): this CTA accumulates k-blocks
  // [kb0, kb0 + nkb) and writes an f32 partial tile to args.part; a second
  // kernel adds the partials in K order (+ R) into Y.
  const bool split = gridDim.z > 1;
  // ... or, with KFLAG_CLUSTER_SPLIT, keeps it in shared memory for the
  // cluster's sum (cluster dims (1, 1, gridDim.z): CTA rank = blockIdx.z).
  const bool csplit = T::kClusterSplitOK && split && (args.flags & KFLAG_CLUSTER_SPLIT) != 0;
  const int kb0 = (int)blockIdx.z * nkb_all / (int)gridDim.z;
  const int nkb = ((int)blockIdx.z + 1) * nkb_all / (int)gridDim.z - kb0;
  const bool withhold = (args.flags & KFLAG_WITHHOLD_PRODUCER) != 0;
  const WaitCtl ctl{args.timeout_ns, abort_flag, args.status};
  // Checked build: a TMA copy's innermost coordinate x (elements of esz
  // bytes) on a 16-byte boundary; a ring slot inside its ring.
  auto x_ok = [&](int x, int esz) -> bool {
    return dcheck((x * esz) % 16 == 0, args.status, CHK_TMA_X, x);
  };
  auto slot_ok = [&](int slot, int n) -> bool {
    return dcheck(slot >= 0 && slot < n, args.status, CHK_STAGE, slot);
  };

  auto a_stage = [&](int s) -> uint32_t { return sbase + T::OFF_OP + s * T::OP_STAGE_BYTES; };
  auto b_stage = [&](int s) -> uint32_t { return a_stage(s) + T::A_BYTES; };
  auto raw_stage = [&](int r) -> uint32_t { return sbase + T::OFF_RAW + r * T::RAW_STAGE_BYTES; };

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int st = 0; st < T::NS; ++st) {
      mbar_init(bar(T::BAR_OP_TMA + st), 1);
      mbar_init(bar(T::BAR_OP_XF + st), T::XF_WARPS);   // one arrive per transform warp
      mbar_init(bar(T::BAR_OP_EMPTY + st), 1);    // tcgen05.commit
    }
    for (int r = 0; r < T::NR; ++r) {
      mbar_init(bar(T::BAR_RAW_FULL + r), 1);
      mbar_init(bar(T::BAR_RAW_EMPTY + r), T::XF_WARPS);
    }
    mbar_init(bar(T::BAR_ACC_FULL), 1);
    for (int e = 0; e < 8; ++e) mbar_init(bar(T::BAR_EPI + e), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();
  if (warp == 0 && lane == 0 && !withhold) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
    if constexpr (T::kSwiglu) tma_prefetch_desc(&tm_u);
    if constexpr (RESID) tma_prefetch_desc(&tm_r);
    tma_prefetch_desc(&tm_y);
    if (args.flags & KFLAG_SWIGLU_BWD) {
      tma_prefetch_desc(&tm_g2);
      tma_prefetch_desc(&tm_u2);
      tma_prefetch_desc(&tm_y2);
    }
  }
  __syncwarp();
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
    tmem_relinquish_alloc_permit();
  }
  // Launched as a programmatic dependent: the set-up above overlapped the
  // previous kernel on the stream; nothing below touches global memory
  // before that kernel has completed.
  pdl_wait();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Every role below runs with its whole warp converged: lane 0 waits and
  // issues, the other lanes follow it loop by loop, and no lane reaches the
  // final CTA barrier while a lane of its warp still has work in flight.
  // Operand-stage TMA producer (X for TF32, W for binary16): the stage's
  // boxes, A's and then W's, are issued by `nroles` warps, box i by role
  // i % nroles, and role 0 also announces the stage's bytes. Issuing a box
  // costs its thread about 70-120 cycles; the weight gradient's stage
  // (four boxes of X^T, four of W) paced its ring with one issuing thread,
  // and warp 3, free in that form, takes half (ffn_up_dw_f32 17.1 / 10.7 ->
  // 15.0 / 9.35 us cold / warm; the five-box stages of the forms that read
  // X gained nothing and keep one issuer).
  constexpr bool kIssueSplit = T::kAmn;
  auto produce = [&](int role, int nroles) {
    int filled = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % T::NS;
      const int n = kb / T::NS;
      if (kb >= T::NS && !lane0_wait_phase(bar(T::BAR_OP_EMPTY + st), (n - 1) & 1, ctl, lane))
        break;
      const int kk = (kb0 + kb) * T::BK;
      // (x of every copy below: kk along K, m0 + j*32 or n0 + j*W_ATOM along
      // M or N, all multiples of 16 bytes; a skipped copy makes the
      // stage's wait run out)
      const bool go = slot_ok(st, T::NS) && x_ok(kk, T::kBT ? T::ESZ : 4) && x_ok(m0, 4) &&
                      x_ok(n0, T::ESZ);
      if (lane == 0) {
        const uint32_t full = bar(T::BAR_OP_TMA + st);
        if (role == 0) mbar_arrive_expect_tx(full, T::OP_TMA_BYTES);
        int box = 0;
        auto issue = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
          if (box++ % nroles == role) tma_load_2d(dst, map, x, y, full);
        };
        if (go) {
          if constexpr (T::kAmn) {
            // X^T: BM/32 boxes of [32 rows of the contraction][32 of the tile's rows]
#pragma unroll
            for (int j = 0; j < T::BM / 32; ++j) issue(a_stage(st) + j * 4096, &tm_a, m0 + j * 32, kk);
          } else if constexpr (!T::kXformA) {
            issue(a_stage(st), &tm_a, kk, m0);
          }
          if constexpr (T::kBT) {
            // W as [N][K]: the tile's BN rows, this k-block's 128 bytes
            issue(b_stage(st), &tm_w, kk, n0);
          } else {
            // W as [K][N]: 128-byte runs of W_ATOM columns, BK rows each
#pragma unroll
            for (int j = 0; j < T::W_BOXES; ++j)
              issue(b_stage(st) + j * T::B_ATOM_BYTES, &tm_w, n0 + j * T::W_ATOM, kk);
          }
        }
      }
      __syncwarp();
      filled = kb + 1;
    }
    // Never leave with copies in flight: wait for the last fill of each slot.
    if (lane == 0)
      for (int kb = (filled > T::NS ? filled - T::NS : 0); kb < filled; ++kb)
        wait_phase(bar(T::BAR_OP_TMA + kb % T::NS), (kb / T::NS) & 1, ctl, false);
    __syncwarp();
  };

  if (warp == 0) {
    if (T::OP_TMA_BYTES > 0 && !withhold) produce(0, kIssueSplit ? 2 : 1);
  } else if (warp == 1) {
    // ---------------- UMMA issuer
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % T::NS;
      const uint32_t ph = (kb / T::NS) & 1;
      if (T::OP_TMA_BYTES > 0 && !lane0_wait_phase(bar(T::BAR_OP_TMA + st), ph, ctl, lane)) break;
      if (T::kXform && !lane0_wait_phase(bar(T::BAR_OP_XF + st), ph, ctl, lane)) break;
      const bool mma_ok = slot_ok(st, T::NS);   // (checked build; skipped UMMAs, not the commit)
      if (lane == 0) {
        tc_fence_after_sync();
#pragma unroll
        for (int k = 0; k < T::NMMA; ++k) {
          if (!mma_ok) break;
          // K-major A: a K step is 32 bytes along the row; MN-major X^T: KSTEP
          // rows of 128 bytes, runs of 32 tile rows 4096 bytes apart
          const uint64_t adesc =
              T::kAmn ? umma_desc_sw128_atom32(a_stage(st) + k * T::KSTEP * 128, 4096, 512)
                      : umma_desc_sw128(a_stage(st) + k * 32, 16, 1024);
          // W given as [N][K]: K-major. Else MN-major: a K step is KSTEP rows
          // of 128 bytes further; runs of W_ATOM columns B_ATOM_BYTES apart;
          // 8-row (binary16) or 4-row (TF32, 32-byte atoms) groups along K.
          const uint64_t bdesc =
              T::kBT ? umma_desc_sw128(b_stage(st) + k * 32, 16, 1024)
              : T::kF16
                  ? umma_desc_sw128(b_stage(st) + k * T::KSTEP * 128, T::B_ATOM_BYTES, 1024)
                  : umma_desc_sw128_atom32(b_stage(st) + k * T::KSTEP * 128, T::B_ATOM_BYTES,
                                           512);
          if constexpr (T::kF16)
            umma_f16(tmem, adesc, bdesc, T::IDESC, (kb | k) != 0);
          else
            umma_tf32(tmem, adesc, bdesc, T::IDESC, (kb | k) != 0);
        }
        umma_commit(bar(T::BAR_OP_EMPTY + st));   // frees the stage when these UMMAs finish
      }
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(bar(T::BAR_ACC_FULL));          // accumulator complete (or drained)
      // Keep TMEM allocated until every issued UMMA has finished.
      wait_phase(bar(T::BAR_ACC_FULL), 0, ctl, false);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ---------------- raw-stage TMA producer (inputs of the transform warps),
    // or the second issuer of the operand stages
    if (kIssueSplit && T::OP_TMA_BYTES > 0 && !withhold) produce(1, 2);
    if (T::kXform && !withhold) {
      const int nraw = nkb * T::RAW_PER_KB;
      int filled = 0;
      for (int t = 0; t < nraw; ++t) {
        const int r = t % T::NR;
        const int n = t / T::NR;
        if (t >= T::NR && !lane0_wait_phase(bar(T::BAR_RAW_EMPTY + r), (n - 1) & 1, ctl, lane))
          break;
        const int kk = (kb0 * T::RAW_PER_KB + t) * 32;   // f32 column of this raw stage
        const bool go = slot_ok(r, T::NR) && x_ok(kk, 4) && x_ok(m0, 4);
        if (lane == 0) {
          const uint32_t full = bar(T::BAR_RAW_FULL + r);
          mbar_arrive_expect_tx(full, T::RAW_STAGE_BYTES);
          if (!go) {
            // (checked build: the stage's wait runs out)
          } else if constexpr (T::kTransA) {
            // X^T: BM/32 boxes of [32 rows of the contraction][32 of the tile's rows]
#pragma unroll
            for (int j = 0; j < T::BM / 32; ++j) {
              tma_load_2d(raw_stage(r) + j * 4096, &tm_a, m0 + j * 32, kk, full);
              if constexpr (T::kSwiglu)
                tma_load_2d(raw_stage(r) + T::RAW_BOX_BYTES + j * 4096, &tm_u, m0 + j * 32, kk,
                            full);
            }
          } else if constexpr (T::kXformA) {
            tma_load_2d(raw_stage(r), &tm_a, kk, m0, full);
            if constexpr (T::kSwiglu)
              tma_load_2d(raw_stage(r) + T::RAW_BOX_BYTES, &tm_u, kk, m0, full);
          }
        }
        __syncwarp();
        filled = t + 1;
      }
      if (lane == 0)
        for (int t = (filled > T::NR ? filled - T::NR : 0); t < filled; ++t)
          wait_phase(bar(T::BAR_RAW_FULL + t % T::NR), (t / T::NR) & 1, ctl, false);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---------------- warps 4-7: transform, then epilogue (warps 8-11 of the
    // f32 SwiGLU form: transform only)
    const int q = warp - 4;                 // TMEM lane quadrant of this warp (warps 4-7)
    const int tid = threadIdx.x - 128;      // 0 .. 32 * XF_WARPS - 1
    bool ok = true;
    int t = 0;
    for (int kb = 0; kb < (T::kXform ? nkb : 0) && ok; ++kb) {
      const int st = kb % T::NS;
      const int n = kb / T::NS;
      if (kb >= T::NS && !warp_wait_phase(bar(T::BAR_OP_EMPTY + st), (n - 1) & 1, ctl)) {
        ok = false;
        break;
      }
#pragma unroll 1
      for (int h = 0; h < T::RAW_PER_KB; ++h, ++t) {
        const int r = t % T::NR;
        if (!warp_wait_phase(bar(T::BAR_RAW_FULL + r), (t / T::NR) & 1, ctl)) {
          ok = false;
          break;
        }
        if constexpr (T::kTransA && T::kSwiglu)
          transpose_swiglu_tile<T::BM>(a_stage(st), raw_stage(r),
                                       raw_stage(r) + T::RAW_BOX_BYTES, q, lane);
        else if constexpr (T::kTransA)
          transpose_tile<T::BM>(a_stage(st), raw_stage(r), q, lane);
        else if constexpr (T::kXformA)
          transform_raw_stage<AMODE, 32 * T::XF_WARPS>(a_stage(st), raw_stage(r), h, tid);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(T::BAR_RAW_EMPTY + r));
      }
      if (!ok) break;
      fence_proxy_async_smem();   // operand writes -> visible to the UMMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(T::BAR_OP_XF + st));
    }
    // The epilogue buffers alias the raw ring: every transform warp must be
    // done reading it first.
    named_bar_sync(1, 32 * T::XF_WARPS);
    if (warp < 8) {

    const int row0 = m0 + q * kEpiRows;
    const bool rows_in = row0 < args.M;      // a box starting past M would store nothing
    // checked build: chunk c's TMEM columns inside the accumulator
    auto tcol_ok = [&](int c) -> bool {
      return dcheck(c >= 0 && (c + 1) * kEpiCols <= BN, args.status, CHK_TMEM, c * kEpiCols);
    };
    const uint32_t buf0 = sbase + T::OFF_EPI + (uint32_t)(q * 2) * T::EPI_BUF_BYTES;
    const uint32_t ebar0 = bar(T::BAR_EPI + q * 2);
    constexpr int NC = BN / kEpiCols;
    int nc = (args.N - n0 + kEpiCols - 1) / kEpiCols;   // chunks inside N
    if (nc > NC) nc = NC;

    // Residual tiles are prefetched one chunk ahead; r_issued / r_done count
    // the chunks whose load was issued / waited for (lane 0's view).
    int r_issued = 0, r_done = 0;
    if (split) {
      // partial tile of (tile, K range): [BN/4 float4 columns][128 rows]
      ok = warp_wait_phase(bar(T::BAR_ACC_FULL), 0, ctl);
      tc_fence_after_sync();
      if (q == 0 && lane == 0) pdl_launch_dependents();   // the split sum may be scheduled
      ok = ok && !withhold && (__shfl_sync(0xffffffffu, *abort_flag, 0) == 0);
      if (ok && csplit) {
        const int r = q * kEpiRows + lane;
        for (int c = 0; c < nc; ++c) {
          uint32_t v[32];
          if (!tcol_ok(c)) break;
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * kEpiCols), v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (dcheck(csplit_off<T>(r, c * 8 + j) + 16 <= T::NS * T::OP_STAGE_BYTES, args.status,
                       CHK_BUFFER, csplit_off<T>(r, c * 8 + j)))
              st_shared_v4(sbase + T::OFF_OP + csplit_off<T>(r, c * 8 + j), v[4 * j + 0],
                           v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      } else if (ok) {
        const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
        float4* part = reinterpret_cast<float4*>(args.part) +
                       (tile * gridDim.z + blockIdx.z) * (BN / 4) * T::BM + q * kEpiRows + lane;
        const long long part_at = (long long)(tile * gridDim.z + blockIdx.z) * (BN / 4) * T::BM +
                                  q * kEpiRows + lane;
        for (int c = 0; c < nc; ++c) {
          uint32_t v[32];
          if (!tcol_ok(c)) break;
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * kEpiCols), v);
          tmem_wait_ld();
          if (!dcheck(part_at + (long long)(c * 8 + 7) * T::BM < args.part_f4, args.status,
                      CHK_PART, part_at + (long long)(c * 8 + 7) * T::BM))
            break;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            part[(size_t)(c * 8 + j) * T::BM] =
                make_float4(__uint_as_float(v[4 * j + 0]), __uint_as_float(v[4 * j + 1]),
                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
      ok = false;   // nothing below: no residual, no store of Y
    }
    if (!split && RESID && rows_in && !withhold && lane == 0 && nc > 0) {
      mbar_arrive_expect_tx(ebar0, T::EPI_BUF_BYTES);
      if (x_ok(n0, 4)) tma_load_2d(buf0, &tm_r, n0, row0, ebar0);
      r_issued = 1;
    }
    if (!split) {
      ok = warp_wait_phase(bar(T::BAR_ACC_FULL), 0, ctl);
      tc_fence_after_sync();
      if (q == 0 && lane == 0) pdl_launch_dependents();   // accumulator complete
      // After any role gave up (or in the self-test, whose tensor maps are
      // empty) the accumulator is not valid: store nothing.
      ok = ok && !withhold && (__shfl_sync(0xffffffffu, *abort_flag, 0) == 0);
    }
    int sw_issued = 0, sw_done = 0;   // GATE/UP chunk loads (lane 0's view)
    if (ok && rows_in && (args.flags & KFLAG_SWIGLU_BWD)) {
      // dA -> dGATE, dUP: GATE and UP arrive by TMA in the warp's two
      // buffers, the gradients replace them there and leave by TMA store
      const uint32_t bg = buf0, bu = buf0 + T::EPI_BUF_BYTES;
      for (int c = 0; c < nc; ++c) {
        if (lane == 0) {
          bulk_wait_group_read<0>();   // the last stores have read both buffers
          mbar_arrive_expect_tx(ebar0, 2 * T::EPI_BUF_BYTES);
          if (x_ok(n0 + c * kEpiCols, 4)) {
            tma_load_2d(bg, &tm_g2, n0 + c * kEpiCols, row0, ebar0);
            tma_load_2d(bu, &tm_u2, n0 + c * kEpiCols, row0, ebar0);
          }
          sw_issued = c + 1;
          if (c + 1 < nc) {   // the next chunk's GATE and UP into L2
            tma_prefetch_l2_2d(&tm_g2, n0 + (c + 1) * kEpiCols, row0);
            tma_prefetch_l2_2d(&tm_u2, n0 + (c + 1) * kEpiCols, row0);
          }
        }
        __syncwarp();
        uint32_t v[32];
        if (tcol_ok(c))
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * kEpiCols), v);
        tmem_wait_ld();
        if (!warp_wait_phase(ebar0, c & 1, ctl)) break;
        sw_done = c + 1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = sw128(lane, j);
          const float4 gt = ld_shared_v4f(bg + off);
          const float4 up = ld_shared_v4f(bu + off);
          float4 dg, du;
          swiglu_backward(__uint_as_float(v[4 * j + 0]), gt.x, up.x, dg.x, du.x);
          swiglu_backward(__uint_as_float(v[4 * j + 1]), gt.y, up.y, dg.y, du.y);
          swiglu_backward(__uint_as_float(v[4 * j + 2]), gt.z, up.z, dg.z, du.z);
          swiglu_backward(__uint_as_float(v[4 * j + 3]), gt.w, up.w, dg.w, du.w);
          st_shared_v4(bg + off, __float_as_uint(dg.x), __float_as_uint(dg.y),
                       __float_as_uint(dg.z), __float_as_uint(dg.w));
          st_shared_v4(bu + off, __float_as_uint(du.x), __float_as_uint(du.y),
                       __float_as_uint(du.z), __float_as_uint(du.w));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (x_ok(n0 + c * kEpiCols, 4)) {
            tma_store_2d(&tm_y, n0 + c * kEpiCols, row0, bg);
            tma_store_2d(&tm_y2, n0 + c * kEpiCols, row0, bu);
          }
          bulk_commit_group();
        }
      }
    } else if (ok && rows_in) {
      for (int c = 0; c < nc; ++c) {
        const int b = c & 1;
        const uint32_t buf = buf0 + b * T::EPI_BUF_BYTES;
        if (lane == 0 && c + 1 < nc) {
          // The other buffer's previous store must have read its source.
          bulk_wait_group_read<0>();
          if constexpr (RESID) {
            const uint32_t nb = ebar0 + 8u * (uint32_t)(b ^ 1);
            mbar_arrive_expect_tx(nb, T::EPI_BUF_BYTES);
            if (x_ok(n0 + (c + 1) * kEpiCols, 4))
              tma_load_2d(buf0 + (b ^ 1) * T::EPI_BUF_BYTES, &tm_r, n0 + (c + 1) * kEpiCols, row0,
                          nb);
            r_issued = c + 2;
          }
        }
        __syncwarp();
        uint32_t v[32];
        if (tcol_ok(c))
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * kEpiCols), v);
        tmem_wait_ld();
        if constexpr (RESID) {
          if (!warp_wait_phase(ebar0 + 8u * (uint32_t)b, (c >> 1) & 1, ctl)) break;
          r_done = c + 1;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t addr = buf + sw128(lane, j);
          float o0 = __uint_as_float(v[4 * j + 0]);
          float o1 = __uint_as_float(v[4 * j + 1]);
          float o2 = __uint_as_float(v[4 * j + 2]);
          float o3 = __uint_as_float(v[4 * j + 3]);
          if constexpr (RESID) {
            const float4 rr = ld_shared_v4f(addr);
            o0 += rr.x;
            o1 += rr.y;
            o2 += rr.z;
            o3 += rr.w;
          }
          st_shared_v4(addr, __float_as_uint(o0), __float_as_uint(o1), __float_as_uint(o2),
                       __float_as_uint(o3));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (x_ok(n0 + c * kEpiCols, 4)) tma_store_2d(&tm_y, n0 + c * kEpiCols, row0, buf);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) {
      // Never leave with a residual load in flight (only on the abort path
      // can one be outstanding).
      for (int c = r_done; c < r_issued; ++c)
        wait_phase(ebar0 + 8u * (uint32_t)(c & 1), (c >> 1) & 1, ctl, false);
      if (sw_issued > sw_done) wait_phase(ebar0, sw_done & 1, ctl, false);
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
    }
  }

  // ---- teardown (a cluster split first sums the partials: every CTA's is
  // complete after the first cluster barrier, and none may leave before the
  // second, while peers still read its shared memory)
  tc_fence_before_sync();
  if (csplit) {
    cluster_sync_all();
    if (!withhold)
      cluster_split_sum<T>(sbase + T::OFF_OP, (int)gridDim.z, (int)blockIdx.z, (int)threadIdx.x,
                           (int)blockDim.x, m0, n0, args);
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

// Host-side launcher of one instantiation.
template <int AMODE, bool RESID, int BN, bool BT = false>
cudaError_t launch_instance(const TensorMaps& m, const KernelArgs& args, cudaStream_t stream) {
  using T = GemmTraits<AMODE, RESID, BN, BT>;
  auto kern = lin_gemm_kernel<AMODE, RESID, BN, BT>;
  // The shared-memory opt-in is per device: remember which devices have it.
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit == 0 || !(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid((unsigned)((args.N + BN - 1) / BN), (unsigned)((args.M + kBM - 1) / kBM),
            (unsigned)(args.split_s > 1 ? args.split_s : 1));
  if (args.flags & KFLAG_WITHHOLD_PRODUCER) grid = dim3(1, 1, 1);
  const bool csplit = grid.z > 1 && (args.flags & KFLAG_CLUSTER_SPLIT) != 0;
  if (csplit && (grid.z > (unsigned)kMaxClusterSplit || !T::kClusterSplitOK))
    return cudaErrorInvalidValue;
  if (csplit && dev < 64) {
    // The largest split up to the one asked for whose clusters are all
    // resident at once (clusters of S CTAs of this size per GPC set the
    // limit; the K ranges follow gridDim.z).
    static std::atomic<int> caps[64][kMaxClusterSplit + 1];
    const unsigned tiles = grid.x * grid.y;
    while (grid.z > 2) {
      int n = caps[dev][grid.z].load(std::memory_order_relaxed);
      if (n == 0) {
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeClusterDimension;
        ca[0].val.clusterDim.x = 1;
        ca[0].val.clusterDim.y = 1;
        ca[0].val.clusterDim.z = grid.z;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(1, 1, grid.z);
        q.blockDim = dim3(T::kThreadsT, 1, 1);
        q.dynamicSmemBytes = T::SMEM_BYTES;
        q.attrs = ca;
        q.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, (void*)kern, &q);
        if (e != cudaSuccess) return e;
        n = n > 0 ? n : -1;
        caps[dev][grid.z].store(n, std::memory_order_relaxed);
      }
      if (n >= (int)tiles) break;
      --grid.z;
    }
  }
  // A programmatic dependent of the previous kernel on the stream (the
  // kernel waits for it in griddepcontrol.wait after its set-up).
  // With a cluster split, the CTAs of one tile form a cluster along z.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = grid.z;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(T::kThreadsT, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = csplit ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, m.a, m.u, m.w, m.r, m.y, m.g2, m.u2, m.y2, args);
}

}  // namespace lin
