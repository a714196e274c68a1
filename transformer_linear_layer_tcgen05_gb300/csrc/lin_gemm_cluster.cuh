// lin_gemm_cluster.cuh -- persistent, clustered tcgen05 GEMM for the
// binary16-weight forms whose A operand is built on chip:
//
//   matmul_residual_swiglu_a_w16   A = f16(silu(GATE) * UP)   (+ R)
//   matmul_w16 / _residual_w16     A = f16(X)                 (+ R)
//
// (page "matmul ve matmul_residual -- Tiled Matrix Multiply (Forward)",
// 03_linear_forward: "Ne Yapar?" and "Önemli Optimizasyonlar" 3).
//
// Why clusters: the A operand of an output row block is the same for every
// N tile. A cluster of CN CTAs side by side along N computes CN tiles of one
// row block at once; each CTA transforms only 128/CN rows of every A
// k-block and writes them into the A stage of every CTA of the cluster
// through distributed shared memory, so each GATE/UP element is read from L2
// and transformed once per cluster instead of once per tile.
//
// Per CTA: a 128 x BN output tile per work item, persistent over work items
// (cluster tiles in a static round-robin), accumulator double-buffered in
// TMEM (2 x BN columns) so the epilogue of one tile overlaps the main loop
// of the next. Sixteen warps:
//   warp 0      TMA producer of the binary16 W tiles (MN-major B operand)
//   warp 1      UMMA issuer; its per-stage commit is multicast to the whole
//               cluster (a stage may be refilled once every CTA read it)
//   warp 2      TMEM allocator (warps 2 and 3 are otherwise idle)
//   warps 4-11  transform, two groups of four taking turns by k-block: each
//               warp loads its rows of GATE/UP (or X) with coalesced 16-byte
//               global loads into registers, several of its k-blocks ahead,
//               turns them into binary16 A rows (silu(GATE)*UP, or X),
//               writes them into the local A stage and bulk-copies them (TMA
//               engine, shared to shared) into the same stage of every other
//               CTA of the cluster; the copies complete on the receiver's
//               full barrier
//   warps 12-15 epilogue: TMEM -> registers, + R, Y; each thread owns one
//               output row and moves it with 16-byte global loads/stores
// The f32 inputs are staged in registers rather than shared memory: the
// register file is as large as shared memory, and shared memory is then left
// whole to the operand ring, whose depth has to cover the round trip of a
// stage (W load or peer copies, UMMA, commit to every CTA).
#pragma once

#include <atomic>

#include "lin_common.cuh"

#ifndef LIN_XF_WARPS
#define LIN_XF_WARPS 8
#endif
#ifndef LIN_W_STAGES
#define LIN_W_STAGES 4
#endif

namespace lin {

// BT: W given as [N][K] (K contiguous, the backward product dY · W^T): its
// tiles are a K-major B operand, one TMA box of BN rows per k-block.
// DUAL: two products of the same A, Y = A @ W and Y2 = A @ W2 (the FFN's
// gate and up projections from one read of X): the B stage holds BN/2
// columns of W and the same BN/2 columns of W2 side by side, so one UMMA of
// N = BN computes both tiles; each CTA then covers BN/2 output columns.
template <int AMODE, bool RESID, int BN_, int CN_, bool V8_ = false, bool BT_ = false,
          bool DUAL_ = false>
struct ClusterTraits {
  static_assert(AMODE == A_CVT_F16 || AMODE == A_SWIGLU_F16 || AMODE == A_TMA_F16,
                "binary16 forms only");
  static constexpr bool kSwiglu = (AMODE == A_SWIGLU_F16);
  // A already binary16 in global memory: the CTA copies every A k-block of
  // its tile by TMA; no transform warps. Such a CTA has no A to share with
  // peers: it runs alone (CN_ == 1) or as one of a CTA pair (CN_ == 2).
  static constexpr bool kTmaA = (AMODE == A_TMA_F16);
  // CTA pair: the two CTAs of a cluster of two compute one 256 x BN tile
  // with UMMAs of M = 256 (tcgen05 .cta_group::2), issued by the even CTA.
  // Each CTA loads its 128 rows of A and half of the tile's W columns (the
  // even CTA the first half), so that W's bytes per CTA and k-block halve,
  // and keeps its 128 rows of the accumulator in its own TMEM.
  static constexpr bool kPair = kTmaA && CN_ == 2;
  static constexpr int BM = kBM;                  // rows of A and of the accumulator per CTA
  static constexpr int TM = kPair ? 2 * kBM : kBM;   // rows of a tile
  static constexpr int BN = BN_;
  static constexpr int CN = kPair ? 1 : CN_;      // CTAs per cluster along N
  static constexpr int CS = CN_;                  // CTAs per cluster
  static constexpr int BNB = kPair ? BN_ / 2 : BN_;   // W columns in this CTA's B stage
  static constexpr int BK = 64;                   // binary16 elements per k-block
  static constexpr int KSTEP = 16;
  static constexpr int NMMA = BK / KSTEP;
  static constexpr int W_ATOM = 64;
  static constexpr bool kBT = BT_;
  static constexpr bool kDual = DUAL_;
  static constexpr int BNO = kDual ? BN_ / 2 : BN_;   // output columns per CTA and product
  static constexpr int W_BOXES = kBT ? 1 : BNB / W_ATOM;
  static constexpr int ROWS = BM / CN;            // A rows this CTA transforms
  static constexpr int INPUTS = kSwiglu ? 2 : 1;  // GATE and UP, or X
  static constexpr int XF_WARPS = kTmaA ? 0 : LIN_XF_WARPS;
  // The transform warps form XF_GROUPS groups that take turns by k-block, so
  // each warp's fixed cost per k-block (a barrier wait, a proxy fence, the
  // copy issue) is spread over XF_GROUPS k-blocks of UMMA time. A single CTA
  // transforming all 128 rows of the SwiGLU form keeps one group, so that a
  // warp's share of a k-block still fits its registers.
  static constexpr int XF_GROUPS = kTmaA ? 1 : ((kSwiglu && CN == 1) ? 1 : XF_WARPS / 4);
  static constexpr int XF_PER_GROUP = kTmaA ? 1 : XF_WARPS / XF_GROUPS;
  static constexpr int RW = ROWS / XF_PER_GROUP;  // A rows per transform warp (contiguous)
  // Each transform warp bulk-copies its RW rows of a stage to every peer as
  // soon as it has written them (measured faster than one copy per group).
  static constexpr uint32_t SLICE_BYTES = RW * 128;
  static constexpr uint32_t REMOTE_BYTES_PER_WARP = SLICE_BYTES * (CN - 1);

  // A lane loads CHUNK consecutive f32 of one row per instruction: 4 (16-byte
  // loads) or, when the inputs allow 32-byte loads, 8, which make one
  // 16-byte binary16 chunk of the A row. A warp instruction covers
  // ROWS_PER_LOAD rows of a 64-wide k-block: LPI loads per input and lane.
  static constexpr bool V8 = V8_;
  static constexpr int CHUNK = V8 ? 8 : 4;
  static constexpr int LANES_PER_ROW = 64 / CHUNK;
  static constexpr int ROWS_PER_LOAD = 32 / LANES_PER_ROW;
  static constexpr int LPI = RW / ROWS_PER_LOAD;
  static constexpr int LOADS = INPUTS * LPI * (CHUNK / 4);   // float4 registers per lane per k-block
  // Register prefetch depth, in the group's own k-blocks: as many as fit in
  // the registers a lane can give to staged input (64 with 16 warps).
  // Measured and left out: twice the depth (registers moved from the other
  // warpgroups with setmaxnreg), twelve transform warps in three groups, and
  // GATE/UP resident in L2 all left the time of the loads unchanged.
  static constexpr int STAGE_REGS = XF_WARPS > 8 ? 32 : 64;   // per lane, for staged input
  static constexpr int PF_FIT = STAGE_REGS / (4 * LOADS);
  static constexpr int PF = PF_FIT < 1 ? 1 : (PF_FIT > 4 ? 4 : PF_FIT);
  // The transform's cursor and the lane's load addresses are kept from one
  // k-block to the next (LaneRows) where the staged registers leave room
  // for them; elsewhere they are computed per k-block.
  static constexpr bool kLaneRows = LOADS <= 8;

  static constexpr uint32_t A_BYTES = BM * 128;
  static constexpr uint32_t B_ATOM_BYTES = kBT ? BNB * 128 : BK * 128;
  static constexpr uint32_t B_BYTES = W_BOXES * B_ATOM_BYTES;

  // Split rings: the SwiGLU form in clusters, whose A stage makes the
  // longest round trip. A stage of its W ring is refilled as soon as this
  // CTA's UMMA has read it (a TMA load from L2: a round trip of about three
  // k-blocks of UMMA time); a stage of its A ring only once every CTA of the
  // cluster has read its copy, and then takes the transform's store and the
  // copies to the peers (about five k-blocks). So its W ring keeps
  // LIN_W_STAGES stages, one full and one empty barrier each, and its A ring
  // takes what shared memory is left. Every other form keeps one ring: a
  // stage of A and of W share one full barrier (the W tile's TMA bytes, the
  // transform group's arrivals, the peers' copied rows) and one empty
  // barrier, so the UMMA thread waits and commits once per k-block (two
  // rings measured slower there: 834 against 934 us on the gate/up pair).
  static constexpr bool kSplit = kSwiglu && CN > 1;

  // Epilogue staging: [32 rows][32 f32] swizzled buffers, EPI_BUFS per
  // epilogue warp. R arrives in them by TMA, the accumulator is added in
  // place and Y leaves by TMA store, so that the epilogue moves whole
  // 128-byte lines instead of one 16-byte piece per row and lane. Two per
  // warp, so that a chunk's R load (or the transposed product's SwiGLU
  // backward's GATE and UP) overlaps the previous chunk's store; the split
  // rings' form keeps one: with K = d_ff its epilogue has a long main loop
  // to overlap, and the shared memory goes to its A ring.
  static constexpr int EPI_BUFS = kSplit ? 1 : 2;
  static constexpr uint32_t EPI_BUF_BYTES = kEpiRows * kEpiCols * 4;   // 4 KB
  static constexpr uint32_t EPI_BYTES = 4 * EPI_BUFS * EPI_BUF_BYTES;

  static constexpr uint32_t SMEM_CAP = 232448;
  static constexpr uint32_t BAR_REGION = 1024;
  static constexpr uint32_t ALIGN_SLACK = 1024;
  static constexpr uint32_t DATA_CAP = SMEM_CAP - BAR_REGION - ALIGN_SLACK - EPI_BYTES;
  static constexpr int NS_FIT = (int)(DATA_CAP / (A_BYTES + B_BYTES));
  static constexpr int NW = kSplit ? LIN_W_STAGES : (NS_FIT > 8 ? 8 : NS_FIT);
  static constexpr int NA_FIT = (int)((DATA_CAP - NW * B_BYTES) / A_BYTES);
  static constexpr int NA = kSplit ? (NA_FIT > 8 ? 8 : NA_FIT) : NW;

  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_W = OFF_A + NA * A_BYTES;
  static constexpr uint32_t OFF_EPI = OFF_W + NW * B_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_EPI + EPI_BYTES;
  static constexpr uint32_t SMEM_BYTES = ALIGN_SLACK + OFF_BAR + BAR_REGION;

  static constexpr int BAR_AFULL = 0;
  static constexpr int BAR_AEMPTY = BAR_AFULL + 8;       // every CTA's UMMA done with the A stage
  static constexpr int BAR_WFULL = BAR_AEMPTY + 8;
  static constexpr int BAR_WEMPTY = BAR_WFULL + 8;       // this CTA's UMMA done with the W stage
  static constexpr int BAR_ACC_FULL = BAR_WEMPTY + 8;    // 2 accumulator buffers
  static constexpr int BAR_ACC_EMPTY = BAR_ACC_FULL + 2;
  static constexpr int BAR_EPI = BAR_ACC_EMPTY + 2;      // R landed, EPI_BUFS per epilogue warp
  static constexpr int BAR_COUNT = BAR_EPI + 8;
  static constexpr uint32_t OFF_TMEM_SLOT = BAR_COUNT * 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;

  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t IDESC = umma_idesc(0u, false, /*b_mn_major=*/!kBT, TM, BN);
  static constexpr uint16_t CLUSTER_MASK = (uint16_t)((1u << CS) - 1u);
  static constexpr int kThreadsC = (8 + XF_WARPS) * 32;

  static_assert(CN == 1 || CN == 2 || CN == 4 || CN == 8, "cluster size");
  static_assert(!kTmaA || CS == 1 || kPair,
                "a binary16 A from global memory: single CTAs or CTA pairs");
  static_assert(!kPair || (!kDual || BN == 256), "pair: the dual form's halves are its two products");
  static_assert(kTmaA || XF_WARPS == 4 || XF_WARPS == 8 || XF_WARPS == 12, "transform warps");
  static_assert(XF_WARPS % XF_GROUPS == 0 && ROWS % XF_PER_GROUP == 0 &&
                    RW % ROWS_PER_LOAD == 0,
                "transform groups");
  static_assert(kTmaA || LOADS <= 16, "staged input per lane");
  // A parity wait is only sound for a waiter at most one phase ahead: a group
  // reaching use u of a stage must already have seen use u-1's UMMA
  // complete, true when its previous k-block (XF_GROUPS earlier) waited for
  // a UMMA no older than the stage's use before last.
  static_assert(XF_GROUPS <= NA, "ring depth vs transform groups");
  static_assert(NA >= 2 && NA <= 8 && NW >= 2 && NW <= 8, "ring depths");
  static_assert(kSplit || NA == NW, "one ring: A and W stages in step");
  static_assert(OFF_ABORT + 4 <= BAR_REGION, "barrier region");
  static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
  // A CTA holding all 512 TMEM columns must be alone on its SM (a second one
  // would wait in tcgen05.alloc while its cluster peers wait for it).
  static_assert(TMEM_COLS < 512 || 2 * SMEM_BYTES > SMEM_CAP + BAR_REGION, "one CTA per SM");
};

// Register-staged inputs of one k-block for one transform lane: load q of
// input i is row (tw*RW + q*ROWS_PER_LOAD + lane/LANES_PER_ROW) of this
// CTA's slice, columns k0 + CHUNK*(lane%LANES_PER_ROW) onwards. Rows at or
// past M and columns at or past K read as zero (K is a multiple of CHUNK on
// each path, so a load is wholly in or out).
template <typename T>
struct Staged {
  float4 v[T::INPUTS][T::LPI][T::CHUNK / 4];
};

template <typename T>
__device__ __forceinline__ void stage_load(Staged<T>& st, const float* __restrict__ a,
                                           const float* __restrict__ u, int row0, int k0,
                                           int M, int K, int tw, int lane, int* status) {
  const int col = k0 + T::CHUNK * (lane % T::LANES_PER_ROW);
  // (K is a multiple of CHUNK on each path: a load is wholly in or out)
  const bool col_in = col < K && dcheck(col + T::CHUNK <= K, status, CHK_GLOBAL, col);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < T::LPI; ++q) {
    const int row = row0 + tw * T::RW + q * T::ROWS_PER_LOAD + lane / T::LANES_PER_ROW;
    const bool in = col_in && row < M;
    const size_t off = (size_t)(in ? row : 0) * (size_t)K + (size_t)(in ? col : 0);
#pragma unroll
    for (int i = 0; i < T::INPUTS; ++i) {
      const float* src = (i == 0 ? a : u) + off;
      if constexpr (T::V8) {
        if (in)
          ldg_stream_v8f(src, st.v[i][q][0], st.v[i][q][1]);
        else
          st.v[i][q][0] = st.v[i][q][1] = zero;
      } else {
        st.v[i][q][0] = in ? ldg_stream_v4f(src) : zero;
      }
    }
  }
}

// The same loads with this lane's first row offset (row * K + its first
// column), the row stride of its loads and the rows left before M computed
// once per work item: per k-block only k0 is added.
struct LaneRows {
  size_t off0;      // first load's row * K + column
  size_t stride;    // ROWS_PER_LOAD * K
  int rows_left;    // M - the first load's row
  int col;          // this lane's first column within a k-block
};

template <typename T>
__device__ __forceinline__ void lane_rows(LaneRows& lr, int row0, int M, int K, int tw,
                                          int lane) {
  lr.col = T::CHUNK * (lane % T::LANES_PER_ROW);
  const int row = row0 + tw * T::RW + lane / T::LANES_PER_ROW;
  lr.rows_left = M - row;
  lr.off0 = (size_t)row * (size_t)K + (size_t)lr.col;
  lr.stride = (size_t)T::ROWS_PER_LOAD * (size_t)K;
}

template <typename T>
__device__ __forceinline__ void stage_load_at(Staged<T>& st, const float* __restrict__ a,
                                              const float* __restrict__ u, const LaneRows& lr,
                                              int k0, int K, int* status) {
  const int col = k0 + lr.col;
  // (K is a multiple of CHUNK on each path: a load is wholly in or out)
  const bool col_in = col < K && dcheck(col + T::CHUNK <= K, status, CHK_GLOBAL, col);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < T::LPI; ++q) {
    const bool in = col_in && q * T::ROWS_PER_LOAD < lr.rows_left;
    const size_t off = in ? lr.off0 + (size_t)q * lr.stride + (size_t)k0 : 0;
#pragma unroll
    for (int i = 0; i < T::INPUTS; ++i) {
      const float* src = (i == 0 ? a : u) + off;
      if constexpr (T::V8) {
        if (in)
          ldg_stream_v8f(src, st.v[i][q][0], st.v[i][q][1]);
        else
          st.v[i][q][0] = st.v[i][q][1] = zero;
      } else {
        st.v[i][q][0] = in ? ldg_stream_v4f(src) : zero;
      }
    }
  }
}

// A values of the staged k-block as binary16 pairs: out[q] holds CHUNK
// consecutive k (CHUNK/2 words).
template <typename T>
__device__ __forceinline__ void stage_compute(const Staged<T>& st,
                                              uint32_t (&out)[T::LPI][T::CHUNK / 2]) {
#pragma unroll
  for (int q = 0; q < T::LPI; ++q) {
#pragma unroll
    for (int h = 0; h < T::CHUNK / 4; ++h) {
      float4 a = st.v[0][q][h];
      if constexpr (T::kSwiglu) {
        const float4 u = st.v[1][q][h];
        a.x = silu_stable_fast(a.x) * u.x;
        a.y = silu_stable_fast(a.y) * u.y;
        a.z = silu_stable_fast(a.z) * u.z;
        a.w = silu_stable_fast(a.w) * u.w;
      }
      out[q][2 * h] = pack_half2(a.x, a.y);
      out[q][2 * h + 1] = pack_half2(a.z, a.w);
    }
  }
}

// Into the A stage (128 rows x 128 bytes, 128-byte swizzle); this CTA's
// slice starts at row crank*ROWS. With 32-byte loads a lane stores one whole
// 16-byte chunk and a warp covers four rows; with 16-byte loads it stores
// half a chunk (lane%16 is the 8-byte quarter-pair) and a warp covers two
// rows. Either way each row's bytes spread over all 32 banks once.
template <typename T>
__device__ __forceinline__ void stage_store(uint32_t a_stage, uint32_t crank, int tw, int lane,
                                            const uint32_t (&out)[T::LPI][T::CHUNK / 2],
                                            int* status) {
  const uint32_t c = (uint32_t)(lane % T::LANES_PER_ROW);
#pragma unroll
  for (int q = 0; q < T::LPI; ++q) {
    const uint32_t r = crank * (uint32_t)T::ROWS +
                       (uint32_t)(tw * T::RW + q * T::ROWS_PER_LOAD + lane / T::LANES_PER_ROW);
    if (!dcheck(r < (uint32_t)T::BM, status, CHK_STAGE, r)) continue;
    if constexpr (T::V8)
      st_shared_v4(a_stage + sw128(r, c), out[q][0], out[q][1], out[q][2], out[q][3]);
    else
      st_shared_v2(a_stage + sw128(r, c >> 1) + (c & 1u) * 8u, out[q][0], out[q][1]);
  }
}

template <int AMODE, bool RESID, int BN, int CN, bool V8, bool BT, bool DUAL>
__global__ void __launch_bounds__(ClusterTraits<AMODE, RESID, BN, CN, V8, BT, DUAL>::kThreadsC, 1)
    lin_gemm_cluster_kernel(const __grid_constant__ CUtensorMap tm_w,
                            const __grid_constant__ CUtensorMap tm_w2,
                            const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ CUtensorMap tm_r,
                            const __grid_constant__ CUtensorMap tm_y,
                            const __grid_constant__ CUtensorMap tm_g2,
                            const __grid_constant__ CUtensorMap tm_u2,
                            const __grid_constant__ CUtensorMap tm_y2, const KernelArgs args) {
  using T = ClusterTraits<AMODE, RESID, BN, CN, V8, BT, DUAL>;
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
  const uint32_t crank = (T::CS > 1) ? cluster_ctarank() : 0u;
  const int cid = blockIdx.x / T::CS;               // cluster id
  const int ncl = gridDim.x / T::CS;                // clusters in the grid
  const int num_m = (args.M + T::TM - 1) / T::TM;
  const int num_ng = (args.N + T::BNO * T::CN - 1) / (T::BNO * T::CN);
  const int num_tiles = num_m * num_ng;
  const int nkb = (args.K + T::BK - 1) / T::BK;
  const WaitCtl ctl{args.timeout_ns, abort_flag, args.status};

  auto a_stage = [&](int s) -> uint32_t { return sbase + T::OFF_A + s * T::A_BYTES; };
  auto b_stage = [&](int s) -> uint32_t { return sbase + T::OFF_W + s * T::B_BYTES; };
  // this CTA's first row and column of tile t (a pair's CTAs: rows apart)
  auto tile_m0 = [&](int t) -> int {
    return tile_coords(t, num_m, num_ng, args.band_ng).m * T::TM +
           (T::kPair ? (int)crank * T::BM : 0);
  };
  auto tile_n0 = [&](int t) -> int {
    return (tile_coords(t, num_m, num_ng, args.band_ng).ng * T::CN + (T::kPair ? 0 : (int)crank)) *
           T::BNO;
  };
  // Work items of this cluster: whole tiles cid + i*ncl, round robin; with a
  // split tail (split_s >= 2), split_r whole tiles and then, for clusters
  // below split_rem*split_s, K range `unit_p` of tail tile split_r*ncl +
  // cid/split_s (unit index = cid).
  const bool split = args.split_s >= 2;
  const int S = split ? args.split_s : 1;
  const int n_full =
      split ? args.split_r : (cid < num_tiles ? (num_tiles - 1 - cid) / ncl + 1 : 0);
  const bool has_unit = split && cid < args.split_rem * S;
  const int n_items = n_full + (has_unit ? 1 : 0);
  const int unit_p = cid % S;
  const int unit_kb0 = unit_p * nkb / S;
  const int unit_kb1 = (unit_p + 1) * nkb / S;
  auto item_tile = [&](int i) -> int {
    return i < n_full ? cid + i * ncl : args.split_r * ncl + cid / S;
  };
  auto item_kb0 = [&](int i) -> int { return i < n_full ? 0 : unit_kb0; };
  auto item_kb1 = [&](int i) -> int { return i < n_full ? nkb : unit_kb1; };

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < T::NA; ++s) {
      // the transform group's warps, and with one ring the producer (its
      // W bytes, or a binary16 A and W from global memory; a pair's stages
      // fill on the even CTA's barrier, whose producer expects both CTAs'
      // bytes)
      mbar_init(bar(T::BAR_AFULL + s), T::kTmaA ? 1 : (T::kSplit ? 0 : 1) + T::XF_PER_GROUP);
      mbar_init(bar(T::BAR_AEMPTY + s), T::CN);    // every UMMA-issuing CTA's commit
    }
    if constexpr (T::kSplit)
      for (int s = 0; s < T::NW; ++s) {
        mbar_init(bar(T::BAR_WFULL + s), 1);       // the producer's TMA bytes
        mbar_init(bar(T::BAR_WEMPTY + s), 1);      // this CTA's UMMA commit
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(T::BAR_ACC_FULL + b), 1);
      // the epilogue warps (a pair's: of both CTAs, on the even CTA's barrier)
      mbar_init(bar(T::BAR_ACC_EMPTY + b), T::kPair ? 8 : 4);
    }
    for (int e = 0; e < 8; ++e) mbar_init(bar(T::BAR_EPI + e), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    if constexpr (T::kTmaA) tma_prefetch_desc(&tm_a);
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
    if constexpr (T::kPair) {   // both CTAs together: the same columns in each
      tmem_alloc_pair(smem_u32(tmem_slot), T::TMEM_COLS);
      tmem_relinquish_alloc_permit_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
      tmem_relinquish_alloc_permit();
    }
  }
  // Launched as a programmatic dependent: the set-up above overlapped the
  // previous kernel on the stream; nothing below touches global memory
  // before that kernel has completed.
  pdl_wait();
  if (args.zero_word && blockIdx.x == 0 && threadIdx.x == 0) *args.zero_word = 0u;
  tc_fence_before_sync();
  // Peers may arrive on our barriers and write our A stages only after every
  // CTA of the cluster initialised them.
  if constexpr (T::CS > 1)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- W producer (local TMA into the B half of each stage);
    // with a binary16 A in global memory also the tile's rows of A
    int g = 0;   // k-blocks issued, across tiles
    bool ok = true;
    for (int i = 0; i < n_items && ok; ++i) {
      const int t = item_tile(i);
      const int n0 = tile_n0(t);
      const int kb1 = item_kb1(i);
      for (int kb = item_kb0(i); kb < kb1; ++kb, ++g) {
        // one ring: the stage's single barriers (every CTA's UMMA done with
        // it; its TMA bytes, A's too when A comes from global memory)
        const int s = g % T::NW;
        const uint32_t wempty = bar((T::kSplit ? T::BAR_WEMPTY : T::BAR_AEMPTY) + s);
        const uint32_t full = bar((T::kSplit ? T::BAR_WFULL : T::BAR_AFULL) + s);
        if (g >= T::NW) {
          bool w = true;
          if (lane == 0)
            w = T::kSplit ? wait_phase(wempty, ((g / T::NW) - 1) & 1, ctl)
                          : wait_phase_cluster(wempty, ((g / T::NW) - 1) & 1, ctl);
          if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
            ok = false;
            break;
          }
        }
        if (lane == 0) {
          constexpr uint32_t bytes = T::B_BYTES + (T::kTmaA ? T::A_BYTES : 0u);
          // A pair's stage is full on the even CTA's barrier: its producer
          // alone arrives, expecting both CTAs' bytes, and the odd CTA's
          // loads complete there too. (Those may land before that arrival:
          // the transaction count runs below zero for a while, but the
          // phase cannot complete without the arrival. An arrival from the
          // odd CTA as well -- a remote arrive with release at cluster
          // scope -- took ~0.4 us per stage to issue and paced the ring.)
          const uint32_t full0 = T::kPair ? mapa_shared(full, 0) : full;
          if (!T::kPair)
            mbar_arrive_expect_tx(full, bytes);
          else if (crank == 0)
            mbar_arrive_expect_tx(full, 2 * bytes);
          auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
            // every map here holds binary16: x a multiple of 8 elements
            if (!dcheck((x & 7) == 0, args.status, CHK_TMA_X, x)) return;
            if (!dcheck(dst >= sbase + T::OFF_A && dst < sbase + T::OFF_EPI, args.status,
                        CHK_STAGE, (long long)(dst - sbase)))
              return;
            if constexpr (T::kPair)
              tma_load_2d_pair(dst, map, x, y, full0);
            else
              tma_load_2d(dst, map, x, y, full);
          };
          // this CTA's columns of the tile's B: all, or a pair's half
          const int nb = T::kPair && !T::kDual ? n0 + (int)crank * T::BNB : n0;
          if constexpr (T::kBT) {
            load(b_stage(s), &tm_w, kb * T::BK, nb);   // W as [N][K]
          } else if constexpr (T::kDual && T::kPair) {
            // the pair's B is [W tile | W2 tile]: the even CTA's half is W's
#pragma unroll
            for (int j = 0; j < T::W_BOXES; ++j)
              load(b_stage(s) + j * T::B_ATOM_BYTES, crank == 0 ? &tm_w : &tm_w2,
                   n0 + j * T::W_ATOM, kb * T::BK);
          } else if constexpr (T::kDual) {   // [W tile | W2 tile], BN/2 columns each
#pragma unroll
            for (int j = 0; j < T::W_BOXES; ++j) {
              const int jj = j % (T::W_BOXES / 2);
              load(b_stage(s) + j * T::B_ATOM_BYTES, j < T::W_BOXES / 2 ? &tm_w : &tm_w2,
                   n0 + jj * T::W_ATOM, kb * T::BK);
            }
          } else {
#pragma unroll
            for (int j = 0; j < T::W_BOXES; ++j)
              load(b_stage(s) + j * T::B_ATOM_BYTES, &tm_w, nb + j * T::W_ATOM, kb * T::BK);
          }
          if constexpr (T::kTmaA) load(a_stage(s), &tm_a, kb * T::BK, tile_m0(t));
        }
        __syncwarp();
      }
    }
    // no TMA load of ours may still be in flight when the CTA leaves (a
    // pair's odd CTA: its loads have landed once the UMMA that read them
    // has released the stage)
    if (lane == 0) {
      for (int x = (g > T::NW ? g - T::NW : 0); x < g; ++x) {
        if (T::kPair && crank != 0)
          wait_phase_cluster(bar(T::BAR_AEMPTY + x % T::NW), (x / T::NW) & 1, ctl, false);
        else
          wait_phase(bar((T::kSplit ? T::BAR_WFULL : T::BAR_AFULL) + x % T::NW), (x / T::NW) & 1,
                     ctl, false);
      }
    }
    __syncwarp();
  } else if (warp == 1 && (!T::kPair || crank == 0)) {
    // ---------------- UMMA issuer (a pair's: in the even CTA, for both)
    // A pair's barriers here see the odd CTA's arrivals and bytes too: the
    // waits acquire at cluster scope, and the commits reach both CTAs.
    auto wait_local = [&](uint32_t b, uint32_t parity) -> bool {
      return T::kPair ? wait_phase_cluster(b, parity, ctl) : wait_phase(b, parity, ctl);
    };
    auto commit_local = [&](uint32_t b) {
      if constexpr (T::kPair)
        umma_commit_pair(b, T::CLUSTER_MASK);
      else
        umma_commit(b);
    };
    int g = 0;
    bool ok = true;
    int committed_tiles = 0;
    for (int i = 0; i < n_items && ok; ++i) {
      const int ab = i & 1;
      const uint32_t d_tmem = tmem + (uint32_t)(ab * T::BN);
      if (i >= 2) {
        bool w = true;
        if (lane == 0) w = wait_local(bar(T::BAR_ACC_EMPTY + ab), ((i >> 1) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      const int kb0 = item_kb0(i), kb1 = item_kb1(i);
      for (int kb = kb0; kb < kb1; ++kb, ++g) {
        const int sa = g % T::NA;
        const int s = g % T::NW;
        bool w = true;
        if (lane == 0) {
          w = wait_local(bar(T::BAR_AFULL + sa), (g / T::NA) & 1) &&
              (!T::kSplit || wait_phase(bar(T::BAR_WFULL + s), (g / T::NW) & 1, ctl));
        }
        if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        // (checked build: the stages and the accumulator's columns in range;
        // a failed check skips the UMMAs, not the commit)
        const bool mma_ok =
            dcheck(sa < T::NA && s < T::NW, args.status, CHK_STAGE, g) &&
            dcheck((ab + 1) * T::BN <= (int)T::TMEM_COLS, args.status, CHK_TMEM, ab * T::BN);
        if (lane == 0) {
          tc_fence_after_sync();
#pragma unroll
          for (int k = 0; k < T::NMMA; ++k) {
            if (!mma_ok) break;
            const uint64_t adesc = umma_desc_sw128(a_stage(sa) + k * 32, 16, 1024);
            const uint64_t bdesc =
                T::kBT ? umma_desc_sw128(b_stage(s) + k * 32, 16, 1024)
                       : umma_desc_sw128(b_stage(s) + k * T::KSTEP * 128, T::B_ATOM_BYTES, 1024);
            if constexpr (T::kPair)
              umma_f16_pair(d_tmem, adesc, bdesc, T::IDESC, kb != kb0 || k != 0);
            else
              umma_f16(d_tmem, adesc, bdesc, T::IDESC, kb != kb0 || k != 0);
          }
          if constexpr (T::CN > 1)
            umma_commit_multicast(bar(T::BAR_AEMPTY + sa), T::CLUSTER_MASK);
          else
            commit_local(bar(T::BAR_AEMPTY + sa));
          if constexpr (T::kSplit) umma_commit(bar(T::BAR_WEMPTY + s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) commit_local(bar(T::BAR_ACC_FULL + ab));
      __syncwarp();
      committed_tiles = i + 1;
    }
    if (lane == 0) {
      // Every issued UMMA must finish before TMEM is released: one more
      // commit on a buffer whose phase we can wait for.
      if (!ok) {
        const int ab = committed_tiles & 1;
        commit_local(bar(T::BAR_ACC_FULL + ab));
        wait_phase(bar(T::BAR_ACC_FULL + ab), (committed_tiles >> 1) & 1, ctl, false);
      } else if (committed_tiles > 0) {
        const int last = committed_tiles - 1;
        wait_phase(bar(T::BAR_ACC_FULL + (last & 1)), (last >> 1) & 1, ctl, false);
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + T::XF_WARPS) {
    if constexpr (!T::kTmaA) {
    // ---------------- transform warps
    const int grp = (warp - 4) / T::XF_PER_GROUP;
    const int tw = (warp - 4) % T::XF_PER_GROUP;
    const uint32_t slice_off = (crank * (uint32_t)T::ROWS + (uint32_t)(tw * T::RW)) * 128u;

    // k-blocks of this CTA, across work items
    const int total = n_full * nkb + (has_unit ? unit_kb1 - unit_kb0 : 0);
    // k-block g (counted across items) -> first row of this CTA's slice, k0
    auto coords = [&](int g, int& row0, int& k0) {
      int i, kb;
      if (g < n_full * nkb) {
        i = g / nkb;
        kb = g - i * nkb;
      } else {
        i = n_full;
        kb = unit_kb0 + (g - n_full * nkb);
      }
      row0 = tile_m0(item_tile(i)) + (int)crank * T::ROWS;
      k0 = kb * T::BK;
    };
    // The group loads its k-blocks in order, XF_GROUPS apart: a cursor steps
    // to the next one within its work item, and only crossing into the next
    // item takes the divisions of `coords` (they would otherwise sit on the
    // path to every load's issue).
    int cur_g = -1, cur_row0 = 0, cur_k0 = 0, cur_kend = 0;
    LaneRows cur_rows;
    auto cursor_to = [&](int g) {
      if (cur_g >= 0 && g - cur_g == T::XF_GROUPS && cur_k0 + T::XF_GROUPS * T::BK < cur_kend) {
        cur_k0 += T::XF_GROUPS * T::BK;
      } else {
        const int row0_before = cur_row0;
        coords(g, cur_row0, cur_k0);
        cur_kend = (g < n_full * nkb ? nkb : unit_kb1) * T::BK;
        if (cur_g < 0 || cur_row0 != row0_before)
          lane_rows<T>(cur_rows, cur_row0, args.M, args.K, tw, lane);
      }
      cur_g = g;
    };
    // the inputs of k-block g into b (instances whose staged registers leave
    // no room for the cursor compute the coordinates every time)
    auto load_kblock = [&](Staged<T>& b, int g) {
      if constexpr (T::kLaneRows) {
        cursor_to(g);
        stage_load_at<T>(b, args.A, args.U, cur_rows, cur_k0, args.K, args.status);
      } else {
        int row0, k0;
        coords(g, row0, k0);
        stage_load<T>(b, args.A, args.U, row0, k0, args.M, args.K, tw, lane, args.status);
      }
    };
    // This group's k-blocks are g = grp + XF_GROUPS * j; buffer j % PF holds
    // the inputs of k-block j, loaded PF of the group's k-blocks ahead.
    Staged<T> buf[T::PF];
#pragma unroll
    for (int d = 0; d < T::PF; ++d) {
      const int g = grp + T::XF_GROUPS * d;
      if (g < total) {
        load_kblock(buf[d], g);
      }
    }
    bool ok = true;
    int g_end = 0;   // k-blocks (of every group) before the first one not filled
    for (int j0 = 0; ok && grp + T::XF_GROUPS * j0 < total; j0 += T::PF) {
#pragma unroll
      for (int d = 0; d < T::PF; ++d) {
        const int g = grp + T::XF_GROUPS * (j0 + d);
        if (g >= total) break;
        uint32_t vals[T::LPI][T::CHUNK / 2];
        stage_compute<T>(buf[d], vals);
        const int gn = g + T::XF_GROUPS * T::PF;
        if (gn < total) {
          load_kblock(buf[d], gn);
        }
        const int s = g % T::NA;
        if (g >= T::NA) {
          // Every CTA's UMMA is done with this stage: ours may be rewritten
          // and the peers' copies of it overwritten.
          const bool w = wait_phase_cluster(bar(T::BAR_AEMPTY + s), ((g / T::NA) - 1) & 1, ctl);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
        }
        stage_store<T>(a_stage(s), crank, tw, lane, vals, args.status);
        fence_proxy_async_smem();   // our rows -> visible to UMMA and to the copy engine
        __syncwarp();
        {
          const uint32_t full = bar(T::BAR_AFULL + s);
          if constexpr (T::CN > 1) {
            // The peers' slices of this stage arrive as copy bytes on our
            // barrier; our slice goes to peer (crank + l) % CN from lane l,
            // so that the copies are issued side by side (measured faster
            // than lane 0 issuing them in turn).
            if (lane == 0) mbar_arrive_expect_tx(full, T::REMOTE_BYTES_PER_WARP);
            if (lane >= 1 && lane < CN) {
              const uint32_t dst = (crank + (uint32_t)lane) % (uint32_t)CN;
              const uint32_t src = a_stage(s) + slice_off;
              if (dcheck(dst < (uint32_t)T::CS && dst != crank, args.status, CHK_PEER, dst))
                bulk_copy_s2cluster(mapa_shared(src, dst), src, T::SLICE_BYTES,
                                    mapa_shared(full, dst));
            }
          } else {
            if (lane == 0) mbar_arrive(full);
          }
        }
        __syncwarp();
        g_end = g + 1;
      }
    }
    // Every peer's commit for the final use of each stage must have landed
    // (they arrive on our barriers, and our copies read our shared memory)
    // before this CTA may leave. The final uses are the CTA's last NA
    // k-blocks, whichever group filled them: waiting instead for this
    // group's own last ones could ask for a phase of a stage that the other
    // group has since used again, whose parity then reads as not yet
    // complete. After a failure, the k-blocks this group reached.
    const int g_last = ok ? total : g_end;
    if (lane == 0)
      for (int x = (g_last > T::NA ? g_last - T::NA : 0); x < g_last; ++x)
        wait_phase_cluster(bar(T::BAR_AEMPTY + x % T::NA), (x / T::NA) & 1, ctl, false);
    __syncwarp();
    }
  } else if (warp >= 4 + T::XF_WARPS) {
    // ---------------- epilogue warps: rows q*32 .. q*32+31 of the tile
    const int q = warp & 3;                        // TMEM lane quadrant
    constexpr int NC = T::BN / kEpiCols;
    constexpr int C4 = T::BN / 4;                  // float4 columns of a tile
    constexpr uint32_t NB = (uint32_t)T::EPI_BUFS;
    const uint32_t buf0 = sbase + T::OFF_EPI + (uint32_t)q * NB * T::EPI_BUF_BYTES;
    auto buf = [&](uint32_t b) -> uint32_t { return buf0 + b * T::EPI_BUF_BYTES; };
    auto ebar = [&](uint32_t b) -> uint32_t { return bar(T::BAR_EPI + q * (int)NB + (int)b); };
    // Chunks of 32 columns this warp has staged so far (across tiles): chunk
    // e uses buffer e % NB and, for R, phase (e / NB) & 1 of that buffer's
    // barrier. R loads are issued and waited for in chunk order: r_issued /
    // r_done count them, e_wait is the chunk of the next one to wait for.
    // With two buffers the R of chunk e+1 is loaded while chunk e is worked
    // on; with one, after chunk e's store has read the buffer.
    auto ebuf = [&](uint32_t e) -> uint32_t { return e % NB; };
    auto ephase = [&](uint32_t e) -> uint32_t { return (e / NB) & 1u; };
    // Checked build: an f32 TMA box at a column x that is a multiple of 4,
    // staged inside this warp's buffers; TMEM columns inside the item's
    // accumulator buffer.
    auto epi_ok = [&](int x, uint32_t smem, uint32_t bytes) -> bool {
      return dcheck((x & 3) == 0, args.status, CHK_TMA_X, x) &&
             dcheck(smem >= buf0 && smem + bytes <= buf0 + NB * T::EPI_BUF_BYTES, args.status,
                    CHK_BUFFER, (long long)(smem - sbase));
    };
    auto tcols_ok = [&](int col, int width) -> bool {
      return dcheck(col >= 0 && col + width <= T::BN, args.status, CHK_TMEM, col);
    };
    uint32_t ec = 0, r_issued = 0, r_done = 0, e_wait = 0;
    // SwiGLU-backward epilogue (two buffers): GATE and UP of a chunk land in
    // this warp's two buffers together (barrier BAR_EPI + 2q, one phase per
    // chunk)
    uint32_t sw_issued = 0, sw_done = 0;
    bool ok = true;
    for (int i = 0; i < n_items && ok; ++i) {
      const int t = item_tile(i);
      const bool is_unit = i >= n_full;            // a K range of a split tail tile
      const int ab = i & 1;
      const int row0 = tile_m0(t) + q * kEpiRows;
      const int n0 = tile_n0(t);
      int nc = n0 < args.N ? (args.N - n0 + kEpiCols - 1) / kEpiCols : 0;
      if (nc > T::BNO / kEpiCols) nc = T::BNO / kEpiCols;
      // chunks staged: nc, or nc of each product (Y's, then Y2's)
      const int nct = T::kDual ? 2 * nc : nc;
      // rows wholly past M: nothing to store (a store box may not start there)
      const bool rows_in = row0 < args.M;
      const bool staged = !is_unit && rows_in && nc > 0;
      if (RESID && staged && lane == 0) {
        // R of the first chunk, into a buffer whose last store has read it
        bulk_wait_group_read<0>();
        mbar_arrive_expect_tx(ebar(ebuf(ec)), T::EPI_BUF_BYTES);
        if (epi_ok(n0, buf(ebuf(ec)), T::EPI_BUF_BYTES))
          tma_load_2d(buf(ebuf(ec)), &tm_r, n0, row0, ebar(ebuf(ec)));
        ++r_issued;
      }
      // (a pair's accumulator is complete when the even CTA's commit says so)
      ok = T::kPair ? warp_wait_phase_cluster(bar(T::BAR_ACC_FULL + ab), (i >> 1) & 1, ctl)
                    : warp_wait_phase(bar(T::BAR_ACC_FULL + ab), (i >> 1) & 1, ctl);
      tc_fence_after_sync();
      // last item's accumulator complete: a split sum may be scheduled
      if (i == n_items - 1 && q == 0 && lane == 0) pdl_launch_dependents();
      ok = ok && (__shfl_sync(0xffffffffu, *abort_flag, 0) == 0);
      if (!ok) break;
      const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * T::BN);
      if (is_unit) {
        // partial tile of this unit: [C4 float4 columns][128 rows], so that
        // the 32 lanes (rows) of a store write 512 consecutive bytes
        float4* part = reinterpret_cast<float4*>(args.part) +
                       (size_t)(cid * T::CS + (int)crank) * C4 * T::BM + q * kEpiRows + lane;
        const long long part_end =
            (long long)(cid * T::CS + (int)crank) * C4 * T::BM + q * kEpiRows + lane;
        for (int c = 0; c < nc; ++c) {
          uint32_t v[32];
          if (!tcols_ok(c * kEpiCols, kEpiCols)) break;
          tmem_ld_32x32b_x32(acc + (uint32_t)(c * kEpiCols), v);
          tmem_wait_ld();
          if (!dcheck(part_end + (long long)(c * 8 + 7) * T::BM < args.part_f4, args.status,
                      CHK_PART, part_end + (long long)(c * 8 + 7) * T::BM))
            break;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            part[(size_t)(c * 8 + j) * T::BM] =
                make_float4(__uint_as_float(v[4 * j + 0]), __uint_as_float(v[4 * j + 1]),
                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      } else if (staged && NB == 2 && (args.flags & KFLAG_SWIGLU_BWD)) {
        // dA -> dGATE, dUP in chunks of 16 columns. The warp's two 4 KB
        // buffers hold four [32 rows][16 f32] tiles (64-byte swizzle): GATE
        // and UP of a chunk land in the first two by TMA, the gradients leave
        // from the other two by TMA store. The next chunk's GATE and UP are
        // requested as soon as this chunk's are in registers, so they load
        // while this chunk's gradients are stored (with one buffer pair
        // doing both, every load waited for the previous chunk's stores).
        constexpr int SC = kSwbCols;
        constexpr uint32_t SB = (uint32_t)(kEpiRows * SC * 4);   // 2 KB
        static_assert(2 * SB == T::EPI_BUF_BYTES, "four swizzled tiles in two buffers");
        const uint32_t gin = buf(0), uin = buf(0) + SB, gout = buf(1), uout = buf(1) + SB;
        int ns = n0 < args.N ? (args.N - n0 + SC - 1) / SC : 0;
        if (ns > T::BNO / SC) ns = T::BNO / SC;
        auto issue = [&](int c) {   // lane 0: GATE and UP of chunk c
          mbar_arrive_expect_tx(ebar(0), 2 * SB);
          if (epi_ok(n0 + c * SC, gin, 2 * SB)) {
            tma_load_2d(gin, &tm_g2, n0 + c * SC, row0, ebar(0));
            tma_load_2d(uin, &tm_u2, n0 + c * SC, row0, ebar(0));
          }
          ++sw_issued;
          // the following chunk's GATE and UP on their way into L2
          if (c + 1 < ns) {
            tma_prefetch_l2_2d(&tm_g2, n0 + (c + 1) * SC, row0);
            tma_prefetch_l2_2d(&tm_u2, n0 + (c + 1) * SC, row0);
          }
        };
        if (lane == 0 && ns > 0) {
          bulk_wait_group_read<0>();   // the last stores have read the input buffers too
          issue(0);
        }
        __syncwarp();
        for (int c = 0; c < ns && ok; ++c) {
          uint32_t v[SC];
          if (tcols_ok(c * SC, SC)) tmem_ld_32x32b_x16(acc + (uint32_t)(c * SC), v);
          tmem_wait_ld();
          if (!warp_wait_phase(ebar(0), sw_done & 1u, ctl)) {
            ok = false;
            break;
          }
          ++sw_done;
          float4 dg[SC / 4], du[SC / 4];
#pragma unroll
          for (int j = 0; j < SC / 4; ++j) {
            const uint32_t off = sw64((uint32_t)lane, (uint32_t)j);
            const float4 gt = ld_shared_v4f(gin + off);
            const float4 up = ld_shared_v4f(uin + off);
            swiglu_backward(__uint_as_float(v[4 * j + 0]), gt.x, up.x, dg[j].x, du[j].x);
            swiglu_backward(__uint_as_float(v[4 * j + 1]), gt.y, up.y, dg[j].y, du[j].y);
            swiglu_backward(__uint_as_float(v[4 * j + 2]), gt.z, up.z, dg[j].z, du[j].z);
            swiglu_backward(__uint_as_float(v[4 * j + 3]), gt.w, up.w, dg[j].w, du[j].w);
          }
          fence_proxy_async_smem();   // our reads of the inputs before the next loads land
          __syncwarp();
          if (lane == 0) {
            if (c + 1 < ns) issue(c + 1);
            bulk_wait_group_read<0>();   // the previous stores have read the output buffers
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < SC / 4; ++j) {
            const uint32_t off = sw64((uint32_t)lane, (uint32_t)j);
            st_shared_v4(gout + off, __float_as_uint(dg[j].x), __float_as_uint(dg[j].y),
                         __float_as_uint(dg[j].z), __float_as_uint(dg[j].w));
            st_shared_v4(uout + off, __float_as_uint(du[j].x), __float_as_uint(du[j].y),
                         __float_as_uint(du[j].z), __float_as_uint(du[j].w));
          }
          fence_proxy_async_smem();   // staged gradients -> visible to the TMA stores
          __syncwarp();
          if (lane == 0) {
            if (epi_ok(n0 + c * SC, gout, 2 * SB)) {
              tma_store_2d(&tm_y, n0 + c * SC, row0, gout);
              tma_store_2d(&tm_y2, n0 + c * SC, row0, uout);
            }
            bulk_commit_group();
          }
          __syncwarp();
        }
      } else if (staged) {
        // online-softmax partials of this lane's row over the tile's columns,
        // and the row's sum over them
        const bool stats = !T::kDual && (args.flags & KFLAG_ROW_STATS) != 0;
        float rm = -INFINITY, rs = 0.0f, rsum = 0.0f;
        for (int c = 0; c < nct && ok; ++c) {
          const uint32_t e = ec + (uint32_t)c;
          const uint32_t b = ebuf(e);
          // DUAL: chunk c < nc is Y's, else Y2's; its TMEM columns follow
          // the B stage ([W tile | W2 tile])
          const bool second = T::kDual && c >= nc;
          const int oc = second ? c - nc : c;                       // chunk of its output
          const int tc = second ? NC / 2 + oc : c;                  // chunk of the accumulator
          if (NB == 2 && lane == 0 && c + 1 < nct) {
            // the other buffer's last store must have read it before it is
            // refilled (or, without R, rewritten below)
            bulk_wait_group_read<0>();
            if constexpr (RESID) {
              mbar_arrive_expect_tx(ebar(b ^ 1u), T::EPI_BUF_BYTES);
              if (epi_ok(n0 + (c + 1) * kEpiCols, buf(b ^ 1u), T::EPI_BUF_BYTES))
                tma_load_2d(buf(b ^ 1u), &tm_r, n0 + (c + 1) * kEpiCols, row0, ebar(b ^ 1u));
              ++r_issued;
            }
          }
          __syncwarp();
          uint32_t v[32];
          if (tcols_ok(tc * kEpiCols, kEpiCols))
            tmem_ld_32x32b_x32(acc + (uint32_t)(tc * kEpiCols), v);
          tmem_wait_ld();
          if constexpr (RESID) {
            if (!warp_wait_phase(ebar(b), ephase(e), ctl)) {
              ok = false;
              break;
            }
            ++r_done;
            e_wait = e + 1;
          } else if ((NB == 1 || c == 0) && lane == 0) {
            bulk_wait_group_read<0>();   // this buffer's last store has read it
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t addr = buf(b) + sw128((uint32_t)lane, (uint32_t)j);
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
          fence_proxy_async_smem();   // staged Y -> visible to the TMA store
          __syncwarp();
          if (lane == 0) {
            if (epi_ok(n0 + oc * kEpiCols, buf(b), T::EPI_BUF_BYTES))
              tma_store_2d(second ? &tm_y2 : &tm_y, n0 + oc * kEpiCols, row0, buf(b));
            bulk_commit_group();
            if (RESID && NB == 1 && c + 1 < nct) {
              // the single buffer: the next chunk's R once this store has read it
              bulk_wait_group_read<0>();
              mbar_arrive_expect_tx(ebar(0), T::EPI_BUF_BYTES);
              if (epi_ok(n0 + (c + 1) * kEpiCols, buf(0), T::EPI_BUF_BYTES))
                tma_load_2d(buf(0), &tm_r, n0 + (c + 1) * kEpiCols, row0, ebar(0));
              ++r_issued;
            }
          }
          __syncwarp();
          if (stats) {
            // (max, sum exp(y - max), sum y) over the chunk's columns below N,
            // merged into the lane's running pair; computed while the chunk's
            // store is in flight. Four partial maxima and sums per quantity,
            // so that no chain is 32 operations long; a column at or past N
            // enters as -inf (exp 0) and adds 0 to the sum.
            constexpr float kLog2e = 1.4426950408889634f;
            const int nv = args.N - (n0 + c * kEpiCols);   // columns in range (>= 1)
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = i < nv ? __uint_as_float(v[i]) : -INFINITY;
            float m4[4], s4[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              m4[q4] = y[q4];
              s4[q4] = q4 < nv ? y[q4] : 0.0f;
            }
#pragma unroll
            for (int i = 4; i < 32; ++i) {
              m4[i & 3] = fmaxf(m4[i & 3], y[i]);
              s4[i & 3] += i < nv ? y[i] : 0.0f;
            }
            const float cm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            rsum += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            const float mn = fmaxf(rm, cm);
            float sum = (rm == -INFINITY) ? 0.0f : rs * ex2_approx((rm - mn) * kLog2e);
            if (mn != -INFINITY) {
              const float off = mn * kLog2e;
              float e4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int i = 0; i < 32; ++i) e4[i & 3] += ex2_approx(fmaf(y[i], kLog2e, -off));
              sum += (e4[0] + e4[1]) + (e4[2] + e4[3]);
            }
            rm = mn;
            rs = sum;
          }
        }
        ec += (uint32_t)nct;
        if (stats && ok && row0 + lane < args.M &&
            dcheck(n0 / T::BN < args.stats_cols, args.status, CHK_STATS, n0 / T::BN))
          args.row_stats[(size_t)(row0 + lane) * args.stats_cols + n0 / T::BN] =
              make_float4(rm, rs, rsum, 0.0f);
      }
      // TMEM reads of this buffer are complete: hand it back to the UMMA warp
      // (a pair's is in the even CTA).
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (T::kPair && crank != 0)
          mbar_arrive_remote(mapa_shared(bar(T::BAR_ACC_EMPTY + ab), 0));
        else
          mbar_arrive(bar(T::BAR_ACC_EMPTY + ab));
      }
    }
    if (lane == 0) {
      // Never leave with an R load in flight (only possible when a wait gave
      // up) or with a store still reading the buffers or writing Y.
      for (uint32_t x = 0; x < r_issued - r_done; ++x) {
        const uint32_t e = e_wait + x;   // the outstanding loads, oldest first
        wait_phase(ebar(ebuf(e)), ephase(e), ctl, false);
      }
      if (sw_issued > sw_done) wait_phase(ebar(0), sw_done & 1u, ctl, false);
      bulk_wait_group_all();
    }
    __syncwarp();
  }

  // ---- teardown: no CTA leaves while a peer may still write to it
  tc_fence_before_sync();
  if constexpr (T::CS > 1)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    if constexpr (T::kPair)
      tmem_dealloc_pair(tmem, T::TMEM_COLS);
    else
      tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

// Launch configuration of one instantiation; the first call per device sets
// the shared-memory attribute and records how many clusters fit at once.
template <int AMODE, bool RESID, int BN, int CN, bool BT = false, bool DUAL = false>
struct ClusterLaunch {
  using T = ClusterTraits<AMODE, RESID, BN, CN, false, BT, DUAL>;
  // attr must hold 2 entries: the cluster shape and, for launches, the
  // programmatic dependence on the previous kernel of the stream.
  static cudaLaunchConfig_t config(cudaLaunchAttribute* attr, cudaStream_t stream,
                                   bool dependent) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T::CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(T::kThreadsC, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 2 : 1;
    return cfg;
  }
  // Clusters resident at once on the current device (> 0), or 0 with *err.
  static int capacity(cudaError_t* err) {
    static std::atomic<uint64_t> attr_done{0};
    static std::atomic<int> max_clusters[64];
    auto kern = lin_gemm_cluster_kernel<AMODE, RESID, BN, CN, false, BT, DUAL>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && dev >= 64) e = cudaErrorInvalidDevice;
    if (e != cudaSuccess) {
      *err = e;
      return 0;
    }
    const uint64_t bit = uint64_t{1} << dev;
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
      if constexpr (!T::kTmaA) {   // the 32-byte-load variant of the transform
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(lin_gemm_cluster_kernel<AMODE, RESID, BN, CN, true, BT, DUAL>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   ClusterTraits<AMODE, RESID, BN, CN, true, BT, DUAL>::SMEM_BYTES);
      }
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = config(attr, nullptr, false);
      cfg.gridDim = dim3(T::CS, 1, 1);
      int n = 0;
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg);
      if (e == cudaSuccess && n < 1) e = cudaErrorInvalidConfiguration;
      if (e != cudaSuccess) {
        *err = e;
        return 0;
      }
      max_clusters[dev].store(n, std::memory_order_release);
      attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return max_clusters[dev].load(std::memory_order_acquire);
  }
  // Grid: every resident cluster when whole rounds remain; with a split tail
  // alone, one cluster per K range; else one per tile.
  static cudaError_t launch(const TensorMaps& m, const KernelArgs& args, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    const int cap = capacity(&e);
    if (cap < 1) return e;
    const int num_m = (args.M + T::TM - 1) / T::TM;
    const int num_ng = (args.N + T::BNO * T::CN - 1) / (T::BNO * T::CN);
    int clusters;
    if (args.split_s >= 2)
      clusters = args.split_r > 0 ? cap : args.split_rem * args.split_s;
    else
      clusters = num_m * num_ng < cap ? num_m * num_ng : cap;
    if (clusters > cap) return cudaErrorInvalidConfiguration;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = config(attr, stream, true);
    cfg.gridDim = dim3((unsigned)(clusters * T::CS), 1, 1);
    if constexpr (!T::kTmaA) {
      if (args.flags & KFLAG_A_V8)
        return cudaLaunchKernelEx(&cfg,
                                  lin_gemm_cluster_kernel<AMODE, RESID, BN, CN, true, BT, DUAL>,
                                  m.w, m.w2, m.a, m.r, m.y, m.g2, m.u2, m.y2, args);
    }
    return cudaLaunchKernelEx(&cfg, lin_gemm_cluster_kernel<AMODE, RESID, BN, CN, false, BT, DUAL>,
                              m.w, m.w2, m.a, m.r, m.y, m.g2, m.u2, m.y2, args);
  }
};

// Sum of a split: one thread per float4 of Y. Thread x is row x % 128 of
// float4 column c4 = (x / 128) % C4 of CTA `crank` of tile j, with
// x / (128 * C4) = j * cn + crank: the order of the partial tiles
// [unit][cta][C4][128 rows], so that consecutive threads load consecutive
// partial float4s. The cn CTAs of a tile sit side by side along N, or
// (pair) one above the other in a tile of 256 rows. Y = sum over the s K
// ranges in K order (+ R): independent of timing, so bitwise reproducible.
template <bool RESID, bool SWB>
__global__ void __launch_bounds__(256)
    lin_split_reduce_kernel(const float4* __restrict__ part, const float* __restrict__ R,
                            float* __restrict__ Y, int M, int N, int cn, int pair, int bn,
                            int tile0, int num_ng, int band, int rem, int s,
                            const float* __restrict__ G2, const float* __restrict__ U2,
                            float* __restrict__ Y2, long long part_f4, int* status) {
  const int c4n = bn / 4;
  const long long per_cta = 128LL * c4n;
  const long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= (long long)rem * cn * per_cta) return;
  const int jc = (int)(x / per_cta);          // j * cn + crank
  const int j = jc / cn, crank = jc % cn;
  const int c4 = (int)((x / 128) % c4n);
  const int r = (int)(x % 128);
  const int t = tile0 + j;
  const int tile_rows = pair ? 256 : 128;
  const TileRC rc = tile_coords(t, (M + tile_rows - 1) / tile_rows, num_ng, band);
  const int row = rc.m * tile_rows + (pair ? crank * 128 : 0) + r;
  const int col = (pair ? rc.ng : rc.ng * cn + crank) * bn + 4 * c4;
  // The next kernel on the stream may be scheduled now: it waits for this
  // grid's completion itself before it touches memory.
  pdl_launch_dependents();
  if (row >= M || col >= N) return;
  // Launched as a programmatic dependent of the GEMM: wait here until the
  // GEMM's partial tiles are complete and visible.
  pdl_wait();
  // Up to 8 partials in flight per thread, added in K order.
  const long long first = ((long long)(j * s * cn + crank) * c4n + c4) * 128 + r;
  const float4* src = part + first;
  const long long stride = (long long)cn * c4n * 128;   // next K range
  if (!dcheck(first + (long long)(s - 1) * stride < part_f4, status, CHK_PART,
              first + (long long)(s - 1) * stride))
    return;
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0; p0 < s; p0 += 8) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (p0 + i < s) v[i] = __ldcg(src + (p0 + i) * stride);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (p0 + i < s) {
        sum.x += v[i].x;
        sum.y += v[i].y;
        sum.z += v[i].z;
        sum.w += v[i].w;
      }
    }
  }
  const size_t off = (size_t)row * (size_t)N + (size_t)col;
  if constexpr (SWB) {   // the SwiGLU backward of the summed dA
    const float4 gt = *reinterpret_cast<const float4*>(G2 + off);
    const float4 up = *reinterpret_cast<const float4*>(U2 + off);
    float4 dg, du;
    swiglu_backward(sum.x, gt.x, up.x, dg.x, du.x);
    swiglu_backward(sum.y, gt.y, up.y, dg.y, du.y);
    swiglu_backward(sum.z, gt.z, up.z, dg.z, du.z);
    swiglu_backward(sum.w, gt.w, up.w, dg.w, du.w);
    *reinterpret_cast<float4*>(Y + off) = dg;
    *reinterpret_cast<float4*>(Y2 + off) = du;
    return;
  }
  if constexpr (RESID) {
    const float4 rv = *reinterpret_cast<const float4*>(R + off);
    sum.x += rv.x;
    sum.y += rv.y;
    sum.z += rv.z;
    sum.w += rv.w;
  }
  *reinterpret_cast<float4*>(Y + off) = sum;
}

}  // namespace lin
