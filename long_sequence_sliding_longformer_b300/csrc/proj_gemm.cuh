// proj_gemm.cuh -- per-head linear projections of hidden states on the
// tensor cores: y = x W^T (+ bias), written straight into head-major
// [n_out, B, H, n, d] tensors (section 3-1, "Linear Projections for Global
// Attention": the band and the global attention each project the hidden
// states with their own W_q, W_k, W_v).
//
// x: [M = B*n, K] bf16, W: [N = n_out*H*d, K] bf16 (the rows of one output
// column are contiguous: both operands are K-major), fp32 accumulation.
// Persistent CTAs (one per SM), 6 warps:
//   warp 0     TMA producer: per 64-wide K step, a [128, 64] tile of x and a
//              [BN, 64] tile of W into a four-stage ring (128-byte swizzle)
//   warp 1     allocates TMEM; issues the tcgen05.mma (M = 128, N = BN,
//              K = 16, four per K step) into one of two accumulators
//   warps 2-5  epilogue: TMEM -> registers (+ bias) -> bf16 -> global; the
//              accumulator is released as soon as it is read, so the next
//              tile's products run during the stores
// Output tiles are [128 rows, BN columns]; tile t of the CTA is
// blockIdx.x + t * gridDim.x over (row block, column block), column blocks
// fastest.  Every wait is bounded (the pipeline limit of lf_internal.cuh).
#pragma once

#include "lf_internal.cuh"

namespace lf {
namespace projk {

constexpr uint32_t kRoleEpilogue = 6;
constexpr int kBM = 128, kBK = 64, kStages = 4;
constexpr int kThreads = 192;

struct ProjParams {
  CUtensorMap tx, tw;  // x [M, K] and W [N, K], boxes [64, 128] and [64, BN]
  const float* bias;   // [N] or nullptr
  __nv_bfloat16* y;    // [n_out, B, H, n, d]
  int32_t M, N, K, B, n, H, d;
  int32_t tiles_n, tiles;  // column blocks, all tiles
};

template <int BN>
struct Cfg {
  static constexpr int kTileA = kBM * kBK * 2;  // 16 KB
  static constexpr int kTileB = BN * kBK * 2;   // 16 or 32 KB
  static constexpr int kStage = kTileA + kTileB;
  static constexpr int kOffBar = kStages * kStage;
  // full[4], empty[4], acc_full[2], acc_empty[2]
  static constexpr int kNumBar = 2 * kStages + 4;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;  // tmem holder, abort flag, wait limit
  static constexpr int kSmem = kOffMisc + 16 + 1024;      // + slack to align the base to 1024
  static constexpr int kTmemCols = 2 * BN;
  static_assert(kSmem <= 232448, "shared memory");
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) proj_gemm_kernel(const __grid_constant__ ProjParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  auto a_tile = [&](int s) { return sbase + s * C::kStage; };
  auto b_tile = [&](int s) { return sbase + s * C::kStage + C::kTileA; };
  auto bar = [&](int i) { return sbase + C::kOffBar + 8 * i; };  // full 0..3, empty 4..7, accf 8..9, acce 10..11
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(s), 1);            // full: the producer's expect_tx
      mbar_init(bar(kStages + s), 1);  // empty: the MMA warp's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(2 * kStages + b), 1);      // accumulator full: commit
      mbar_init(bar(2 * kStages + 2 + b), 4);  // accumulator empty: the four epilogue warps
    }
    *abort = 0;
    *cta_wait_limit(abort) = wait_limit_ns();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int ksteps = p.K / kBK;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int last_fill[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last_fill[s] = -1;
    uint32_t it = 0;  // K steps issued over all tiles
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
      const int m0 = (tile / p.tiles_n) * kBM, n0 = (tile % p.tiles_n) * BN;
      for (int kb = 0; kb < ksteps; ++kb, ++it) {
        const int s = it % kStages;
        if (!warp_wait(bar(kStages + s), ((it / kStages) & 1) ^ 1, abort, kRoleProducer)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(s), C::kStage);
          tma_load_3d(a_tile(s), &p.tx, kb * kBK, m0, 0, bar(s));
          tma_load_3d(b_tile(s), &p.tw, kb * kBK, n0, 0, bar(s));
        }
        last_fill[s] = (int)it;
      }
    }
    // every copy issued must land before the CTA can exit
    int dummy = 0;
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (last_fill[s] >= 0) mbar_wait(bar(s), ((uint32_t)last_fill[s] / kStages) & 1, &dummy, kRoleDrain, kDrainLimitNs);
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, 0);
    uint32_t it = 0, lt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x, ++lt) {
      const int ab = lt & 1;
      // the epilogue has read this accumulator's previous tile
      if (!warp_wait(bar(2 * kStages + 2 + ab), ((lt >> 1) & 1) ^ 1, abort, kRoleMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + ab * BN;
      for (int kb = 0; kb < ksteps; ++kb, ++it) {
        const int s = it % kStages;
        if (!warp_wait(bar(s), (it / kStages) & 1, abort, kRoleMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(a_tile(s), 16, 1024);
        const uint64_t bd = smem_desc_sw128(b_tile(s), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16_ss_w(acc, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(bar(kStages + s));  // the stage is free once these products are done
      }
      if (!ok) break;
      mma_commit_w(bar(2 * kStages + ab));  // the tile's accumulator is complete
    }
    // every MMA issued must finish before TMEM is freed: wait for the last commits
    int dummy = 0;
    if (it > 0) {
      const uint32_t last = it - 1;
      mbar_wait(bar(kStages + last % kStages), (last / kStages) & 1, &dummy, kRoleDrain, kDrainLimitNs);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;  // TMEM lanes 32*q4 .. 32*q4 + 31
    const int row_in_tile = 32 * q4 + lane;
    uint32_t lt = 0;
    const int Hd = p.H * p.d;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++lt) {
      const int ab = lt & 1;
      if (!warp_wait(bar(2 * kStages + ab), (lt >> 1) & 1, abort, kRoleEpilogue)) break;
      tc_fence_after();
      const int m0 = (tile / p.tiles_n) * kBM, n0 = (tile % p.tiles_n) * BN;
      const int row = m0 + row_in_tile;  // token b*n + i
      const bool row_ok = row < p.M;
      const int b = row_ok ? row / p.n : 0, i = row_ok ? row - (row / p.n) * p.n : 0;
      const uint32_t tbase = tmem + ((uint32_t)(32 * q4) << 16) + ab * BN;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32_nw(tbase + c0, r);
        tmem_wait_ld();
        if (c0 + 32 >= BN) {
          // the accumulator is read: release it to the next tile's products
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(2 * kStages + 2 + ab));
        }
        if (!row_ok) continue;
        const int col = n0 + c0;  // 32 columns of one head (d is a multiple of 32)
        const int t = col / Hd, h = (col % Hd) / p.d, c = col % p.d;
        __nv_bfloat16* dst = p.y + ((((int64_t)t * p.B + b) * p.H + h) * p.n + i) * p.d + c;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float lo = __uint_as_float(r[2 * e]), hi = __uint_as_float(r[2 * e + 1]);
          if (p.bias) {
            lo += __ldg(p.bias + col + 2 * e);
            hi += __ldg(p.bias + col + 2 * e + 1);
          }
          pk[e] = pack_bf16x2(lo, hi);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
          reinterpret_cast<uint4*>(dst)[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace projk
}  // namespace lf
