// band_tc.cuh -- bf16 band-attention kernel on the sm_103a tensor cores.
//
// Computes the sliding / dilated / causal window part of Longformer attention
// (velog.io/@lainshower/Longformer, section 3-1 "Sliding Window", "Dilated
// Sliding Window", section 4.1 for the look-back-only pattern) plus the
// global tokens' key columns ("Global Attention"), for every row.  Rows of
// global tokens are overwritten afterwards by the global-row kernels.
//
// Dilation is handled by residue classes: with dilation delta, row
// i = r + delta*m only ever attends rows of the same residue r, and in the
// coordinate m the window is a plain +-w/2 band.  Each work item is one tile
// of 128 consecutive m of one (batch, head, residue); a TMA tensor map whose
// row stride is delta rows gives the tile and its key tiles directly.
//
// Per CTA (one per SM, persistent over work items), 6 warps:
//   warp 0     producer: TMA loads of Q and of the K/V tiles that intersect
//              the item's window into a ring of shared-memory stages, and a
//              gather of the global tokens' K/V rows for the global-column tile
//   warp 1     allocates TMEM; lane 0 issues tcgen05.mma:
//              S = Q K^T into one of two TMEM score buffers, O += P V into TMEM
//   warps 2-5  one query row per thread: read S from TMEM, apply the window,
//              padding and global-column masks, fp32 online softmax (exp2),
//              write P (bf16) to shared memory, rescale O in TMEM when the
//              running maximum grows, and finally normalise O and store it.
// Every wait is bounded; a timeout sets the device error word and all roles
// leave their loops, drain their in-flight copies and free TMEM.
#pragma once

#include "lf_internal.cuh"

namespace lf {

template <int D>
struct BandCfg {
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kTile = 128 * D * 2;  // bytes of one [128, D] bf16 tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTile;       // stage s: K at +2*s*kTile, V at +(2*s+1)*kTile
  static constexpr int kOffP = kOffKV + kStages * 2 * kTile;
  static constexpr int kOffGcol = kOffP + 128 * 128 * 2;  // per stage: gpos[128], gm[128]
  static constexpr int kOffBar = kOffGcol + kStages * 2 * 128 * 4;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], s_empty[2], p_full, pv_done, o_empty, fin
  static constexpr int kNumBar = 2 + 2 * kStages + 4 + 4;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kSmem = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr int kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256, 256+D)
  static constexpr int kOCol = 256;
};

struct ItemInfo {
  int b, h, r, delta, n_r, set, m0, Lb, Lm, kstart, kend, nb, ngt;
  int i_last;  // position of the tile's last valid query row
  bool zero;
};

__device__ __forceinline__ ItemInfo decode_item(const BandParams& p, int item) {
  ItemInfo it;
  it.b = item / p.items_per_b;
  const int rem = item - it.b * p.items_per_b;
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seg[mid].begin <= rem) lo = mid; else hi = mid - 1;
  }
  it.h = p.seg[lo].h;
  it.r = p.seg[lo].r;
  it.delta = p.seg[lo].delta;
  it.n_r = p.seg[lo].n_r;
  it.set = p.seg[lo].set;
  it.m0 = (rem - p.seg[lo].begin) * 128;
  it.Lb = p.n - p.pad[it.b];
  const int Lm = (it.Lb > it.r) ? (it.Lb - it.r + it.delta - 1) / it.delta : 0;
  it.Lm = min(Lm, it.n_r);
  it.zero = it.m0 >= it.Lm;
  it.kstart = max(0, it.m0 - p.half);
  const int lastq = min(it.m0 + 127, it.Lm - 1);
  it.kend = min(it.Lm - 1, lastq + p.right);  // last key any row of the tile attends
  it.i_last = it.r + it.delta * lastq;
  it.nb = it.zero ? 0 : (it.kend - it.kstart) / 128 + 1;
  it.ngt = it.zero ? 0 : (p.G + 127) / 128;
  return it;
}

// keys of global tile gt: ranks [128*gt, 128*gt + cnt), padded to a multiple of 16
__device__ __forceinline__ int global_tile_count(const BandParams& p, int gt) {
  return min(128, p.G - gt * 128);
}

template <int D>
struct BandSmem {
  using C = BandCfg<D>;
  uint8_t* base;
  uint32_t sbase;
  __device__ __forceinline__ uint32_t q() const { return sbase + C::kOffQ; }
  __device__ __forceinline__ uint32_t k(int s) const { return sbase + C::kOffKV + 2 * s * C::kTile; }
  __device__ __forceinline__ uint32_t v(int s) const { return sbase + C::kOffKV + (2 * s + 1) * C::kTile; }
  __device__ __forceinline__ uint8_t* k_ptr(int s) const { return base + C::kOffKV + 2 * s * C::kTile; }
  __device__ __forceinline__ uint8_t* v_ptr(int s) const { return base + C::kOffKV + (2 * s + 1) * C::kTile; }
  __device__ __forceinline__ uint32_t pbuf() const { return sbase + C::kOffP; }
  __device__ __forceinline__ uint8_t* p_ptr() const { return base + C::kOffP; }
  __device__ __forceinline__ int* gpos(int s) const { return reinterpret_cast<int*>(base + C::kOffGcol + s * 1024); }
  __device__ __forceinline__ int* gm(int s) const { return gpos(s) + 128; }
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + C::kOffBar + 8 * i; }
  __device__ __forceinline__ uint32_t q_full() const { return bar(0); }
  __device__ __forceinline__ uint32_t q_empty() const { return bar(1); }
  __device__ __forceinline__ uint32_t kv_full(int s) const { return bar(2 + s); }
  __device__ __forceinline__ uint32_t kv_empty(int s) const { return bar(2 + C::kStages + s); }
  __device__ __forceinline__ uint32_t s_full(int b) const { return bar(2 + 2 * C::kStages + b); }
  __device__ __forceinline__ uint32_t s_empty(int b) const { return bar(4 + 2 * C::kStages + b); }
  __device__ __forceinline__ uint32_t p_full() const { return bar(6 + 2 * C::kStages); }
  __device__ __forceinline__ uint32_t pv_done() const { return bar(7 + 2 * C::kStages); }
  __device__ __forceinline__ uint32_t o_empty() const { return bar(8 + 2 * C::kStages); }
  __device__ __forceinline__ uint32_t fin() const { return bar(9 + 2 * C::kStages); }
  __device__ __forceinline__ uint32_t* tmem_holder() const { return reinterpret_cast<uint32_t*>(base + C::kOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + C::kOffMisc + 4); }
};

// 16-byte chunk `ch` of row `row` inside a [rows, D] bf16 tile stored as D/64
// blocks of [128 rows, 64] with the 128-byte swizzle TMA uses.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
  return (uint32_t)((ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void band_producer(const BandParams& p, const BandSmem<D>& sm, int lane) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  uint32_t kv_it = 0, q_it = 0;
  int last_fill[C::kStages];
#pragma unroll
  for (int s = 0; s < C::kStages; ++s) last_fill[s] = -1;
  int last_q = -1;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const ItemInfo it = decode_item(p, item);
    if (it.zero) continue;
    const int bh = it.b * p.H + it.h;

    if (!warp_wait(sm.q_empty(), (q_it & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
    if (lane == 0) {
      mbar_arrive_expect_tx(sm.q_full(), C::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sm.q() + c * 16384, &p.tq[it.set], c * 64, it.m0, bh, sm.q_full());
    }
    last_q = (int)q_it;
    ++q_it;

    for (int j = 0; j < it.nb; ++j, ++kv_it) {
      const int s = kv_it % C::kStages;
      const uint32_t ph = (kv_it / C::kStages) & 1;
      if (!warp_wait(sm.kv_empty(s), ph ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(sm.kv_full(s), 2 * C::kTile);
        const int y = it.kstart + 128 * j;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sm.k(s) + c * 16384, &p.tk[it.set], c * 64, y, bh, sm.kv_full(s));
          tma_load_3d(sm.v(s) + c * 16384, &p.tv[it.set], c * 64, y, bh, sm.kv_full(s));
        }
      }
      last_fill[s] = (int)kv_it;
    }
    if (!ok) break;

    for (int gt = 0; gt < it.ngt; ++gt, ++kv_it) {
      const int s = kv_it % C::kStages;
      const uint32_t ph = (kv_it / C::kStages) & 1;
      if (!warp_wait(sm.kv_empty(s), ph ^ 1, abort, kRoleProducer)) { ok = false; break; }
      const int g0 = gt * 128;
      const int cnt = global_tile_count(p, gt);
      const int ng = (cnt + 15) & ~15;
      int* gpos = sm.gpos(s);
      int* gm = sm.gm(s);
      // a global key no row of this tile may attend (padding, or after the
      // tile's last row when causal) is stored as zeros
      const int g_lim = p.causal ? min(it.Lb - 1, it.i_last) : it.Lb - 1;
      for (int c = lane; c < 128; c += 32) {
        const int g = (c < cnt) ? p.gidx[g0 + c] : -1;
        const bool valid = (c < cnt) && g <= g_lim;
        gpos[c] = valid ? g : -1;
        int mg = -(1 << 29);  // "not in this residue class": never inside the band
        if (valid && (g - it.r) % it.delta == 0) mg = (g - it.r) / it.delta;
        gm[c] = mg;
      }
      const __nv_bfloat16* kb = p.k + (size_t)bh * p.n * D;
      const __nv_bfloat16* vb = p.v + (size_t)bh * p.n * D;
      constexpr int CH = D / 8;  // 16-byte chunks per row
      uint8_t* ks = sm.k_ptr(s);
      uint8_t* vs = sm.v_ptr(s);
      for (int idx = lane; idx < ng * CH; idx += 32) {
        const int row = idx / CH, ch = idx - (idx / CH) * CH;
        uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
        if (row < cnt) {
          const int g = p.gidx[g0 + row];
          if (g <= g_lim) {
            kx = __ldg(reinterpret_cast<const uint4*>(kb + (size_t)g * D) + ch);
            vx = __ldg(reinterpret_cast<const uint4*>(vb + (size_t)g * D) + ch);
          }
        }
        const uint32_t off = sw128_offset(row, ch);
        *reinterpret_cast<uint4*>(ks + off) = kx;
        *reinterpret_cast<uint4*>(vs + off) = vx;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.kv_full(s));
      last_fill[s] = -1;  // completed synchronously
    }
  }
  // Let every TMA copy this warp issued land before the CTA can exit.
#pragma unroll
  for (int s = 0; s < C::kStages; ++s)
    if (last_fill[s] >= 0) {
      int dummy = 0;
      mbar_wait(sm.kv_full(s), ((uint32_t)last_fill[s] / C::kStages) & 1, &dummy, kRoleDrain, 200000000ull);
    }
  if (last_q >= 0) {
    int dummy = 0;
    mbar_wait(sm.q_full(), (uint32_t)last_q & 1, &dummy, kRoleDrain, 200000000ull);
  }
}

// ------------------------------------------------------------------ MMA issuer (one thread)
template <int D>
__device__ void band_mma(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
  uint32_t kv_it = 0, q_it = 0, s_it = 0, pf_it = 0, o_it = 0;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const ItemInfo it = decode_item(p, item);
    if (it.zero) continue;
    const int J = it.nb + it.ngt;
    if (!mbar_wait(sm.q_full(), q_it & 1, abort, kRoleMma)) { ok = false; break; }
    ++q_it;
    tc_fence_after();

    auto issue_s = [&](int j) -> bool {
      const uint32_t kvj = kv_it + j;
      const int s = kvj % C::kStages;
      if (!mbar_wait(sm.kv_full(s), (kvj / C::kStages) & 1, abort, kRoleMma)) return false;
      const int sb = s_it & 1;
      if (!mbar_wait(sm.s_empty(sb), ((s_it >> 1) & 1) ^ 1, abort, kRoleMma)) return false;
      tc_fence_after();
      int N = 128;
      if (j >= it.nb) N = (global_tile_count(p, j - it.nb) + 15) & ~15;
      const uint32_t idesc = (N == 128) ? idesc_s : idesc_bf16_f32(128, N, 0);
      const uint32_t dt = tmem + sb * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qa = sm.q() + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t ka = sm.k(s) + (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16_ss(dt, smem_desc_sw128(qa, 16, 1024), smem_desc_sw128(ka, 16, 1024), idesc, kk > 0);
      }
      mma_commit(sm.s_full(sb));
      ++s_it;
      return true;
    };

    if (!issue_s(0)) { ok = false; break; }
    for (int j = 0; j < J; ++j) {
      if (j + 1 < J) {
        if (!issue_s(j + 1)) { ok = false; break; }
      } else {
        mma_commit(sm.q_empty());  // Q may be replaced once every S of this item is done
      }
      if (!mbar_wait(sm.p_full(), pf_it & 1, abort, kRoleMma)) { ok = false; break; }
      ++pf_it;
      if (j == 0) {
        if (!mbar_wait(sm.o_empty(), (o_it & 1) ^ 1, abort, kRoleMma)) { ok = false; break; }
        ++o_it;
      }
      tc_fence_after();
      const int s = (kv_it + j) % C::kStages;
      int K = 128;
      if (j >= it.nb) K = (global_tile_count(p, j - it.nb) + 15) & ~15;
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint32_t pa = sm.pbuf() + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t va = sm.v(s) + kk * 2048;
        mma_bf16_ss(tmem + C::kOCol, smem_desc_sw128(pa, 16, 1024), smem_desc_sw128(va, 16384, 1024),
                    idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(sm.kv_empty(s));
      mma_commit(sm.pv_done());
    }
    kv_it += J;
  }
  // Wait until every MMA this thread issued has finished before TMEM is freed.
  mma_commit(sm.fin());
  int dummy = 0;
  mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, 200000000ull);
}

// ------------------------------------------------------------------ softmax / epilogue
template <int D>
__device__ void band_softmax(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem, int warp,
                             int lane) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  const int wq = warp & 3;  // TMEM lane quarter this warp may access
  const int row = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const float NEG_INF = -__int_as_float(0x7f800000);
  uint32_t kv_it = 0, s_it = 0, pv_it = 0;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const ItemInfo it = decode_item(p, item);
    const int bh = it.b * p.H + it.h;
    const int m_q = it.m0 + row;
    const int i_q = it.r + it.delta * m_q;
    const bool row_exists = m_q < it.n_r;
    const bool row_valid = m_q < it.Lm;
    uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)bh * p.n + (row_exists ? i_q : 0)) * D);
    if (it.zero) {
      if (row_exists) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const int J = it.nb + it.ngt;
    float m_run = NEG_INF, l_run = 0.f;

    for (int j = 0; j < J; ++j) {
      const uint32_t kvj = kv_it + j;
      const int s = kvj % C::kStages;
      const bool is_band = j < it.nb;
      const int sb = s_it & 1;
      if (!warp_wait(sm.s_full(sb), (s_it >> 1) & 1, abort, kRoleSoftmax)) { ok = false; break; }
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float tmp[32];
        tmem_ld32(tmem + lane_base + sb * 128 + c4 * 32, tmp);
#pragma unroll
        for (int t = 0; t < 32; ++t) sv[c4 * 32 + t] = tmp[t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.s_empty(sb));
      ++s_it;

      // ---- masks, scaling to the exp2 domain, tile maximum
      float tmax = NEG_INF;
      if (is_band) {
        const int kb = it.kstart + 128 * j;
        int clo = max(0, m_q - kb - p.half);
        int chi = min(127, min(m_q - kb + p.right, it.Lm - 1 - kb));
        if (!row_valid) { clo = 1; chi = 0; }
        if (clo == 0 && chi == 127) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            sv[c] *= p.sl2;
            tmax = fmaxf(tmax, sv[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            sv[c] = (c >= clo && c <= chi) ? sv[c] * p.sl2 : NEG_INF;
            tmax = fmaxf(tmax, sv[c]);
          }
        }
      } else {
        // global-key columns: wait for the gather (its shared-memory tables)
        if (!warp_wait(sm.kv_full(s), (kvj / C::kStages) & 1, abort, kRoleSoftmax)) { ok = false; break; }
        const int* gpos = sm.gpos(s);
        const int* gmv = sm.gm(s);
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int g = gpos[c];
          const int mg = gmv[c];
          const bool in_band = (m_q - mg <= p.half) && (mg - m_q <= p.right);
          const bool keep = row_valid && g >= 0 && (!p.causal || g <= i_q) && !in_band;
          sv[c] = keep ? sv[c] * p.sl2 : NEG_INF;
          tmax = fmaxf(tmax, sv[c]);
        }
      }
      const float m_new = fmaxf(m_run, tmax);
      const float m_use = (m_new == NEG_INF) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);

      uint32_t pk[64];
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2_approx(sv[2 * c] - m_use);
        const float p1 = ex2_approx(sv[2 * c + 1] - m_use);
        lsum += p0 + p1;
        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
        pk[c] = *reinterpret_cast<uint32_t*>(&h2);
      }
      l_run = l_run * alpha + lsum;

      // ---- the previous P.V must be done: P buffer free, O stable
      if (j > 0) {
        if (!warp_wait(sm.pv_done(), pv_it & 1, abort, kRoleSoftmax)) { ok = false; break; }
        ++pv_it;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            float o[32];
            tmem_ld32(tmem + lane_base + C::kOCol + c4 * 32, o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] *= alpha;
            tmem_st32(tmem + lane_base + C::kOCol + c4 * 32, o);
          }
        }
      }
      // ---- value rows after the last key any row of the tile attends (the
      // padding, and keys outside every window of the tile) are zeroed, so
      // whatever they hold cannot reach the output through 0 * value
      if (is_band) {
        const int kb = it.kstart + 128 * j;
        if (kb + 127 > it.kend) {
          if (!warp_wait(sm.kv_full(s), (kvj / C::kStages) & 1, abort, kRoleSoftmax)) { ok = false; break; }
          if (kb + row > it.kend) {
            uint8_t* vs = sm.v_ptr(s);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
#pragma unroll
              for (int t = 0; t < 8; ++t)
                *reinterpret_cast<uint4*>(vs + c * 16384 + row * 128 + t * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // ---- P row to shared memory (two [128, 64] swizzled blocks)
      uint8_t* pb = sm.p_ptr();
#pragma unroll
      for (int ch = 0; ch < 16; ++ch)
        *reinterpret_cast<uint4*>(pb + sw128_offset(row, ch)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full());
      m_run = m_new;
    }
    if (!ok) break;
    kv_it += J;

    // ---- epilogue: O / l -> bf16 -> global
    if (!warp_wait(sm.pv_done(), pv_it & 1, abort, kRoleSoftmax)) { ok = false; break; }
    ++pv_it;
    tc_fence_after();
    float o[D];
#pragma unroll
    for (int c4 = 0; c4 < D / 32; ++c4) {
      float tmp[32];
      tmem_ld32(tmem + lane_base + C::kOCol + c4 * 32, tmp);
#pragma unroll
      for (int t = 0; t < 32; ++t) o[c4 * 32 + t] = tmp[t];
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.o_empty());
    const float inv = (row_valid && l_run > 0.f) ? 1.0f / l_run : 0.f;
    if (row_exists) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        __nv_bfloat162 a = __floats2bfloat162_rn(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
        __nv_bfloat162 b = __floats2bfloat162_rn(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
        __nv_bfloat162 e = __floats2bfloat162_rn(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
        __nv_bfloat162 f = __floats2bfloat162_rn(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
        orow[c] = make_uint4(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b),
                             *reinterpret_cast<uint32_t*>(&e), *reinterpret_cast<uint32_t*>(&f));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(192, 1) band_tc_kernel(const __grid_constant__ BandParams p) {
  using C = BandCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  BandSmem<D> sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    sm.base = smem_raw + pad;
    sm.sbase = raw + pad;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full(), 1);
    mbar_init(sm.q_empty(), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(sm.kv_full(s), 1);
      mbar_init(sm.kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm.s_full(b), 1);
      mbar_init(sm.s_empty(b), 4);
    }
    mbar_init(sm.p_full(), 4);
    mbar_init(sm.pv_done(), 1);
    mbar_init(sm.o_empty(), 4);
    mbar_init(sm.fin(), 1);
    *sm.abort_flag() = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(sm.tmem_holder()), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder();

  if (warp == 0) {
    band_producer<D>(p, sm, lane);
  } else if (warp == 1) {
    if (lane == 0) band_mma<D>(p, sm, tmem);
    __syncwarp();
  } else {
    band_softmax<D>(p, sm, tmem, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
static lf_status launch_band_tc_d(const BandParams& p, int grid, cudaStream_t s) {
  using C = BandCfg<D>;
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(band_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute(band kernel): %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
    attr_set = true;
  }
  band_tc_kernel<D><<<grid, 192, C::kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("band kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

lf_status launch_band_tc(const BandParams& p, int d, int grid, cudaStream_t s) {
  if (d == 64) return launch_band_tc_d<64>(p, grid, s);
  if (d == 128) return launch_band_tc_d<128>(p, grid, s);
  set_error("band kernel: unsupported head dimension %d", d);
  return LF_ERR_UNSUPPORTED;
}

}  // namespace lf
