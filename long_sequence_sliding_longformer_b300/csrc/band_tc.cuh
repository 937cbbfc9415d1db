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
// coordinate m the window is a plain band of half steps back and `right`
// steps ahead.  A TMA tensor map whose row stride is delta rows presents a
// residue class as a dense matrix.
//
// Work item: two consecutive 128-row query tiles X = 0, 1 (256 rows of m) of
// one (batch, head, residue).  Their key tiles overlap, so the item streams
// the union of the two windows once (128-key "entries", then the gathered
// global-token keys) and both tiles consume the shared entries.
//
// One CTA per SM, persistent over items, 12 warps:
//   warps 0-3  softmax of tile 0, warps 4-7 softmax of tile 1: one query row
//              per thread; S rows are read from TMEM, masked, turned into
//              P = exp2(S*scale - m) with a lazily updated row maximum, and P
//              (bf16) is written back to TMEM for the P.V product
//   warp 8     producer: TMA loads of Q and of the K/V entries into two
//              rings of shared-memory slots; gathers of global-token rows
//   warp 9     allocates TMEM; lane 0 issues every tcgen05.mma:
//              S_X = Q_X K^T (both operands in shared memory) and
//              O_X += P_X V (P from TMEM, V from shared memory)
//   warps 10-11 idle (they complete the third warpgroup, whose registers go
//              to the softmax warps)
// While the softmax warps of one tile work, the tensor cores run the other
// tile's products (ping-pong), so the exponentials and the MMAs overlap.
//
// TMEM: S_0, S_1 (128 columns each) and O_0, O_1 (D columns each).  P_X
// (two bf16 per column) overwrites the first 64 columns of S_X once the row
// has been read, chunk by chunk, so no register array holds all of P; the MMA
// of the next entry's S_X is issued after the P.V that reads P_X (the tensor
// core executes one thread's MMAs in order).  The completion of S_X(j+1)
// therefore also tells the softmax that P_X(j).V is done and O_X is stable.
//
// Every wait is bounded; a timeout sets the device error word and all roles
// leave their loops, drain their in-flight copies and free TMEM.
#pragma once

#include "lf_internal.cuh"

namespace lf {

template <int D>
struct BandCfg {
  static constexpr int kQBuf = (D == 64) ? 2 : 1;
  static constexpr int kKSt = (D == 64) ? 4 : 3;
  static constexpr int kVSt = (D == 64) ? 4 : 2;
  static constexpr int kTile = 128 * D * 2;     // bytes of one [128, D] bf16 tile
  static constexpr int kOffQ = 0;               // Q[qb][X] at kOffQ + (2*qb + X) * kTile
  static constexpr int kOffK = kQBuf * 2 * kTile;
  static constexpr int kOffV = kOffK + kKSt * kTile;
  static constexpr int kOffBar = kOffV + kVSt * kTile;
  // q_full[2], q_empty[2], k_full[4], k_empty[4], v_full[4], v_empty[4], v_land,
  // s_full[2], (unused)[2], p_full[2], pv_done[2], o_empty[2], fin
  static constexpr int kNumBar = 2 + 2 + 4 + 4 + 4 + 4 + 1 + 2 + 2 + 2 + 2 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kSmem = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColS = 0;     // S_X (and P_X) at 128*X
  static constexpr uint32_t kColO = 256;   // O_X at 256 + D*X
};

// Everything the roles need to know about one work item.  Computed the same
// way by every role from the item number alone.
struct PairItem {
  int b, h, r, delta, n_r, set, m0, Lb, Lm, bh;
  bool zero;        // no valid row in the pair: output zeros only
  int act[2];       // tile X has at least one valid row
  int U0, nU, nE;   // first key (m coordinate) of the band entries, their count, all entries
  int khi;          // last key any row of the pair attends in the band
  int b0[2], nb[2]; // band entries of tile X: [b0, b0 + nb)
  int klo[2], kend[2]; // first and last key (m coordinate) tile X attends in the band
  int gcnt[2];      // global tokens visible to tile X (a prefix of the sorted list)
  int ngt[2];       // global entries of tile X
  int gbase[2];     // first global entry of tile X
  int len[2];       // entries tile X consumes
  bool gsplit;      // causal: each tile has global entries of its own
};

__device__ __forceinline__ int upper_bound_gidx(const BandParams& p, int lim) {
  // number of global positions <= lim (gidx is strictly increasing)
  int lo = 0, hi = p.G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (p.gidx[mid] <= lim) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ PairItem decode_pair(const BandParams& p, int item) {
  PairItem it;
  it.b = item / p.items_per_b;
  const int rem = item - it.b * p.items_per_b;
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seg[mid].begin <= rem) lo = mid; else hi = mid - 1;
  }
  const BandSeg& sg = p.seg[lo];
  it.h = sg.h;
  it.r = sg.r;
  it.delta = sg.delta;
  it.n_r = sg.n_r;
  it.set = sg.set;
  it.m0 = (rem - sg.begin) * 256;
  it.bh = it.b * p.H + it.h;
  it.Lb = p.n - p.pad[it.b];
  const int Lm = (it.Lb > it.r) ? (it.Lb - it.r + it.delta - 1) / it.delta : 0;
  it.Lm = min(Lm, it.n_r);
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    const int q0 = it.m0 + 128 * X;
    it.act[X] = q0 < it.Lm;
    const int qlast = min(q0 + 127, it.Lm - 1);
    it.klo[X] = max(0, q0 - p.half);
    it.kend[X] = min(it.Lm - 1, qlast + p.right);
    int glim = it.Lb - 1;
    if (p.causal) glim = min(glim, it.r + it.delta * qlast);
    it.gcnt[X] = (it.act[X] && p.G > 0) ? upper_bound_gidx(p, glim) : 0;
    it.ngt[X] = (it.gcnt[X] + 127) >> 7;
  }
  it.zero = !it.act[0];
  if (it.zero) {
    it.nE = it.nU = 0;
    it.len[0] = it.len[1] = 0;
    return it;
  }
  it.U0 = it.klo[0];
  it.khi = it.act[1] ? it.kend[1] : it.kend[0];
  it.nU = (it.khi - it.U0) / 128 + 1;
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    if (it.act[X]) {
      it.b0[X] = (it.klo[X] - it.U0) / 128;
      it.nb[X] = (it.kend[X] - it.U0) / 128 - it.b0[X] + 1;
    } else {
      it.b0[X] = 0;
      it.nb[X] = 0;
    }
    it.len[X] = it.nb[X] + it.ngt[X];
  }
  // global entries: shared by both tiles unless causal (then each tile sees its own prefix)
  it.gbase[0] = it.nU;
  it.gsplit = p.causal != 0;
  if (it.gsplit) {
    it.gbase[1] = it.nU + it.ngt[0];
    it.nE = it.nU + it.ngt[0] + it.ngt[1];
  } else {
    it.gbase[1] = it.nU;
    it.nE = it.nU + max(it.ngt[0], it.ngt[1]);
  }
  return it;
}

// entry consumed by tile X at its step j
__device__ __forceinline__ int entry_of(const PairItem& it, int X, int j) {
  const int nb = X ? it.nb[1] : it.nb[0];
  return j < nb ? (X ? it.b0[1] : it.b0[0]) + j : (X ? it.gbase[1] : it.gbase[0]) + (j - nb);
}

// step at which tile Y consumes entry e, or -1
__device__ __forceinline__ int step_of(const PairItem& it, int Y, int e) {
  if (!(Y ? it.act[1] : it.act[0])) return -1;
  const int nb = Y ? it.nb[1] : it.nb[0];
  if (e < it.nU) {
    const int j = e - (Y ? it.b0[1] : it.b0[0]);
    return (j >= 0 && j < nb) ? j : -1;
  }
  const int g = e - (Y ? it.gbase[1] : it.gbase[0]);
  return (g >= 0 && g < (Y ? it.ngt[1] : it.ngt[0])) ? nb + g : -1;
}

// The MMAs of an item are issued in the order of (step, tile); the entry may
// be released after the product of its last consumer in that order.
__device__ __forceinline__ bool last_consumer(const PairItem& it, int X, int j) {
  const int jy = step_of(it, 1 - X, entry_of(it, X, j));
  return jy < 0 || j > jy || (j == jy && X == 1);
}

// global entry e (>= nU): the tile whose visible set it holds, and its tile index
__device__ __forceinline__ void global_entry(const PairItem& it, int e, int& X, int& gt) {
  if (!it.gsplit || e < it.gbase[0] + it.ngt[0]) {
    X = 0;
    gt = e - it.gbase[0];
  } else {
    X = 1;
    gt = e - it.gbase[1];
  }
}

// a[X] for a two-element member array without dynamic indexing (which would
// send the whole item descriptor to local memory)
__device__ __forceinline__ int pick(const int (&a)[2], int X) { return X ? a[1] : a[0]; }

__device__ __forceinline__ int global_count(const PairItem& it, int X, int gt) {
  return min(128, pick(it.gcnt, X) - 128 * gt);
}

template <int D>
struct BandSmem {
  using C = BandCfg<D>;
  uint8_t* base;
  uint32_t sbase;
  __device__ __forceinline__ uint32_t q(int qb, int X) const { return sbase + C::kOffQ + (2 * qb + X) * C::kTile; }
  __device__ __forceinline__ uint32_t k(int s) const { return sbase + C::kOffK + s * C::kTile; }
  __device__ __forceinline__ uint32_t v(int s) const { return sbase + C::kOffV + s * C::kTile; }
  __device__ __forceinline__ uint8_t* k_ptr(int s) const { return base + C::kOffK + s * C::kTile; }
  __device__ __forceinline__ uint8_t* v_ptr(int s) const { return base + C::kOffV + s * C::kTile; }
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + C::kOffBar + 8 * i; }
  __device__ __forceinline__ uint32_t q_full(int b) const { return bar(0 + b); }
  __device__ __forceinline__ uint32_t q_empty(int b) const { return bar(2 + b); }
  __device__ __forceinline__ uint32_t k_full(int s) const { return bar(4 + s); }
  __device__ __forceinline__ uint32_t k_empty(int s) const { return bar(8 + s); }
  __device__ __forceinline__ uint32_t v_full(int s) const { return bar(12 + s); }
  __device__ __forceinline__ uint32_t v_empty(int s) const { return bar(16 + s); }
  __device__ __forceinline__ uint32_t v_land() const { return bar(20); }
  __device__ __forceinline__ uint32_t s_full(int X) const { return bar(21 + X); }
  __device__ __forceinline__ uint32_t p_full(int X) const { return bar(25 + X); }
  __device__ __forceinline__ uint32_t pv_done(int X) const { return bar(27 + X); }
  __device__ __forceinline__ uint32_t o_empty(int X) const { return bar(29 + X); }
  __device__ __forceinline__ uint32_t fin() const { return bar(31); }
  __device__ __forceinline__ uint32_t* tmem_holder() const { return reinterpret_cast<uint32_t*>(base + C::kOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + C::kOffMisc + 4); }
};

// 16-byte chunk `ch` of row `row` inside a [rows, D] bf16 tile stored as D/64
// blocks of [128 rows, 64] with the 128-byte swizzle TMA uses.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
  return (uint32_t)((ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// m coordinate of global position g in residue class r, or a value that is
// never inside a band when g is not in the class
__device__ __forceinline__ int residue_coord(int g, int r, int delta) {
  if (delta == 1) return g;
  const int d = g - r;
  return (d >= 0 && d % delta == 0) ? d / delta : -(1 << 29);
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void band_producer(const BandParams& p, const BandSmem<D>& sm, int lane) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  uint32_t kv = 0, q_it = 0, land = 0;
  int land_pending = -1;  // v_land phase of a zeroing load not yet seen to land
  int last_k[C::kKSt], last_v[C::kVSt], last_q[C::kQBuf];
#pragma unroll
  for (int s = 0; s < C::kKSt; ++s) last_k[s] = -1;
#pragma unroll
  for (int s = 0; s < C::kVSt; ++s) last_v[s] = -1;
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s) last_q[s] = -1;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const PairItem it = decode_pair(p, item);
    if (it.zero) continue;

    // ---- Q of both tiles
    const int qb = q_it % C::kQBuf;
    if (!warp_wait(sm.q_empty(qb), ((q_it / C::kQBuf) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
    if (lane == 0) {
      mbar_arrive_expect_tx(sm.q_full(qb), (it.act[1] ? 2 : 1) * C::kTile);
#pragma unroll
      for (int X = 0; X < 2; ++X) {
        if (!it.act[X]) continue;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm.q(qb, X) + c * 16384, &p.tq[it.set], c * 64, it.m0 + 128 * X, it.bh, sm.q_full(qb));
      }
    }
    last_q[qb] = (int)q_it;
    ++q_it;

    const __nv_bfloat16* kb = p.k + (size_t)it.bh * p.n * D;
    const __nv_bfloat16* vb = p.v + (size_t)it.bh * p.n * D;
    constexpr int CH = D / 8;  // 16-byte chunks per row

    for (int e = 0; e < it.nE; ++e, ++kv) {
      const int ks = kv % C::kKSt, vs = kv % C::kVSt;
      // ---------------- K
      if (!warp_wait(sm.k_empty(ks), ((kv / C::kKSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (e < it.nU) {
        if (lane == 0) {
          mbar_arrive_expect_tx(sm.k_full(ks), C::kTile);
          const int y = it.U0 + 128 * e;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sm.k(ks) + c * 16384, &p.tk[it.set], c * 64, y, it.bh, sm.k_full(ks));
        }
        last_k[ks] = (int)kv;
      } else {
        int X, gt;
        global_entry(it, e, X, gt);
        const int cnt = global_count(it, X, gt);
        const int ng = (cnt + 15) & ~15;
        uint8_t* dst = sm.k_ptr(ks);
        for (int idx = lane; idx < ng * CH; idx += 32) {
          const int row = idx / CH, ch = idx - (idx / CH) * CH;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (row < cnt) x = __ldg(reinterpret_cast<const uint4*>(kb + (size_t)p.gidx[128 * gt + row] * D) + ch);
          *reinterpret_cast<uint4*>(dst + sw128_offset(row, ch)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.k_full(ks));
        last_k[ks] = -1;  // completed synchronously
      }
      // ---------------- V
      if (!warp_wait(sm.v_empty(vs), ((kv / C::kVSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (e < it.nU) {
        const int y = it.U0 + 128 * e;
        // rows past the last key any row of the pair attends (padding, or the
        // end of the window union) but inside the tensor are zeroed, so that
        // whatever they hold cannot reach the output through 0 * value
        const int z0 = it.khi - y + 1, z1 = min(128, it.n_r - y);
        if (z0 < z1) {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_land(), C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sm.v(vs) + c * 16384, &p.tv[it.set], c * 64, y, it.bh, sm.v_land());
          }
          land_pending = (int)land;
          const bool landed = warp_wait(sm.v_land(), land & 1, abort, kRoleProducer);
          ++land;
          if (!landed) { ok = false; break; }
          land_pending = -1;
          uint8_t* dst = sm.v_ptr(vs);
          for (int idx = lane; idx < (z1 - z0) * CH; idx += 32) {
            const int row = z0 + idx / CH, ch = idx - (idx / CH) * CH;
            *reinterpret_cast<uint4*>(dst + sw128_offset(row, ch)) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.v_full(vs));
          last_v[vs] = -1;
        } else {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_full(vs), C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sm.v(vs) + c * 16384, &p.tv[it.set], c * 64, y, it.bh, sm.v_full(vs));
          }
          last_v[vs] = (int)kv;
        }
      } else {
        int X, gt;
        global_entry(it, e, X, gt);
        const int cnt = global_count(it, X, gt);
        const int ng = (cnt + 15) & ~15;
        uint8_t* dst = sm.v_ptr(vs);
        for (int idx = lane; idx < ng * CH; idx += 32) {
          const int row = idx / CH, ch = idx - (idx / CH) * CH;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (row < cnt) x = __ldg(reinterpret_cast<const uint4*>(vb + (size_t)p.gidx[128 * gt + row] * D) + ch);
          *reinterpret_cast<uint4*>(dst + sw128_offset(row, ch)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.v_full(vs));
        last_v[vs] = -1;
      }
    }
  }
  // Let every TMA copy this warp issued land before the CTA can exit.
  int dummy = 0;
#pragma unroll
  for (int s = 0; s < C::kKSt; ++s)
    if (last_k[s] >= 0) mbar_wait(sm.k_full(s), ((uint32_t)last_k[s] / C::kKSt) & 1, &dummy, kRoleDrain, 200000000ull);
#pragma unroll
  for (int s = 0; s < C::kVSt; ++s)
    if (last_v[s] >= 0) mbar_wait(sm.v_full(s), ((uint32_t)last_v[s] / C::kVSt) & 1, &dummy, kRoleDrain, 200000000ull);
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s)
    if (last_q[s] >= 0) mbar_wait(sm.q_full(s), ((uint32_t)last_q[s] / C::kQBuf) & 1, &dummy, kRoleDrain, 200000000ull);
  if (land_pending >= 0) mbar_wait(sm.v_land(), (uint32_t)land_pending & 1, &dummy, kRoleDrain, 200000000ull);
}

// ------------------------------------------------------------------ MMA issuer (one thread)
template <int D>
__device__ void band_mma(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
  uint32_t kv = 0, q_it = 0;
  uint32_t p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const PairItem it = decode_pair(p, item);
    if (it.zero) continue;
    const int qb = q_it % C::kQBuf;
    if (!mbar_wait(sm.q_full(qb), (q_it / C::kQBuf) & 1, abort, kRoleMma)) { ok = false; break; }
    ++q_it;
    tc_fence_after();
    const int s_total = it.len[0] + it.len[1];
    int s_done = 0;

    // columns of the entry (128 for band entries, the padded global count otherwise)
    auto ncols = [&](int X, int e) -> int {
      if (e < it.nU) return 128;
      int Xg, gt;
      global_entry(it, e, Xg, gt);
      return (global_count(it, Xg, gt) + 15) & ~15;
    };

    auto issue_s = [&](int X, int j) -> bool {
      const int e = entry_of(it, X, j);
      const uint32_t ke = kv + e;
      const int ks = ke % C::kKSt;
      if (!mbar_wait(sm.k_full(ks), (ke / C::kKSt) & 1, abort, kRoleMma)) return false;
      tc_fence_after();
      const int N = ncols(X, e);
      const uint32_t idesc = idesc_bf16_f32(128, N, 0);
      const uint32_t dt = tmem + C::kColS + 128 * X;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qa = sm.q(qb, X) + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t ka = sm.k(ks) + (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16_ss(dt, smem_desc_sw128(qa, 16, 1024), smem_desc_sw128(ka, 16, 1024), idesc, kk > 0);
      }
      mma_commit(sm.s_full(X));
      if (last_consumer(it, X, j)) mma_commit(sm.k_empty(ks));
      if (++s_done == s_total) mma_commit(sm.q_empty(qb));  // Q may be replaced
      return true;
    };

    auto issue_pv = [&](int X, int j) -> bool {
      const int e = entry_of(it, X, j);
      const uint32_t ve = kv + e;
      const int vs = ve % C::kVSt;
      if (!mbar_wait(sm.v_full(vs), (ve / C::kVSt) & 1, abort, kRoleMma)) return false;
      if (!mbar_wait(sm.p_full(X), p_cnt[X] & 1, abort, kRoleMma)) return false;
      ++p_cnt[X];
      if (j == 0) {
        if (!mbar_wait(sm.o_empty(X), (o_cnt[X] & 1) ^ 1, abort, kRoleMma)) return false;
        ++o_cnt[X];
      }
      tc_fence_after();
      // key steps of 16 that some row of tile X attends: value rows outside
      // them (the partner tile's keys) are never read
      int kk0 = 0, kk1 = ncols(X, e) / 16 - 1;
      if (e < it.nU) {
        const int kb = it.U0 + 128 * e;
        kk0 = max(0, pick(it.klo, X) - kb) >> 4;
        kk1 = min(127, pick(it.kend, X) - kb) >> 4;
      }
      const uint32_t pt = tmem + C::kColS + 128 * X;
      const uint32_t ot = tmem + C::kColO + D * X;
      for (int kk = kk0; kk <= kk1; ++kk) {
        const uint32_t va = sm.v(vs) + kk * 2048;
        mma_bf16_ts(ot, pt + kk * 8, smem_desc_sw128(va, 16384, 1024), idesc_pv, (j > 0 || kk > kk0) ? 1u : 0u);
      }
      if (j + 1 == pick(it.len, X)) mma_commit(sm.pv_done(X));  // O_X complete
      if (last_consumer(it, X, j)) mma_commit(sm.v_empty(vs));
      return true;
    };

#pragma unroll
    for (int X = 0; X < 2; ++X)
      if (ok && pick(it.len, X) > 0 && !issue_s(X, 0)) ok = false;
    const int steps = max(it.len[0], it.len[1]);
    for (int j = 0; ok && j < steps; ++j) {
#pragma unroll
      for (int X = 0; X < 2; ++X) {
        const int lenX = pick(it.len, X);
        if (!ok || j >= lenX) continue;
        if (!issue_pv(X, j)) ok = false;
        else if (j + 1 < lenX && !issue_s(X, j + 1)) ok = false;
      }
    }
    kv += it.nE;
  }
  // Wait until every MMA this thread issued has finished before TMEM is freed.
  mma_commit(sm.fin());
  int dummy = 0;
  mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, 200000000ull);
}

// ------------------------------------------------------------------ softmax / epilogue
// Lazy rescaling: the running maximum of a row is raised only when a new
// score exceeds it by more than kLazy in the exp2 domain, so that O is
// rescaled rarely; P values stay below 2^kLazy.
constexpr float kLazy = 8.0f;

// Bits [lo, hi] of a 32-bit word (empty when hi < lo); lo, hi may lie outside [0, 31].
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 31);
  if (hi < lo) return 0u;
  const uint32_t upto = (hi == 31) ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
  return upto & ~((1u << lo) - 1u);
}

// Softmax of tile X (one query row per thread; warp quarter wq of TMEM lanes).
template <int D>
__device__ void band_softmax(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem, int X,
                             int wq, int lane) {
  using C = BandCfg<D>;
  volatile int* abort = sm.abort_flag();
  const int row = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS + 128 * X;  // S_X, then P_X
  const uint32_t tO = tmem + lane_base + C::kColO + D * X;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float sl2 = p.sl2;
  uint32_t s_cnt = 0, pv_cnt = 0;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const PairItem it = decode_pair(p, item);
    const int m_q = it.m0 + 128 * X + row;
    const bool row_exists = m_q < it.n_r;
    const bool row_valid = m_q < it.Lm;
    if (it.zero || !(X ? it.act[1] : it.act[0])) {
      if (row_exists) {
        uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + it.r + (size_t)it.delta * m_q) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const int len = pick(it.len, X), nb = pick(it.nb, X), b0 = pick(it.b0, X), gb = pick(it.gbase, X);
    float m_run = NEG_INF, l_run = 0.f;

    for (int j = 0; j < len; ++j) {
      const bool is_band = j < nb;
      const int e = is_band ? b0 + j : gb + (j - nb);
      // ---- keep[c]: bit t set where this row attends column 32c + t
      uint32_t keep[4];
      if (is_band) {
        const int kb = it.U0 + 128 * e;
        int clo = m_q - p.half - kb;
        int chi = min(m_q + p.right, it.Lm - 1) - kb;
        if (!row_valid) chi = clo - 1;
#pragma unroll
        for (int c = 0; c < 4; ++c) keep[c] = bit_range(clo - 32 * c, chi - 32 * c);
      } else {
        int gx, gt;
        global_entry(it, e, gx, gt);
        const int gcnt = global_count(it, gx, gt);
        const int i_q = it.r + it.delta * m_q;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t k = 0;
          const int tend = max(0, min(32, gcnt - 32 * c));
#pragma unroll 1
          for (int t = 0; t < tend; ++t) {
            const int g = p.gidx[128 * gt + 32 * c + t];
            const int mg = residue_coord(g, it.r, it.delta);
            const bool in_band = (m_q - mg <= p.half) && (mg - m_q <= p.right);
            k |= (uint32_t)((!p.causal || g <= i_q) && !in_band) << t;
          }
          keep[c] = row_valid ? k : 0u;
        }
      }
      // chunks some lane of the warp needs, and chunks every lane needs whole
      uint32_t on = 0, full = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (__any_sync(0xffffffffu, keep[c] != 0u)) on |= 1u << c;
        if (__all_sync(0xffffffffu, keep[c] == 0xffffffffu)) full |= 1u << c;
      }

      // S_X(j) complete; it was issued after P_X(j-1).V, so that is complete too
      if (!warp_wait(sm.s_full(X), s_cnt & 1, abort, kRoleSoftmax)) { ok = false; break; }
      ++s_cnt;
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_nw(tS + 32 * c, sr + 32 * c);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(sr + 32 * c);
      float* s = reinterpret_cast<float*>(sr);

      // ---- masks, and the maximum of the raw scores (the scale is positive)
      float mx = NEG_INF;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (!(full & (1u << c))) {
#pragma unroll
          for (int t = 0; t < 32; ++t) s[32 * c + t] = ((keep[c] >> t) & 1u) ? s[32 * c + t] : NEG_INF;
        }
#pragma unroll
        for (int t = 0; t < 32; t += 2) mx = max3f(mx, s[32 * c + t], s[32 * c + t + 1]);
      }
      const float mt = mx * sl2;
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_run + kLazy) {
        alpha = ex2_approx(m_run - mt);  // 0 while m_run is -inf
        m_run = mt;
        resc = true;
      }
      // ---- O_X *= alpha where the maximum moved (O_X is overwritten at j = 0)
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32_nw(tO + 32 * c, o);
          tmem_wait_ld();
          reg_fence32(o);
          float2* of = reinterpret_cast<float2*>(o);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int t = 0; t < 16; ++t) of[t] = __fmul2_rn(of[t], a2);
          tmem_st16_nw(tO + 32 * c, o);
          tmem_st16_nw(tO + 32 * c + 16, o + 16);
        }
      }
      // ---- P = exp2(s * scale - m) chunk by chunk into TMEM, row sum
      const float mneg = (m_run == NEG_INF) ? 0.f : -m_run;
      float2 sum2 = make_float2(0.f, 0.f);
      const float2 sc2 = make_float2(sl2, sl2), of2 = make_float2(mneg, mneg);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
        if (on & (1u << c)) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float2 x = __ffma2_rn(make_float2(s[32 * c + 2 * t], s[32 * c + 2 * t + 1]), sc2, of2);
            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            sum2 = __fadd2_rn(sum2, make_float2(p0, p1));
            pk[t] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) pk[t] = 0u;
        }
        tmem_st16_nw(tS + 16 * c, pk);
      }
      l_run = l_run * alpha + (sum2.x + sum2.y);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(X));
    }
    if (!ok) break;

    // ---- epilogue: O / l -> bf16 (32 columns at a time) -> global
    if (!warp_wait(sm.pv_done(X), pv_cnt & 1, abort, kRoleSoftmax)) { ok = false; break; }
    ++pv_cnt;
    tc_fence_after();
    const float inv = (row_valid && l_run > 0.f) ? 1.0f / l_run : 0.f;
    uint32_t ob[D / 2];  // the row in bf16 pairs
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32_nw(tO + 32 * c, o);
      tmem_wait_ld();
      reg_fence32(o);
      const float* of = reinterpret_cast<const float*>(o);
#pragma unroll
      for (int t = 0; t < 16; ++t) ob[16 * c + t] = pack_bf16x2(of[2 * t] * inv, of[2 * t + 1] * inv);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.o_empty(X));
    if (row_exists) {
      uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + it.r + (size_t)it.delta * m_q) * D);
      // padded rows (inv = 0) are written as zeros; O is finite there since
      // every value row such a row could meet is finite or zeroed
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        orow[c] = row_valid ? make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3])
                            : make_uint4(0, 0, 0, 0);
    }
  }
}

// Three warpgroups: two of softmax warps, one holding the producer warp, the
// MMA warp and two idle warps.  Launched at 168 registers per thread
// (384 x 168 = 64512 of the SM's 65536), the third warpgroup gives registers
// back (setmaxnreg.dec to kRegsOther) and the softmax warpgroups take them
// (setmaxnreg.inc to kRegsSoftmax): 256 x 200 + 128 x 96 = 63488 <= 64512.
constexpr int kBandThreads = 384;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 96;
constexpr int kRegsAtLaunchMin = (256 * kRegsSoftmax + 128 * kRegsOther + kBandThreads - 1) / kBandThreads;

template <int D>
__global__ void __launch_bounds__(kBandThreads, 1) band_tc_kernel(const __grid_constant__ BandParams p) {
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm.q_full(b), 1);
      mbar_init(sm.q_empty(b), 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 1);
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 1);
    }
    mbar_init(sm.v_land(), 1);
    for (int X = 0; X < 2; ++X) {
      mbar_init(sm.s_full(X), 1);
      mbar_init(sm.p_full(X), 4);
      mbar_init(sm.pv_done(X), 1);
      mbar_init(sm.o_empty(X), 4);
    }
    mbar_init(sm.fin(), 1);
    *sm.abort_flag() = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(sm.tmem_holder()), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder();

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    band_softmax<D>(p, sm, tmem, warp >> 2, warp & 3, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == 8) {
      band_producer<D>(p, sm, lane);
    } else if (warp == 9) {
      if (lane == 0) band_mma<D>(p, sm, tmem);
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
    // The register hand-over between warpgroups needs the launch allocation
    // it was planned for; with fewer registers setmaxnreg.inc could never be
    // satisfied, so refuse to launch rather than wait.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, band_tc_kernel<D>);
    if (e != cudaSuccess) {
      set_error("cudaFuncGetAttributes(band kernel): %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
    if (fa.numRegs < kRegsAtLaunchMin || fa.numRegs * kBandThreads > 65536) {
      set_error("band kernel built with %d registers per thread; its register split needs %d..%d",
                fa.numRegs, kRegsAtLaunchMin, 65536 / kBandThreads);
      return LF_ERR_UNSUPPORTED;
    }
    attr_set = true;
  }
  band_tc_kernel<D><<<grid, kBandThreads, C::kSmem, s>>>(p);
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
