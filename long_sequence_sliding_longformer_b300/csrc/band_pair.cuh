// band_pair.cuh -- bf16 band-attention kernel for D = 128 on the sm_103a tensor
// cores: two 128-row query tiles per CTA sharing their key/value entries.
//
// Computes the sliding / dilated / causal window part of Longformer attention
// (velog.io/@lainshower/Longformer, section 3-1 "Sliding Window", "Dilated
// Sliding Window", section 4.1 for the look-back-only pattern) plus the
// global tokens' key columns ("Global Attention"), for every row except the
// rows at global tokens' positions, which the global-row pass writes (it may
// run at the same time).
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
//   warp 0     allocates TMEM; V producer: TMA loads of the V entries into
//              a ring of shared-memory slots, gathers of global-token rows
//   warp 1     Q/K producer: TMA loads of Q and of the K entries
//   warps 2-3  no role (they keep the register split of the warpgroups)
//   warps 4-7  softmax of tile 0, warps 8-11 softmax of tile 1: one query row
//              per thread; S rows are read from TMEM, masked, turned into
//              P = exp2(S*scale - m) with a lazily updated row maximum, and P
//              (bf16) is written back to TMEM; an elected lane of the tile's
//              first warp then issues the tile's tcgen05.mma products,
//              O_X += P_X V (V read MN-major straight from the TMA slot: the
//              instruction descriptor's transpose bit, the two 64-column
//              boxes one leading-dimension offset apart) and the next
//              S_X = Q_X K^T (both operands in shared memory)
// While the softmax warps of one tile compute, the tensor cores can run the
// other tile's products.
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
namespace pairk {

template <int D>
struct BandCfg {
  static constexpr int kQBuf = 1;                  // Q is reloaded ~2 steps before an item ends
  static constexpr int kKSt = (D == 64) ? 5 : 2;   // K slots
  static constexpr int kVSt = 3;                   // V slots (as loaded: [keys, D]; the P.V operand)
  static constexpr int kTile = 128 * D * 2;     // bytes of one [128, D] bf16 tile
  static constexpr int kOffQ = 0;               // Q[qb][X] at kOffQ + (2*qb + X) * kTile
  static constexpr int kOffK = kQBuf * 2 * kTile;
  static constexpr int kOffV = kOffK + kKSt * kTile;
  static constexpr int kOffBar = kOffV + kVSt * kTile;
  // q_full[2], q_empty[2], k_full[8], k_empty[8], v_full[4], v_empty[4], v_land,
  // s_full[2], (unused)[2], p_full[2], pv_done[2], (unused)[2], fin, (unused)[8]
  static constexpr int kNumBar = 2 + 2 + 8 + 8 + 4 + 4 + 1 + 2 + 2 + 2 + 2 + 2 + 1 + 4 + 4;
  static_assert(kKSt <= 8 && kVSt <= 4 && kQBuf <= 2, "barrier arrays");
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kSmem = kOffMisc + 16 + kMaxSeg * (int)sizeof(BandSeg) + 32 + 1024;  // + slack to align the base to 1024
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kColS = 0;     // S_X at 128*X
  static constexpr uint32_t kColO = 256;   // O_X at 256 + D*X

};

// Everything the roles need to know about one work item.  Computed the same
// way by every role from the item number alone.
struct PairItem {
  int b, h, r, delta, n_r, set, m0, Lb, Lm, bh;
  int half, right;  // the head's window reach in steps: back, ahead
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

// `segs`: the launch's segment table, copied to shared memory at kernel start
// (a search over the kernel parameters would miss the constant cache).
__device__ __forceinline__ PairItem decode_pair(const BandParams& p, const BandSeg* segs, int item) {
  PairItem it;
  it.b = item / p.items_per_b;
  const int rem = item - it.b * p.items_per_b;
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].begin <= rem) lo = mid; else hi = mid - 1;
  }
  const BandSeg sg = segs[lo];
  it.h = sg.h;
  it.r = sg.r;
  it.delta = sg.delta;
  it.half = sg.half;
  it.right = p.causal ? 0 : sg.half;
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
    it.klo[X] = max(0, q0 - it.half);
    it.kend[X] = min(it.Lm - 1, qlast + it.right);
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
  __device__ __forceinline__ uint32_t k_empty(int s) const { return bar(12 + s); }
  __device__ __forceinline__ uint32_t v_full(int s) const { return bar(20 + s); }
  __device__ __forceinline__ uint32_t v_empty(int s) const { return bar(24 + s); }
  __device__ __forceinline__ uint32_t v_land() const { return bar(28); }
  __device__ __forceinline__ uint32_t s_full(int X) const { return bar(29 + X); }
  __device__ __forceinline__ uint32_t p_full(int X) const { return bar(33 + X); }
  __device__ __forceinline__ uint32_t pv_done(int X) const { return bar(35 + X); }
  __device__ __forceinline__ uint32_t fin() const { return bar(39); }
  __device__ __forceinline__ uint32_t* tmem_holder() const { return reinterpret_cast<uint32_t*>(base + C::kOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + C::kOffMisc + 4); }
  __device__ __forceinline__ BandSeg* segs() const { return reinterpret_cast<BandSeg*>(base + C::kOffMisc + 16); }
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

// ------------------------------------------------------------------ producers
// Two warps: KV = false loads Q and the K entries, KV = true the V entries,
// so that a full V ring (waiting for the P.V products) never holds back the
// K an S product needs.
template <int D, bool kIsV>
__device__ void band_producer(const BandParams& p, const BandSmem<D>& sm, int lane) {
  using C = BandCfg<D>;
  constexpr int kSt = kIsV ? C::kVSt : C::kKSt;
  volatile int* abort = sm.abort_flag();
  uint32_t kv = 0, q_it = 0, land = 0;
  int land_pending = -1;  // v_land phase of a zeroing load not yet seen to land
  int last_fill[kSt], last_q[C::kQBuf];
#pragma unroll
  for (int s = 0; s < kSt; ++s) last_fill[s] = -1;
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s) last_q[s] = -1;
  bool ok = true;
  Tracer tr;
  if (blockIdx.x == 0 && lane == 0) tr.track = kIsV ? 5 : 3;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const PairItem it = decode_pair(p, sm.segs(), item);
    if (it.zero) continue;

    if (!kIsV) {
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
    }

    const __nv_bfloat16* src = (kIsV ? p.v : p.k) + (size_t)it.bh * p.n * D;
    const CUtensorMap* map = kIsV ? &p.tv[it.set] : &p.tk[it.set];
    constexpr int CH = D / 8;  // 16-byte chunks per row

    for (int e = 0; e < it.nE; ++e, ++kv) {
      const int slot = kv % kSt;
      const uint32_t full = kIsV ? sm.v_full(slot) : sm.k_full(slot);
      const uint32_t empty = kIsV ? sm.v_empty(slot) : sm.k_empty(slot);
      const uint32_t dst = kIsV ? sm.v(slot) : sm.k(slot);
      uint8_t* dst_ptr = kIsV ? sm.v_ptr(slot) : sm.k_ptr(slot);
      tr.ev(30);
      if (!warp_wait(empty, ((kv / kSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      tr.ev(31);
      if (e < it.nU) {
        const int y = it.U0 + 128 * e;
        // value rows past the last key any row of the pair attends (padding,
        // or the end of the window union) but inside the tensor are zeroed,
        // so that whatever they hold cannot reach the output through 0 * value
        const int z0 = it.khi - y + 1, z1 = min(128, it.n_r - y);
        if (kIsV && z0 < z1) {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_land(), C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(dst + c * 16384, map, c * 64, y, it.bh, sm.v_land());
          }
          land_pending = (int)land;
          const bool landed = warp_wait(sm.v_land(), land & 1, abort, kRoleProducer);
          ++land;
          if (!landed) { ok = false; break; }
          land_pending = -1;
          for (int idx = lane; idx < (z1 - z0) * CH; idx += 32) {
            const int row = z0 + idx / CH, ch = idx - (idx / CH) * CH;
            *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch)) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full);
          last_fill[slot] = -1;
        } else {
          if (lane == 0) {
            mbar_arrive_expect_tx(full, C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * 16384, map, c * 64, y, it.bh, full);
          }
          last_fill[slot] = (int)kv;
        }
      } else {
        // rows of the global tokens visible to the entry's tile, zeros after
        int X, gt;
        global_entry(it, e, X, gt);
        const int cnt = global_count(it, X, gt);
        const int ng = (cnt + 15) & ~15;
        for (int idx = lane; idx < ng * CH; idx += 32) {
          const int row = idx / CH, ch = idx - (idx / CH) * CH;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (row < cnt) x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)p.gidx[128 * gt + row] * D) + ch);
          *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
        last_fill[slot] = -1;  // completed synchronously
      }
      tr.ev(32);
    }
  }
  tr.done();
  // Let every TMA copy this warp issued land before the CTA can exit.
  int dummy = 0;
#pragma unroll
  for (int s = 0; s < kSt; ++s)
    if (last_fill[s] >= 0)
      mbar_wait(kIsV ? sm.v_full(s) : sm.k_full(s), ((uint32_t)last_fill[s] / kSt) & 1, &dummy, kRoleDrain, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s)
    if (last_q[s] >= 0) mbar_wait(sm.q_full(s), ((uint32_t)last_q[s] / C::kQBuf) & 1, &dummy, kRoleDrain, kDrainLimitNs);
  if (land_pending >= 0) mbar_wait(sm.v_land(), (uint32_t)land_pending & 1, &dummy, kRoleDrain, kDrainLimitNs);
}

// ------------------------------------------------------------------ MMA issue (per tile)
// Each softmax warpgroup issues the products of its own tile: after the four
// warps have written P_X(j) they meet at a named barrier, and one elected
// lane of the first warp issues O_X += P_X(j) V(j) and then S_X(j+1) =
// Q_X K(j+1)^T (in that order: S_X(j+1) overwrites P_X(j)).  The whole warp
// runs the bookkeeping so that descriptors stay in uniform registers.
//
// K and V slots are released by both tiles: each slot's "empty" barrier
// takes one arrival per tile and fill, from tcgen05.commit after the tile's
// last product that reads it, or a plain arrival from a tile that does not
// use the entry once that fill is visible (so the arrival cannot count
// towards the slot's previous fill).
template <int D>
struct TileIssuer {
  using C = BandCfg<D>;
  static constexpr uint32_t kTile16 = C::kTile >> 4;  // a slot, in descriptor address units
  const BandSmem<D>& sm;
  volatile int* abort;
  Tracer* tr = nullptr;
  int X;
  uint32_t tmem;
  uint64_t qdesc0, kdesc0, vdesc0;
  uint32_t idesc_s128, idesc_pv;

  __device__ TileIssuer(const BandSmem<D>& sm_, uint32_t tmem_, int X_)
      : sm(sm_), abort(sm_.abort_flag()), X(X_), tmem(tmem_) {
    qdesc0 = smem_desc_sw128(sm.q(0, 0), 16, 1024);
    kdesc0 = smem_desc_sw128(sm.k(0), 16, 1024);
    // V as loaded: MN-major (D contiguous), 64-column boxes of [128 keys,
    // 128 bytes] one after the other (the leading-dimension offset between
    // the boxes), 8-key groups 1024 bytes apart
    vdesc0 = smem_desc_sw128(sm.v(0), 128 * 128, 1024);
    idesc_s128 = idesc_bf16_f32(128, 128, 0);
    idesc_pv = idesc_bf16_f32(128, D, 1);
  }

  // columns of global entry e (its padded token count)
  __device__ __forceinline__ int gcols(const PairItem& it, int e) const {
    int Xg, gt;
    global_entry(it, e, Xg, gt);
    return (global_count(it, Xg, gt) + 15) & ~15;
  }

  // Entry e (fill kv + e) is not read by this tile: release its K slot
  // (skip_k) and its V slot (skip_v).  A tile must not wait for a V fill
  // it skips before issuing the P.V of its own earlier entries: with a
  // shallow ring that fill may need the very slot the P.V still holds.
  __device__ bool skip_k(uint32_t kv, int e) const {
    const uint32_t f = kv + e;
    const int ks = f % C::kKSt;
    if (!warp_wait(sm.k_full(ks), (f / C::kKSt) & 1, abort, kRoleSoftmax)) return false;
    if (elect_one()) mbar_arrive(sm.k_empty(ks));
    __syncwarp();
    return true;
  }
  __device__ bool skip_v(uint32_t kv, int e) const {
    const uint32_t f = kv + e;
    const int vs = f % C::kVSt;
    if (!warp_wait(sm.v_full(vs), (f / C::kVSt) & 1, abort, kRoleSoftmax)) return false;
    if (elect_one()) mbar_arrive(sm.v_empty(vs));
    __syncwarp();
    return true;
  }
  __device__ bool skip(uint32_t kv, int e) const { return skip_k(kv, e) && skip_v(kv, e); }

  // K(e) has landed
  __device__ bool wait_k(uint32_t kv, int e) const {
    const uint32_t f = kv + e;
    return warp_wait(sm.k_full(f % C::kKSt), (f / C::kKSt) & 1, abort, kRoleSoftmax);
  }
  // V(e) has landed
  __device__ bool wait_v(uint32_t kv, int e) const {
    const uint32_t f = kv + e;
    return warp_wait(sm.v_full(f % C::kVSt), (f / C::kVSt) & 1, abort, kRoleSoftmax);
  }

  // S_X = Q_X K(e)^T into TMEM (K(e) already waited for); `last_s` also releases Q
  __device__ bool issue_s(const PairItem& it, uint32_t kv, int qb, int e, bool last_s,
                          bool waited = false) const {
    const uint32_t f = kv + e;
    const int ks = f % C::kKSt;
    const uint32_t idesc = (e < it.nU) ? idesc_s128 : idesc_bf16_f32(128, gcols(it, e), 0);
    const uint64_t qd = qdesc0 + (2 * qb + X) * kTile16;
    const uint64_t kd = kdesc0 + ks * kTile16;
    const uint32_t dt = tmem + C::kColS + 128 * X;
    if (!waited && !wait_k(kv, e)) return false;
    if (tr) tr->ev(22);
    tc_fence_after();
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
        mma_bf16_ss(dt, qd + off, kd + off, idesc, kk > 0);
      }
      mma_commit(sm.s_full(X));
      mma_commit(sm.k_empty(ks));
      if (last_s) mma_commit(sm.q_empty(qb));
    }
    __syncwarp();
    if (tr) tr->ev(23);
    return true;
  }

  // O_X (+)= P_X V(e); `first` starts the accumulation, `last` signals O_X complete
  __device__ bool issue_pv(const PairItem& it, uint32_t kv, int e, bool first, bool last,
                           bool waited = false) const {
    const uint32_t f = kv + e;
    const int vs = f % C::kVSt;
    // key steps of 16 that some row of this tile attends: value rows outside
    // them (the partner tile's keys) are never read
    int kk0 = 0, kk1;
    if (e < it.nU) {
      const int kb = it.U0 + 128 * e;
      kk0 = max(0, pick(it.klo, X) - kb) >> 4;
      kk1 = min(127, pick(it.kend, X) - kb) >> 4;
    } else {
      kk1 = gcols(it, e) / 16 - 1;
    }
    const bool full = kk0 == 0 && kk1 == 7;
    const uint32_t acc0 = first ? 0u : 1u;
    const uint32_t pt = tmem + C::kColS + 128 * X;  // P_X over the first 64 columns of S_X
    const uint32_t ot = tmem + C::kColO + D * X;
    // V: a 16-key step is 16 rows of 128 bytes
    const uint64_t vd = vdesc0 + vs * kTile16;
    if (!waited && !wait_v(kv, e)) return false;
    if (tr) tr->ev(20);
    tc_fence_after();
    if (elect_one()) {
      if (full) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk * 16 * 128) >> 4;
          mma_bf16_ts(ot, pt + kk * 8, vd + off, idesc_pv, kk > 0 ? 1u : acc0);
        }
      } else {
        for (int kk = kk0; kk <= kk1; ++kk) {
          const uint32_t off = (kk * 16 * 128) >> 4;
          mma_bf16_ts(ot, pt + kk * 8, vd + off, idesc_pv, kk > kk0 ? 1u : acc0);
        }
      }
      if (last) mma_commit(sm.pv_done(X));  // O_X complete: the epilogue may read it
      mma_commit(sm.v_empty(vs));
    }
    __syncwarp();
    if (tr) tr->ev(21);
    return true;
  }
};

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

// Global entry e, chunk c: bit t set where this row attends global column
// 32c + t (a global key already in the row's band is counted there, once).
__device__ __forceinline__ uint32_t global_keep(const BandParams& p, const PairItem& it, int e, int c,
                                                int m_q, bool row_valid, int half, int right) {
  int gx, gt;
  global_entry(it, e, gx, gt);
  const int tend = max(0, min(32, global_count(it, gx, gt) - 32 * c));
  const int i_q = it.r + it.delta * m_q;
  uint32_t k = 0;
#pragma unroll 1
  for (int t = 0; t < tend; ++t) {
    const int g = p.gidx[128 * gt + 32 * c + t];
    const int mg = residue_coord(g, it.r, it.delta);
    const bool in_band = (m_q - mg <= half) && (mg - m_q <= right);
    k |= (uint32_t)((!p.causal || g <= i_q) && !in_band) << t;
  }
  return row_valid ? k : 0u;
}

// Maximum over the kept columns of a 32-column chunk of raw scores.
__device__ __forceinline__ float chunk_max(const uint32_t (&x)[32], uint32_t keep, uint32_t whole) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  float v[32];
  if (whole) {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(x[t]);
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = ((keep >> t) & 1u) ? __uint_as_float(x[t]) : NEG_INF;
  }
  float a = max3f(v[0], v[1], v[2]), b = max3f(v[3], v[4], v[5]), c = max3f(v[6], v[7], v[8]),
        d = max3f(v[9], v[10], v[11]);
#pragma unroll
  for (int t = 12; t < 28; t += 8) {
    a = max3f(a, v[t], v[t + 1]);
    b = max3f(b, v[t + 2], v[t + 3]);
    c = max3f(c, v[t + 4], v[t + 5]);
    d = max3f(d, v[t + 6], v[t + 7]);
  }
  return fmaxf(max3f(a, b, v[28]), max3f(c, d, max3f(v[29], v[30], v[31])));
}

// Relative position bias of a 32-column chunk, in place: x <- x * scale +
// bias(t0 + t) for t = 0..31 (scale = 1/sqrt(d); the exp2 scaling by log2(e)
// is applied with the maximum).  The step is clamped to the table [tlo, thi];
// a clamped column is masked anyway.
__device__ __forceinline__ void chunk_bias(uint32_t (&x)[32], float scale, const float* brow, int t0, int tlo,
                                           int thi) {
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const int st = min(max(t0 + t, tlo), thi);
    x[t] = __float_as_uint(fmaf(__uint_as_float(x[t]), scale, __ldg(brow + st)));
  }
}

// P for a 32-column chunk: p = exp2(s * sl2 - m) on the kept columns, 0
// elsewhere, packed to bf16 pairs; returns the two partial row sums.
__device__ __forceinline__ float2 chunk_exp(const uint32_t (&x)[32], uint32_t keep, uint32_t whole,
                                            float sl2, float mneg, uint32_t (&pk)[16]) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float2 sc2 = make_float2(sl2, sl2), of2 = make_float2(mneg, mneg);
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    float s0 = __uint_as_float(x[2 * t]), s1 = __uint_as_float(x[2 * t + 1]);
    if (!whole) {
      s0 = ((keep >> (2 * t)) & 1u) ? s0 : NEG_INF;
      s1 = ((keep >> (2 * t + 1)) & 1u) ? s1 : NEG_INF;
    }
    const float2 y = __ffma2_rn(make_float2(s0, s1), sc2, of2);
    const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
    if (t & 1) sb = __fadd2_rn(sb, make_float2(p0, p1));
    else sa = __fadd2_rn(sa, make_float2(p0, p1));
    pk[t] = pack_bf16x2(p0, p1);
  }
  return __fadd2_rn(sa, sb);
}

// Softmax of tile X (one query row per thread; warp quarter wq of TMEM lanes).
// kB: the band entries' scores carry the relative position bias.  kW: heads'
// windows differ (each item's reach comes from its segment).
template <int D, bool kB, bool kW>
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
  uint32_t s_cnt = 0, pv_cnt = 0, p_cnt = 0, kv = 0, q_it = 0;
  bool ok = true;
  const bool leader = wq == 0;  // issues this tile's MMAs
  TileIssuer<D> iss(sm, tmem, X);
  Tracer tr;
  if (blockIdx.x == 0 && wq == 0 && lane == 0) tr.track = X;
#ifdef LF_TRACE
  iss.tr = &tr;
#endif

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const PairItem it = decode_pair(p, sm.segs(), item);
    tr.ev(0);
    const int m_q = it.m0 + 128 * X + row;
    // rows at the positions of global tokens are written by the global-row
    // pass, which may run at the same time: this kernel leaves them alone
    bool write_row = m_q < it.n_r;
    if (p.G > 0) {
      const int m_t = it.m0 + 128 * X;
      const int i_lo = it.r + it.delta * m_t;
      const int i_hi = it.r + it.delta * min(m_t + 127, it.n_r - 1);
      if (m_t < it.n_r && upper_bound_gidx(p, i_hi) > upper_bound_gidx(p, i_lo - 1) && write_row) {
        const int i_q = it.r + it.delta * m_q;
        if (upper_bound_gidx(p, i_q) > upper_bound_gidx(p, i_q - 1)) write_row = false;
      }
    }
    const bool row_valid = m_q < it.Lm;
    if (it.zero || !(X ? it.act[1] : it.act[0])) {
      if (write_row) {
        uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + it.r + (size_t)it.delta * m_q) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      }
      if (!it.zero) {
        // the pair is active but this tile is not: release Q and every entry
        if (leader) {
          const int qb = q_it % C::kQBuf;
          if (!warp_wait(sm.q_full(qb), (q_it / C::kQBuf) & 1, abort, kRoleSoftmax)) { ok = false; break; }
          if (elect_one()) mbar_arrive(sm.q_empty(qb));
          __syncwarp();
          for (int e = 0; ok && e < it.nE; ++e) ok = iss.skip(kv, e);
          if (!ok) break;
        }
        kv += it.nE;
        ++q_it;
      }
      continue;
    }
    const int len = pick(it.len, X), nb = pick(it.nb, X), b0 = pick(it.b0, X), gb = pick(it.gbase, X);
    const int qb = q_it % C::kQBuf;
    auto entry = [&](int j) { return j < nb ? b0 + j : gb + (j - nb); };
    if (leader) {
      // Q, the entries before this tile's first one, and S_X(0)
      if (!warp_wait(sm.q_full(qb), (q_it / C::kQBuf) & 1, abort, kRoleSoftmax)) { ok = false; break; }
      for (int e = 0; ok && e < entry(0); ++e) ok = iss.skip(kv, e);
      if (!ok || !iss.issue_s(it, kv, qb, entry(0), len == 1)) { ok = false; break; }
    }
    float m_run = NEG_INF, l_run = 0.f;
    // the window reach of this item's head
    const int half = kW ? it.half : p.half, right = kW ? it.right : p.right;
    // the bias of this row's head, indexed by window step
    const float* brow = kB ? p.rel_bias + (size_t)it.h * p.rb_stride + p.rb_half : nullptr;

    for (int j = 0; j < len; ++j) {
      const bool is_band = j < nb;
      // with the bias, pass 1 writes the band scores back scaled and biased
      const bool scaled = kB && is_band;
      const int e = entry(j);
      // ---- keep c: bit t set where this row attends column 32c + t
      uint32_t keep0, keep1, keep2, keep3;
      if (is_band) {
        const int kb = it.U0 + 128 * e;
        const int clo = m_q - half - kb;
        int chi = min(m_q + right, it.Lm - 1) - kb;
        if (!row_valid) chi = clo - 1;
        keep0 = bit_range(clo, chi);
        keep1 = bit_range(clo - 32, chi - 32);
        keep2 = bit_range(clo - 64, chi - 64);
        keep3 = bit_range(clo - 96, chi - 96);
      } else {
        keep0 = global_keep(p, it, e, 0, m_q, row_valid, half, right);
        keep1 = global_keep(p, it, e, 1, m_q, row_valid, half, right);
        keep2 = global_keep(p, it, e, 2, m_q, row_valid, half, right);
        keep3 = global_keep(p, it, e, 3, m_q, row_valid, half, right);
      }
      // chunks some lane of the warp needs, and chunks every lane needs whole
      const uint32_t onm = (__any_sync(0xffffffffu, keep0 != 0u) ? 1u : 0u) |
                     (__any_sync(0xffffffffu, keep1 != 0u) ? 2u : 0u) |
                     (__any_sync(0xffffffffu, keep2 != 0u) ? 4u : 0u) |
                     (__any_sync(0xffffffffu, keep3 != 0u) ? 8u : 0u);
      const uint32_t fullm = (__all_sync(0xffffffffu, keep0 == ~0u) ? 1u : 0u) |
                             (__all_sync(0xffffffffu, keep1 == ~0u) ? 2u : 0u) |
                             (__all_sync(0xffffffffu, keep2 == ~0u) ? 4u : 0u) |
                             (__all_sync(0xffffffffu, keep3 == ~0u) ? 8u : 0u);

      // S_X(j) complete; it was issued after P_X(j-1).V, so that is complete too
      tr.ev(1);
      if (!warp_wait(sm.s_full(X), s_cnt & 1, abort, kRoleSoftmax)) { ok = false; break; }
      tr.ev(2);
      ++s_cnt;
      tc_fence_after();

      // ---- pass 1: row maximum of the raw scores (the scale is positive),
      // one 32-column chunk at a time (TMEM reads are cheap; the loop body
      // stays small for the instruction cache)
      float mx = NEG_INF;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        if (!((onm >> c) & 1u)) continue;
        uint32_t x[32];
        tmem_ld32_nw(tS + 32 * c, x);
        tmem_wait_ld();
        reg_fence32(x);
        const uint32_t kc = c == 0 ? keep0 : c == 1 ? keep1 : c == 2 ? keep2 : keep3;
        if (scaled) {
          chunk_bias(x, sl2 * (1.f / kLog2e), brow, it.U0 + 128 * e + 32 * c - m_q, -p.rb_half,
                     p.rb_stride - 1 - p.rb_half);
          tmem_st16_nw(tS + 32 * c, x);
          tmem_st16_nw(tS + 32 * c + 16, x + 16);
        }
        mx = fmaxf(mx, chunk_max(x, kc, (fullm >> c) & 1u));
      }
      if (scaled) tmem_wait_st();  // pass 2 reads the biased scores back
      const float mt = mx * (scaled ? kLog2e : sl2);
      tr.ev(3);
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
      // ---- pass 2: P = exp2(s * scale - m) chunk by chunk; P chunk c goes to
      // columns [16c, 16c + 16) of S_X, whose scores (chunk c/2) are already read
      const float mneg = (m_run == NEG_INF) ? 0.f : -m_run;
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
        if ((onm >> c) & 1u) {
          uint32_t x[32];
          tmem_ld32_nw(tS + 32 * c, x);
          tmem_wait_ld();
          reg_fence32(x);
          const uint32_t kc = c == 0 ? keep0 : c == 1 ? keep1 : c == 2 ? keep2 : keep3;
          sum2 = __fadd2_rn(sum2, chunk_exp(x, kc, (fullm >> c) & 1u, scaled ? kLog2e : sl2, mneg, pk));
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
      tr.ev(4);
      if (leader) {
        // While the other warps finish: the operands of this step's products,
        // and the entries this tile passes over.  Then all four warps have
        // written P_X(j) (a bounded wait, never bar.sync: a warp that gave up
        // must not leave the others blocked).
        const int e_next = (j + 1 < len) ? entry(j + 1) : it.nE;
        ok = iss.wait_v(kv, e);
        for (int e2 = e + 1; ok && e2 < e_next; ++e2) ok = iss.skip_k(kv, e2);
        if (ok && j + 1 < len) ok = iss.wait_k(kv, e_next);
        if (!ok || !warp_wait(sm.p_full(X), p_cnt & 1, abort, kRoleSoftmax)) { ok = false; break; }
        tr.ev(9);
        ++p_cnt;
        tc_fence_after();
        if (!iss.issue_pv(it, kv, e, j == 0, j + 1 == len, true)) { ok = false; break; }
        for (int e2 = e + 1; ok && e2 < e_next; ++e2) ok = iss.skip_v(kv, e2);
        if (!ok) break;
        // S_X(j+1) overwrites P_X(j): issued after the P.V that reads it
        if (j + 1 < len && !iss.issue_s(it, kv, qb, e_next, j + 2 == len, true)) { ok = false; break; }
        tr.ev(8);
      }
    }
    if (!ok) break;
    kv += it.nE;
    ++q_it;

    // ---- epilogue: O / l -> bf16 (32 columns at a time) -> global
    tr.ev(5);
    if (!warp_wait(sm.pv_done(X), pv_cnt & 1, abort, kRoleSoftmax)) { ok = false; break; }
    tr.ev(6);
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
    if (write_row) {
      uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + it.r + (size_t)it.delta * m_q) * D);
      // padded rows (inv = 0) are written as zeros; O is finite there since
      // every value row such a row could meet is finite or zeroed
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        orow[c] = row_valid ? make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3])
                            : make_uint4(0, 0, 0, 0);
    }
    tr.ev(7);
  }
  tr.done();
  if (leader) {
    // every MMA this tile issued must finish before TMEM is freed
    if (elect_one()) mma_commit(sm.fin());
    __syncwarp();
    int dummy = 0;
    mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, kDrainLimitNs);
    __syncwarp();
  }
}

// Three warpgroups: the producer warps and two warps without a role, then
// two of softmax warps.  Launched at 168 registers per thread
// (384 x 168 = 64512 of the SM's 65536), the third warpgroup gives registers
// back (setmaxnreg.dec to kRegsOther) and the softmax warpgroups take them
// (setmaxnreg.inc to kRegsSoftmax): 256 x 200 + 128 x 96 = 63488 <= 64512.
constexpr int kBandThreads = 384;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 96;
constexpr int kRegsAtLaunchMin = (256 * kRegsSoftmax + 128 * kRegsOther + kBandThreads - 1) / kBandThreads;

template <int D, bool kB, bool kW>
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
      mbar_init(sm.q_empty(b), 2);   // one arrival per tile
    }
    for (int s = 0; s < 8; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 2);   // one arrival per tile
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 2);   // one release per tile
    }
    mbar_init(sm.v_land(), 1);
    for (int X = 0; X < 2; ++X) {
      mbar_init(sm.s_full(X), 1);
      mbar_init(sm.p_full(X), 4);   // the tile's four softmax warps
      mbar_init(sm.pv_done(X), 1);
    }
    mbar_init(sm.fin(), 2);  // one commit per tile's issuing lane
    *sm.abort_flag() = 0;
    *cta_wait_limit(sm.abort_flag()) = wait_limit_ns();
    for (int i = 0; i < 8; ++i) reinterpret_cast<volatile int*>(sm.segs() + kMaxSeg)[i] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  for (int i = threadIdx.x; i < p.nseg; i += blockDim.x) sm.segs()[i] = p.seg[i];
  if (warp == 0) {
    tmem_alloc(smem_u32(sm.tmem_holder()), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder();

  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    band_softmax<D, kB, kW>(p, sm, tmem, (warp >> 2) - 1, warp & 3, lane);
  } else {
    // the issuing warps are the oldest of the CTA: the schedulers favour them
    // over the busy softmax warps that share their sub-partitions
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == 0) {
      band_producer<D, true>(p, sm, lane);
    } else if (warp == 1) {
      band_producer<D, false>(p, sm, lane);
    }  // warps 2-3: no role (P.V reads V as loaded)
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kB, bool kW>
static lf_status launch_band_tc_d(const BandParams& p, int grid, cudaStream_t s) {
  using C = BandCfg<D>;
  static std::atomic<uint64_t> attr_done{0};
  static std::atomic<bool> regs_checked{false};
  lf_status st = smem_attr_once((const void*)band_tc_kernel<D, kB, kW>, C::kSmem, attr_done, "band kernel");
  if (st != LF_OK) return st;
  if (!regs_checked.load(std::memory_order_acquire)) {
    cudaError_t e;
    // The register hand-over between warpgroups needs the launch allocation
    // it was planned for; with fewer registers setmaxnreg.inc could never be
    // satisfied, so refuse to launch rather than wait.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, band_tc_kernel<D, kB, kW>);
    if (e != cudaSuccess) {
      set_error("cudaFuncGetAttributes(band kernel): %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
    if (fa.numRegs < kRegsAtLaunchMin || fa.numRegs * kBandThreads > 65536) {
      set_error("band kernel built with %d registers per thread; its register split needs %d..%d",
                fa.numRegs, kRegsAtLaunchMin, 65536 / kBandThreads);
      return LF_ERR_UNSUPPORTED;
    }
    regs_checked.store(true, std::memory_order_release);
  }
  band_tc_kernel<D, kB, kW><<<grid, kBandThreads, C::kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("band kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

// D = 128 only (D = 64 runs the ring kernel of band_ring.cuh).
inline lf_status launch(const BandParams& p, int grid, cudaStream_t s) {
  if (p.rel_bias) return launch_band_tc_d<128, true, false>(p, grid, s);
  return p.varwin ? launch_band_tc_d<128, false, true>(p, grid, s) : launch_band_tc_d<128, false, false>(p, grid, s);
}

}  // namespace pairk
}  // namespace lf
