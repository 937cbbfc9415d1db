// band_ring.cuh -- bf16 band-attention kernel for D = 64 on the sm_103a tensor
// cores: one 128-row query tile per CTA, two CTAs per SM, S computed ahead
// into a ring of TMEM buffers.
//
// Computes the sliding / dilated / causal window part of Longformer attention
// (velog.io/@lainshower/Longformer, section 3-1 "Sliding Window", "Dilated
// Sliding Window", section 4.1 for the look-back-only pattern) plus the
// global tokens' key columns ("Global Attention"), for every row except the
// rows at global tokens' positions, which the global-row pass writes (it may
// run at the same time).  A second instantiation (kG = true) is that pass for
// many global tokens: the query rows are the global tokens, the keys every
// valid key (see BandParams::gmode).
//
// Dilation is handled by residue classes: with dilation delta, row
// i = r + delta*m only ever attends rows of the same residue r, and in the
// coordinate m the window is a plain band of half steps back and `right`
// steps ahead.  A TMA tensor map whose row stride is delta rows presents a
// residue class as a dense matrix.
//
// Work item: one 128-row query tile of one (batch, head, residue).  It streams
// the kE-key "entries" that intersect the tile's windows, then the gathered
// keys of the global tokens, and accumulates O = softmax(S) V online.
//
// Persistent CTAs (two per SM), 8 warps each:
//   warp 0     allocates TMEM; issues every tcgen05.mma (an elected lane of
//              the converged warp): per entry g, O += P V of entry g once
//              the softmax has written P, then S = Q K^T of entry g + kSBuf
//              into the buffer that P.V read
//   warp 1     Q/K producer: TMA loads of Q and of the K entries
//   warp 2     V producer: TMA loads of the V entries into a ring of four
//              slots, each freed by the completion of the P.V that reads it
//              (the global tokens' K/V rows are gathered by the producers
//              with plain loads)
//   warp 3     no role: the P.V products read V MN-major straight from its
//              slot (the instruction descriptor's transpose bit)
//   warps 4-7  softmax and epilogue: one query row per thread; S rows are read
//              from TMEM, masked, turned into P = exp2(S*scale - m) with a
//              lazily updated row maximum, and P (bf16) is written back over
//              the S buffer it came from
// Because S is computed ahead into a ring of buffers, the softmax warps do not
// wait for the tensor cores between entries, and the products of one entry
// run while the softmax works on the next.
//
// TMEM: S buffers b = 0..kSBuf-1 at kE*b (P over their first kE/2 columns,
// two bf16 per column), then O (D columns).  The MMA warp issues the S of
// entry g + kSBuf into buffer g % kSBuf after the P.V of entry g that reads it
// (one thread's MMAs execute in order).
//
// Every wait is bounded; a timeout sets the device error word and all roles
// leave their loops, drain their in-flight copies and free TMEM.
#pragma once

#include "lf_internal.cuh"

namespace lf {
namespace ringk {

// Global positions kept in shared memory (the rest, if any, are read from
// the kernel parameters).
constexpr int kGSmem = 1024;

// D = 64: two CTAs per SM (so that two softmax warps share each SM
// sub-partition and hide each other's latencies), 64-key entries, 256 TMEM
// columns each.  D = 128: one CTA per SM, 128-key entries, all 512 columns.
template <int D>
struct BandCfg {
  static constexpr bool kWide = (D == 128);  // 128-key entries, one CTA per SM
  static constexpr int kE = kWide ? 128 : 64;       // keys per entry
  static constexpr int kCtaPerSm = kWide ? 1 : 2;
  static constexpr int kQBuf = 2;                  // Q tiles (the next item's Q loads early)
  static constexpr int kKSt = (D == 64) ? 3 : 2;   // K slots
  static constexpr int kVSt = (D == 64) ? 4 : 1;   // V slots (as loaded: [keys, D]; the P.V operand)
  static constexpr int kSBuf = 3;                  // S buffers in TMEM
  static constexpr int kTileQ = 128 * D * 2;       // bytes of one [128, D] bf16 query tile
  static constexpr int kTile = kE * D * 2;         // bytes of one [kE, D] key/value tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBuf * kTileQ;
  static constexpr int kOffV = kOffK + kKSt * kTile;
  static constexpr int kOffBar = kOffV + kVSt * kTile;
  // q_full[2], q_empty[2], k_full[4], (unused)[4], v_full[4], (unused)[8],
  // pv_done[4], v_land, s_full[3], p_full[3], (unused), o_empty, fin
  static constexpr int kNumBar = 2 + 2 + 4 * 6 + 1 + 3 + 3 + 1 + 1 + 1;
  static_assert(kKSt <= 4 && kVSt <= 4 && kQBuf <= 2 && kSBuf <= 3, "barrier arrays");
  // A K slot is free once the S product that read it is done, and a V slot
  // once its P.V product is done: the S and P.V completions are those of the
  // K and V slots only while the rings are as deep as s_full and pv_done.
  static_assert(D != 64 || (kKSt == kSBuf && kVSt == 4), "K ring = S buffers, V ring = pv_done barriers");
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  // after the barriers: TMEM address and abort flag (16 bytes), the segment
  // table, the batch rows' padding and the first kGSmem global positions
  static constexpr int kOffSeg = kOffMisc + 16;
  static constexpr int kOffPad = kOffSeg + kMaxSeg * (int)sizeof(BandSeg);
  static constexpr int kOffGidx = kOffPad + kMaxBatch * 4;
  static constexpr int kSmem = kOffGidx + kGSmem * 4 + 1024;  // + slack to align the base
  static constexpr int kTmemCols = kWide ? 512 : 256;
  static constexpr uint32_t kColO = kSBuf * kE;     // S buffers at kE * b, then O (D columns)
  static_assert(kColO + D <= kTmemCols, "TMEM budget");
  static_assert(kCtaPerSm == 1 || 2 * (kSmem + 1024) <= 233472, "two CTAs per SM must fit");
};

// Everything the roles need to know about one work item.  Computed the same
// way by every role from the item number alone.
// The launch's lookup tables, copied to shared memory at kernel start (a
// data-dependent read of the kernel parameters would miss the constant cache).
struct Tables {
  const BandSeg* seg;
  const int32_t* pad;   // [B] padding of each batch row
  const int32_t* gidx;  // [min(G, kGSmem)] global positions
};

__device__ __forceinline__ int gidx_at(const BandParams& p, const Tables& tb, int i) {
  return i < kGSmem ? tb.gidx[i] : p.gidx[i];
}

struct TileItem {
  int b, h, r, delta, n_r, set, m0, Lb, Lm, bh;
  int half, right;  // the head's window reach in steps: back, ahead
  bool act;     // the tile has at least one valid row
  int U0, nU;   // band entries: keys (m coordinate) [U0 + kE*e, U0 + kE*e + kE), e < nU
  int klo, khi; // first and last key any row of the tile attends in the band
  int gcnt;     // global tokens visible to the tile (a prefix of the sorted list)
  int nE;       // entries: nU band entries, then ceil(gcnt / kE) global entries
};

__device__ __forceinline__ int upper_bound_gidx(const BandParams& p, const Tables& tb, int lim) {
  // number of global positions <= lim (gidx is strictly increasing)
  int lo = 0, hi = p.G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (gidx_at(p, tb, mid) <= lim) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Not inlined: every role calls it once per item, and one out-of-line copy
// keeps the per-entry loops small in the instruction cache.
template <int kE, bool kG>
__device__ __noinline__ TileItem decode_tile(const BandParams& p, const Tables& tb, int item) {
  const BandSeg* segs = tb.seg;
  TileItem it;
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
  it.m0 = (rem - sg.begin) * 128;
  it.bh = it.b * p.H + it.h;
  it.Lb = p.n - tb.pad[it.b];
  if (kG) {
    // query rows m: global tokens m0 .. m0 + 127 (of nrow_g); keys: [0, Lb)
    it.Lm = it.Lb;
    it.act = it.m0 < p.nrow_g && it.Lb > 0;
    it.gcnt = 0;
    if (!it.act) {
      it.nE = it.nU = 0;
      it.U0 = it.klo = it.khi = 0;
      return it;
    }
    const int qlast = min(it.m0 + 127, p.nrow_g - 1);
    it.klo = 0;
    it.khi = p.causal ? min(it.Lb - 1, gidx_at(p, tb, qlast)) : it.Lb - 1;
    it.U0 = 0;
    it.nU = it.khi / kE + 1;
    it.nE = it.nU;
    return it;
  }
  const int Lm = (it.Lb > it.r) ? (it.Lb - it.r + it.delta - 1) / it.delta : 0;
  it.Lm = min(Lm, it.n_r);
  it.act = it.m0 < it.Lm;
  if (!it.act) {
    it.nE = it.nU = it.gcnt = 0;
    it.U0 = it.klo = it.khi = 0;
    return it;
  }
  const int qlast = min(it.m0 + 127, it.Lm - 1);
  it.klo = max(0, it.m0 - it.half);
  it.khi = min(it.Lm - 1, qlast + it.right);
  it.U0 = it.klo;
  it.nU = (it.khi - it.klo) / kE + 1;
  int glim = it.Lb - 1;
  if (p.causal) glim = min(glim, it.r + it.delta * qlast);
  it.gcnt = (p.G > 0) ? upper_bound_gidx(p, tb, glim) : 0;
  it.nE = it.nU + (it.gcnt + kE - 1) / kE;
  return it;
}

// tokens held by global entry e (>= nU)
template <int kE>
__device__ __forceinline__ int global_count(const TileItem& it, int e) {
  return min(kE, it.gcnt - kE * (e - it.nU));
}

template <int D>
struct BandSmem {
  using C = BandCfg<D>;
  uint8_t* base;
  uint32_t sbase;
  __device__ __forceinline__ uint32_t q(int qb) const { return sbase + C::kOffQ + qb * C::kTileQ; }
  __device__ __forceinline__ uint32_t k(int s) const { return sbase + C::kOffK + s * C::kTile; }
  __device__ __forceinline__ uint32_t v(int s) const { return sbase + C::kOffV + s * C::kTile; }
  __device__ __forceinline__ uint8_t* k_ptr(int s) const { return base + C::kOffK + s * C::kTile; }
  __device__ __forceinline__ uint8_t* v_ptr(int s) const { return base + C::kOffV + s * C::kTile; }
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + C::kOffBar + 8 * i; }
  __device__ __forceinline__ uint32_t q_full(int b) const { return bar(0 + b); }
  __device__ __forceinline__ uint32_t q_empty(int b) const { return bar(2 + b); }
  __device__ __forceinline__ uint32_t k_full(int s) const { return bar(4 + s); }
  __device__ __forceinline__ uint32_t v_full(int s) const { return bar(12 + s); }
  __device__ __forceinline__ uint32_t v_land() const { return bar(28); }
  __device__ __forceinline__ uint32_t s_full(int b) const { return bar(29 + b); }
  __device__ __forceinline__ uint32_t p_full(int b) const { return bar(32 + b); }
  // Completion of the P.V of entry k arrives on pv_done(k & 3); it also frees
  // V slot k % 4.  The softmax waits only for the completions it needs (the
  // previous entry's before it rescales O, the last one before the epilogue);
  // the V producer waits for the one four entries back.  A waiter for entry k
  // knows that the P.V of entry k - 4 is done and that of k + 4 cannot be, so
  // the barrier is in the phase of entry k.
  __device__ __forceinline__ uint32_t pv_done(uint32_t k) const { return bar(24 + (k & 3)); }
  __device__ __forceinline__ uint32_t o_empty() const { return bar(36); }
  __device__ __forceinline__ uint32_t fin() const { return bar(37); }
  __device__ __forceinline__ uint32_t* tmem_holder() const { return reinterpret_cast<uint32_t*>(base + C::kOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + C::kOffMisc + 4); }
  __device__ __forceinline__ BandSeg* segs() const { return reinterpret_cast<BandSeg*>(base + C::kOffSeg); }
  __device__ __forceinline__ int32_t* pad() const { return reinterpret_cast<int32_t*>(base + C::kOffPad); }
  __device__ __forceinline__ int32_t* gidx() const { return reinterpret_cast<int32_t*>(base + C::kOffGidx); }
  __device__ __forceinline__ Tables tables() const { return Tables{segs(), pad(), gidx()}; }
};

// 16-byte chunk `ch` of row `row` inside a [rows, D] bf16 tile stored as D/64
// blocks of [rows, 64] with the 128-byte swizzle TMA uses.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch, int rows) {
  return (uint32_t)((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// m coordinate of global position g in residue class r, or a value that is
// never inside a band when g is not in the class
__device__ __forceinline__ int residue_coord(int g, int r, int delta) {
  if (delta == 1) return g;
  const int d = g - r;
  return (d >= 0 && d % delta == 0) ? d / delta : -(1 << 29);
}

// ------------------------------------------------------------------ producers
// kIsV = false loads Q and the K entries, kIsV = true the V entries, so that a
// full V ring (waiting for the P.V products) never holds back a K.
template <int D, bool kIsV, bool kG>
__device__ void band_producer(const BandParams& p, const BandSmem<D>& sm, int lane) {
  using C = BandCfg<D>;
  constexpr int kSt = kIsV ? C::kVSt : C::kKSt;
  volatile int* abort = sm.abort_flag();
  const Tables tb = sm.tables();
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
  Prof pf;

  // Query tiles run one item ahead: the next active item's Q is issued as
  // soon as its buffer is free (polled between the K loads of the current
  // item), so that its latency hides behind a whole item.
  int q_item = blockIdx.x;  // the next item whose Q is to be issued
  bool q_have = false;      // ... and it exists (is active)
  TileItem qt;              // its description
  auto q_seek = [&]() {
    q_have = false;
    for (; q_item < p.total_items; q_item += gridDim.x) {
      qt = decode_tile<C::kE, kG>(p, tb, q_item);
      if (qt.act) { q_have = true; return; }
    }
  };
  // Issues the pending Q if its buffer is free (waiting for that if `block`);
  // false on abort.
  auto q_issue = [&](bool block) -> bool {
    const int qb = q_it % C::kQBuf;
    const uint32_t par = ((q_it / C::kQBuf) & 1) ^ 1;
    if (block) {
      if (!warp_wait(sm.q_empty(qb), par, abort, kRoleProducer)) return false;
    } else if (!__all_sync(0xffffffffu, mbar_test_wait(sm.q_empty(qb), par))) {
      return true;
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(sm.q_full(qb), C::kTileQ);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sm.q(qb) + c * 16384, &p.tq[qt.set], c * 64, qt.m0, qt.bh, sm.q_full(qb));
    }
    last_q[qb] = (int)q_it;
    ++q_it;
    q_item += gridDim.x;
    q_seek();
    return true;
  };
  if (!kIsV) q_seek();
  uint32_t n_act = 0;  // active items started

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const TileItem it = decode_tile<C::kE, kG>(p, tb, item);
    if (!it.act) continue;
    if (!kIsV && q_it == n_act && !q_issue(true)) { ok = false; break; }  // this item's Q
    ++n_act;

    const __nv_bfloat16* src = (kIsV ? p.v : p.k) + (size_t)it.bh * p.n * D;
    const CUtensorMap* map = kIsV ? &p.tv[it.set] : &p.tk[it.set];
    constexpr int CH = D / 8;  // 16-byte chunks per row

    for (int e = 0; e < it.nE; ++e, ++kv) {
      if (!kIsV && q_it == n_act && q_have && !q_issue(false)) { ok = false; break; }  // the next item's Q
      const int slot = kv % kSt;
      const uint32_t full = kIsV ? sm.v_full(slot) : sm.k_full(slot);
      // a K slot is free when the S product of the entry kKSt back (same S buffer)
      // is done, a V slot when the P.V product of the entry kVSt back is
      const uint32_t empty = kIsV ? sm.pv_done(kv) : sm.s_full(slot);
      const uint32_t dst = kIsV ? sm.v(slot) : sm.k(slot);
      uint8_t* dst_ptr = kIsV ? sm.v_ptr(slot) : sm.k_ptr(slot);
      // A global entry is gathered row by row with plain loads; the first
      // kPre 16-byte chunks of every lane are read before the wait for the
      // slot, so that their latency hides behind it.
      constexpr int kPre = 4;
      uint4 pre[kPre];
      if (e >= it.nU) {
        const int gt = e - it.nU;
        const int cnt = global_count<C::kE>(it, e);
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
          const int idx = lane + 32 * j, row = idx / CH, ch = idx - (idx / CH) * CH;
          pre[j] = make_uint4(0, 0, 0, 0);
          if (row < cnt) pre[j] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)gidx_at(p, tb, C::kE * gt + row) * D) + ch);
        }
      }
      tr.ev(30);
      pf.lap(0);
      if (!warp_wait(empty, ((kv / kSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      tr.ev(31);
      pf.lap(1);
      if (e < it.nU) {
        const int y = it.U0 + C::kE * e;
        // value rows past the last key any row of the tile attends (padding,
        // or the end of the tile's windows) but inside the tensor are zeroed,
        // so that whatever they hold cannot reach the output through 0 * value
        const int z0 = it.khi - y + 1, z1 = min(C::kE, it.n_r - y);
        if (kIsV && z0 < z1) {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_land(), C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * C::kE * 128, map, c * 64, y, it.bh, sm.v_land());
          }
          land_pending = (int)land;
          const bool landed = warp_wait(sm.v_land(), land & 1, abort, kRoleProducer);
          ++land;
          if (!landed) { ok = false; break; }
          land_pending = -1;
          for (int idx = lane; idx < (z1 - z0) * CH; idx += 32) {
            const int row = z0 + idx / CH, ch = idx - (idx / CH) * CH;
            *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch, C::kE)) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full);
          last_fill[slot] = -1;
        } else {
          if (lane == 0) {
            mbar_arrive_expect_tx(full, C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * C::kE * 128, map, c * 64, y, it.bh, full);
          }
          last_fill[slot] = (int)kv;
        }
      } else {
        // rows of the global tokens visible to the tile, zeros after
        const int gt = e - it.nU;
        const int cnt = global_count<C::kE>(it, e);
        const int ng = (cnt + 15) & ~15;  // at least 16 rows: 32 * kPre chunks when D = 64
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
          const int idx = lane + 32 * j, row = idx / CH, ch = idx - (idx / CH) * CH;
          if (idx < ng * CH) *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch, C::kE)) = pre[j];
        }
        for (int idx = lane + 32 * kPre; idx < ng * CH; idx += 32) {
          const int row = idx / CH, ch = idx - (idx / CH) * CH;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (row < cnt) x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)gidx_at(p, tb, C::kE * gt + row) * D) + ch);
          *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch, C::kE)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
        last_fill[slot] = -1;  // completed synchronously
      }
      tr.ev(32);
      pf.lap(2);
    }
  }
  tr.done();
  pf.flush(kIsV ? 7 : 6, lane == 0);
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

// ------------------------------------------------------------------ MMA issuer (one warp)
// Walks the same sequence of entries as the softmax warps.  Two cursors: one
// for the S products, running up to kSBuf entries ahead, and one for the
// P.V products.  The whole warp runs the bookkeeping (descriptors stay in
// uniform registers); one elected lane issues.
struct EntryCursor {
  TileItem it;
  int item, e;       // current item and entry in it
  uint32_t g;        // entry number over the whole stream (selects the S buffer)
  uint32_t kv;       // first fill of the current item in the K / V rings
  uint32_t n_items;  // active items before the current one (selects the Q buffer)
  bool valid;
};

template <int kE, bool kG>
__device__ __forceinline__ void cursor_seek(const BandParams& p, const Tables& tb, EntryCursor& c) {
  // first active item at or after c.item
  while (c.item < p.total_items) {
    c.it = decode_tile<kE, kG>(p, tb, c.item);
    if (c.it.act) return;
    c.item += gridDim.x;
  }
  c.valid = false;
}

template <int kE, bool kG>
__device__ __forceinline__ void cursor_start(const BandParams& p, const Tables& tb, EntryCursor& c) {
  c.item = blockIdx.x;
  c.e = 0;
  c.g = 0;
  c.kv = 0;
  c.n_items = 0;
  c.valid = true;
  cursor_seek<kE, kG>(p, tb, c);
}

template <int kE, bool kG>
__device__ __forceinline__ void cursor_next(const BandParams& p, const Tables& tb, EntryCursor& c) {
  ++c.g;
  if (++c.e < c.it.nE) return;
  c.kv += c.it.nE;
  ++c.n_items;
  c.e = 0;
  c.item += gridDim.x;
  cursor_seek<kE, kG>(p, tb, c);
}

template <int D, bool kG>
__device__ void band_mma(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem) {
  using C = BandCfg<D>;
  constexpr uint32_t kTile16 = C::kTile >> 4;    // a K / V slot, in descriptor address units
  constexpr uint32_t kTileQ16 = C::kTileQ >> 4;  // a Q tile
  volatile int* abort = sm.abort_flag();
  const uint32_t idesc_sband = idesc_bf16_f32(128, C::kE, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);  // V as loaded: MN-major (D contiguous)
  const uint64_t qdesc0 = smem_desc_sw128(sm.q(0), 16, 1024);
  const uint64_t kdesc0 = smem_desc_sw128(sm.k(0), 16, 1024);
  const uint64_t vdesc0 = smem_desc_sw128(sm.v(0), 16, 1024);
  const uint32_t ot = tmem + C::kColO;
  const Tables tb = sm.tables();
  uint32_t o_cnt = 0;
  bool ok = true;
  Tracer tr;
  if (blockIdx.x == 0 && (threadIdx.x & 31) == 0) tr.track = 2;
  Prof pf;

  EntryCursor cs, cp;  // S cursor (ahead), P.V cursor
  cursor_start<C::kE, kG>(p, tb, cs);
  cursor_start<C::kE, kG>(p, tb, cp);

  // S of the entry under cs into buffer cs.g % kSBuf (the MMAs, issued by an
  // elected lane of the converged warp; the caller has waited for Q and K)
  auto mma_s = [&]() {
    const TileItem& it = cs.it;
    const int qb = cs.n_items % C::kQBuf;
    const uint32_t f = cs.kv + cs.e;
    const int ks = f % C::kKSt;
    const uint32_t idesc =
        (cs.e < it.nU) ? idesc_sband : idesc_bf16_f32(128, (global_count<C::kE>(it, cs.e) + 15) & ~15, 0);
    const uint64_t qd = qdesc0 + qb * kTileQ16;
    const uint64_t kd = kdesc0 + ks * kTile16;
    const uint32_t buf = cs.g % C::kSBuf;
    const uint32_t dt = tmem + C::kE * buf;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      // 16 columns of D: 32 bytes within a 64-column block of 128-byte rows
      const uint32_t qoff = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
      const uint32_t koff = ((kk >> 2) * (C::kE * 128) + (kk & 3) * 32) >> 4;
      mma_bf16_ss_w(dt, qd + qoff, kd + koff, idesc, kk > 0);
    }
    mma_commit_w(sm.s_full(buf));  // also frees K slot ks (= buf)
    if (cs.e + 1 == it.nE) mma_commit_w(sm.q_empty(qb));  // the item's last S: Q may be replaced
  };
  // waits (by the whole warp) for what the S of the entry under cs reads
  auto wait_s = [&]() -> bool {
    const int qb = cs.n_items % C::kQBuf;
    const uint32_t f = cs.kv + cs.e;
    if (cs.e == 0 && !warp_wait(sm.q_full(qb), (cs.n_items / C::kQBuf) & 1, abort, kRoleMma)) return false;
    return warp_wait(sm.k_full(f % C::kKSt), (f / C::kKSt) & 1, abort, kRoleMma);
  };
  // P.V of the entry under cp, P from buffer cp.g % kSBuf (elected lane)
  auto mma_pv = [&]() {
    const TileItem& it = cp.it;
    const uint32_t f = cp.kv + cp.e;
    const int vs = f % C::kVSt;
    const uint32_t buf = cp.g % C::kSBuf;
    const int ksteps = (cp.e < it.nU) ? C::kE / 16 : ((global_count<C::kE>(it, cp.e) + 15) >> 4);
    const uint32_t pt = tmem + C::kE * buf;  // P over the first kE/2 columns of the buffer
    const uint64_t vd = vdesc0 + vs * kTile16;
    const uint32_t acc0 = cp.e > 0 ? 1u : 0u;
    if (ksteps == C::kE / 16) {
#pragma unroll
      for (int kk = 0; kk < C::kE / 16; ++kk) {
        const uint32_t off = (kk * 16 * 128) >> 4;  // 16 value rows of 128 bytes
        mma_bf16_ts_w(ot, pt + kk * 8, vd + off, idesc_pv, kk > 0 ? 1u : acc0);
      }
    } else {
      for (int kk = 0; kk < ksteps; ++kk) {
        const uint32_t off = (kk * 16 * 128) >> 4;
        mma_bf16_ts_w(ot, pt + kk * 8, vd + off, idesc_pv, kk > 0 ? 1u : acc0);
      }
    }
    mma_commit_w(sm.pv_done(cp.g));  // also frees V slot vs
  };

  // the first kSBuf S products
  while (ok && cs.valid && cs.g < (uint32_t)C::kSBuf) {
    ok = wait_s();
    if (!ok) break;
    tc_fence_after();
    mma_s();
    cursor_next<C::kE, kG>(p, tb, cs);
  }
  // then per entry: the P.V of the entry under cp and the S of the one kSBuf
  // ahead (cs), which goes into the buffer that P.V reads (so after it).
  // Everything the pair needs is tested at once; only if something is not
  // ready yet are the bounded waits taken one by one.
  while (ok && cp.valid) {
    tr.ev(12);
    pf.lap(7);
    const bool has_s = cs.valid;
    const uint32_t fp = cp.kv + cp.e, fs = cs.kv + cs.e;
    const int qb = cs.n_items % C::kQBuf;
    // (tests are reads: the ones not needed this time are made anyway and
    // ignored, so that all five are in flight together)
    const bool r_vt = mbar_test_wait(sm.v_full(fp % C::kVSt), (fp / C::kVSt) & 1);
    const bool r_p = mbar_test_wait(sm.p_full(cp.g % C::kSBuf), (cp.g / C::kSBuf) & 1);
    const bool r_o = mbar_test_wait(sm.o_empty(), (o_cnt & 1) ^ 1);
    const bool r_k = mbar_test_wait(sm.k_full(fs % C::kKSt), (fs / C::kKSt) & 1);
    const bool r_q = mbar_test_wait(sm.q_full(qb), (cs.n_items / C::kQBuf) & 1);
    const bool ready = r_vt && r_p && (r_o || cp.e != 0) && (!has_s || (r_k && (r_q || cs.e != 0)));
    if (__all_sync(0xffffffffu, ready)) {
      tr.ev(13);
      pf.lap(5);
      tc_fence_after();
      mma_pv();
      if (has_s) mma_s();
    } else {
      // the P.V goes as soon as its own inputs are there (the epilogue of
      // an item waits for its last P.V), then the S
      ok = warp_wait(sm.v_full(fp % C::kVSt), (fp / C::kVSt) & 1, abort, kRoleMma) &&
           warp_wait(sm.p_full(cp.g % C::kSBuf), (cp.g / C::kSBuf) & 1, abort, kRoleMma);
      // O is overwritten by the first P.V of an item: the previous item's epilogue must have read it
      if (ok && cp.e == 0) ok = warp_wait(sm.o_empty(), (o_cnt & 1) ^ 1, abort, kRoleMma);
      if (!ok) break;
      tr.ev(13);
      pf.lap(5);
      tc_fence_after();
      mma_pv();
      if (has_s) {
        if (!wait_s()) { ok = false; break; }
        tc_fence_after();
        mma_s();
      }
    }
    if (cp.e == 0) ++o_cnt;
    tr.ev(14);
    pf.lap(8);
    cursor_next<C::kE, kG>(p, tb, cp);
    if (has_s) cursor_next<C::kE, kG>(p, tb, cs);
  }
  tr.done();
  pf.lap(7);
  pf.flush(4, (threadIdx.x & 31) == 0);
  // Wait until every MMA this warp issued has finished before TMEM is freed.
  if (elect_one()) mma_commit(sm.fin());
  __syncwarp();
  int dummy = 0;
  mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, kDrainLimitNs);
  __syncwarp();
}

// ------------------------------------------------------------------ softmax / epilogue
// Lazy rescaling: the running maximum of a row is raised only when a new
// score exceeds it by more than kLazy in the exp2 domain, so that O is
// rescaled rarely; P values stay below 2^kLazy.
constexpr float kLazy = 8.0f;

__device__ __forceinline__ int floor_div_i(int a, int b) {  // b > 0
  const int q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
}
__device__ __forceinline__ int ceil_div_i(int a, int b) { return -floor_div_i(-a, b); }

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
template <int kE>
__device__ __forceinline__ uint32_t global_keep(const BandParams& p, const Tables& tb, const TileItem& it,
                                                int e, int c, int m_q, bool row_valid, int half, int right) {
  const int gt = e - it.nU;
  const int tend = max(0, min(32, global_count<kE>(it, e) - 32 * c));
  const int i_q = it.r + it.delta * m_q;
  uint32_t k = 0;
#pragma unroll 1
  for (int t = 0; t < tend; ++t) {
    const int g = gidx_at(p, tb, kE * gt + 32 * c + t);
    const int mg = residue_coord(g, it.r, it.delta);
    const bool in_band = (m_q - mg <= half) && (mg - m_q <= right);
    k |= (uint32_t)((!p.causal || g <= i_q) && !in_band) << t;
  }
  return row_valid ? k : 0u;
}

// Columns of a 32-column chunk whose keep bit is clear become -inf.
__device__ __forceinline__ void mask32(uint32_t* x, uint32_t keep) {
  const uint32_t kNegInf = 0xff800000u;
#pragma unroll
  for (int t = 0; t < 32; ++t) x[t] = ((keep >> t) & 1u) ? x[t] : kNegInf;
}

// Maximum of 64 raw scores (four independent max3 chains).
__device__ __forceinline__ float max64(const uint32_t* x) {
#define LF_V(i) __uint_as_float(x[i])
  float a = max3f(LF_V(0), LF_V(1), LF_V(2)), b = max3f(LF_V(3), LF_V(4), LF_V(5)),
        c = max3f(LF_V(6), LF_V(7), LF_V(8)), d = max3f(LF_V(9), LF_V(10), LF_V(11));
#pragma unroll
  for (int t = 12; t < 60; t += 8) {
    a = max3f(a, LF_V(t), LF_V(t + 1));
    b = max3f(b, LF_V(t + 2), LF_V(t + 3));
    c = max3f(c, LF_V(t + 4), LF_V(t + 5));
    d = max3f(d, LF_V(t + 6), LF_V(t + 7));
  }
  a = max3f(a, LF_V(60), LF_V(61));
  b = max3f(b, LF_V(62), LF_V(63));
#undef LF_V
  return fmaxf(max3f(a, b, c), d);
}

// P for 32 columns of an entry: p = exp2(s * sl2 - m), packed to bf16 pairs
// (pk[t] holds columns 2t, 2t + 1); returns the sum of the p values.
// Masked columns hold -inf and give p = 0.
__device__ __forceinline__ float exp32(const uint32_t* x, float sl2, float mneg, uint32_t (&pk)[16]) {
  const float2 sc2 = make_float2(sl2, sl2), of2 = make_float2(mneg, mneg);
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const float2 y = __ffma2_rn(make_float2(__uint_as_float(x[2 * t]), __uint_as_float(x[2 * t + 1])), sc2, of2);
    const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
    if (t & 1) sb = __fadd2_rn(sb, make_float2(p0, p1));
    else sa = __fadd2_rn(sa, make_float2(p0, p1));
    pk[t] = pack_bf16x2(p0, p1);
  }
  const float2 s = __fadd2_rn(sa, sb);
  return s.x + s.y;
}

// Softmax and epilogue (one query row per thread; warp quarter wq of TMEM lanes).
// kB: the band entries' scores carry the relative position bias.  kW: heads'
// windows differ (each item's reach comes from its segment).
template <int D, bool kG, bool kB, bool kW>
__device__ void band_softmax(const BandParams& p, const BandSmem<D>& sm, uint32_t tmem, int wq, int lane) {
  using C = BandCfg<D>;
  static_assert(C::kE == 64 || C::kE == 128, "the softmax holds one entry in registers");
  constexpr int NC = C::kE / 32;  // 32-column chunks per entry
  volatile int* abort = sm.abort_flag();
  const Tables tb = sm.tables();
  const int row = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tO = tmem + lane_base + C::kColO;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float sl2 = p.sl2;
  uint32_t g = 0;
  bool ok = true;
  Tracer tr;
  if (blockIdx.x == 0 && wq == 0 && lane == 0) tr.track = 0;
  Prof pf;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const TileItem it = decode_tile<C::kE, kG>(p, sm.tables(), item);
    tr.ev(0);
    const int m_q = it.m0 + row;
    // rows at the positions of global tokens are written by the global-row
    // pass, which may run at the same time: this kernel leaves them alone
    bool write_row = kG ? m_q < p.nrow_g : m_q < it.n_r;
    const int g_pos = (kG && write_row) ? gidx_at(p, tb, m_q) : 0;  // global-row mode: the token's position
    if (p.G > 0) {
      const int i_lo = it.r + it.delta * it.m0;
      const int i_hi = it.r + it.delta * min(it.m0 + 127, it.n_r - 1);
      if (upper_bound_gidx(p, tb, i_hi) > upper_bound_gidx(p, tb, i_lo - 1) && write_row) {
        const int i_q = it.r + it.delta * m_q;
        if (upper_bound_gidx(p, tb, i_q) > upper_bound_gidx(p, tb, i_q - 1)) write_row = false;
      }
    }
    const bool row_valid = kG ? (write_row && g_pos < it.Lb) : m_q < it.Lm;
    uint4* orow = reinterpret_cast<uint4*>(
        p.out + ((size_t)it.bh * p.n + (kG ? (size_t)g_pos : it.r + (size_t)it.delta * m_q)) * D);
    if (!it.act) {
      if (write_row) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    float m_run = NEG_INF, l_run = 0.f;
    // the window reach of this item's head
    const int half = kW ? it.half : p.half, right = kW ? it.right : p.right;
    // the bias of this row's head, indexed by window step
    const float* brow = kB ? p.rel_bias + (size_t)it.h * p.rb_stride + p.rb_half : nullptr;
    // Band entries e in [e_all0, e_all1] are attended whole by every row of
    // this warp, those outside [e_any0, e_any1] by none of them (the rows'
    // windows together span keys [mw - half, min(mw_last + right, Lm - 1)]).
    int e_all0, e_all1, e_any0, e_any1;
    {
      const int mw = it.m0 + 32 * wq;  // first row of this warp
      const int mw_last = min(mw + 31, it.Lm - 1);
      const int hi_w = min(mw + right, it.Lm - 1);  // last key the warp's first row attends
      if (mw + 31 < it.Lm) {
        e_all0 = ceil_div_i(mw + 31 - half - it.U0, C::kE);
        e_all1 = floor_div_i(hi_w - (C::kE - 1) - it.U0, C::kE);
      } else {
        e_all0 = 1;
        e_all1 = 0;
      }
      if (mw < it.Lm) {
        e_any0 = ceil_div_i(mw - half - (C::kE - 1) - it.U0, C::kE);
        e_any1 = floor_div_i(min(mw_last + right, it.Lm - 1) - it.U0, C::kE);
      } else {
        e_any0 = 1;
        e_any1 = 0;
      }
    }
    pf.lap(0);

    for (int e = 0; e < it.nE; ++e, ++g) {
      // ---- keep[c]: bit t set where this row attends column 32c + t
      // mode 0: no row of the warp attends a column of the entry; 1: every
      // row attends every column; 2: masked
      uint32_t keep[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) keep[c] = ~0u;
      int mode;
      if (kG) {
        // every key in [0, Lb), up to the token itself when causal
        const int kb = C::kE * e;
        const int chi = row_valid ? (p.causal ? min(g_pos, it.Lb - 1) : it.Lb - 1) - kb : -1;
        uint32_t any_bits = 0u, all_bits = ~0u;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          keep[c] = bit_range(-kb - 32 * c, chi - 32 * c);
          any_bits |= keep[c];
          all_bits &= keep[c];
        }
        const bool any = __any_sync(0xffffffffu, any_bits != 0u);
        const bool all = __all_sync(0xffffffffu, all_bits == ~0u);
        mode = !any ? 0 : (all ? 1 : 2);
      } else if (e < it.nU) {
        mode = (e >= e_all0 && e <= e_all1) ? 1 : (e >= e_any0 && e <= e_any1) ? 2 : 0;
        if (mode == 2) {
          const int kb = it.U0 + C::kE * e;
          const int clo = m_q - half - kb;
          int chi = min(min(m_q + right, it.Lm - 1) - kb, C::kE - 1);
          if (!row_valid) chi = clo - 1;
#pragma unroll
          for (int c = 0; c < NC; ++c) keep[c] = bit_range(clo - 32 * c, chi - 32 * c);
        }
      } else {
        uint32_t any_bits = 0u, all_bits = ~0u;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          keep[c] = global_keep<C::kE>(p, tb, it, e, c, m_q, row_valid, half, right);
          any_bits |= keep[c];
          all_bits &= keep[c];
        }
        const bool any = __any_sync(0xffffffffu, any_bits != 0u);
        const bool all = __all_sync(0xffffffffu, all_bits == ~0u);
        mode = !any ? 0 : (all ? 1 : 2);
      }

      const uint32_t buf = g % C::kSBuf;
      const uint32_t tS = tmem + lane_base + C::kE * buf;  // S of this entry, then P
      tr.ev(1);
      pf.lap(1);
      if (!warp_wait(sm.s_full(buf), (g / C::kSBuf) & 1, abort, kRoleSoftmax)) { ok = false; break; }
      tr.ev(2);
      pf.lap(2);
      tc_fence_after();

      // ---- the entry's raw scores stay in registers for both passes
      uint32_t x[C::kE];
      float mx = NEG_INF;
      if (mode != 0) {
#pragma unroll
        for (int c = 0; c < NC; ++c) tmem_ld32_nw(tS + 32 * c, x + 32 * c);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < NC; ++c) reg_fence32(x + 32 * c);
        pf.lap(3);
        if (mode == 2) {
#pragma unroll
          for (int c = 0; c < NC; ++c) mask32(x + 32 * c, keep[c]);
        }
        if (kB && e < it.nU) {
          // scores -> s / sqrt(d) + bias (the exp2 scaling by log2(e) is
          // applied with the maximum); masked columns stay -inf (their
          // clamped table index is never used)
          const int t0 = it.U0 + C::kE * e - m_q;  // window step of column 0
          const int tmax = p.rb_stride - 1 - p.rb_half;
          const float scale = sl2 * (1.f / kLog2e);
#pragma unroll
          for (int c = 0; c < C::kE; ++c) {
            const int t = min(max(t0 + c, -p.rb_half), tmax);
            x[c] = __float_as_uint(fmaf(__uint_as_float(x[c]), scale, __ldg(brow + t)));
          }
        }
        mx = max64(x);  // row maximum of the raw scores (the scale is positive)
        if (NC == 4) mx = fmaxf(mx, max64(x + 64));
      }
      pf.lap(4);
      // with the bias the band entries' scores are already scaled by 1/sqrt(d)
      const bool scaled = kB && e < it.nU;
      const float mt = mx * (scaled ? kLog2e : sl2);
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_run + kLazy) {
        alpha = ex2_approx(m_run - mt);  // 0 while m_run is -inf
        m_run = mt;
        resc = true;
      }
      const bool any_resc = e > 0 && __any_sync(0xffffffffu, resc);
      pf.lap(5);
      tr.ev(3);
      // ---- P = exp2(s * scale - m) over the entry's first 32 columns
      // (bf16 pairs), aliasing the scores already read
      if (mode != 0) {
        const float mneg = (m_run == NEG_INF) ? 0.f : -m_run;
        uint32_t pk[16];
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          l += exp32(x + 32 * c, scaled ? kLog2e : sl2, mneg, pk);
          tmem_st16_nw(tS + 16 * c, pk);  // P chunk c over columns [16c, 16c + 16) (already read)
        }
        l_run = l_run * alpha + l;
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) pk[t] = 0u;
#pragma unroll
        for (int c = 0; c < NC; ++c) tmem_st16_nw(tS + 16 * c, pk);
        l_run = l_run * alpha;
      }
      pf.lap(7);
      // ---- O *= alpha before the P.V of this entry adds to it; that needs
      // every earlier P.V of the item done, and they complete in order, so
      // the previous entry's completion suffices.  (The S of this entry was
      // written after the P.V of entry g - 3.)
      if (any_resc) {
        if (!warp_wait(sm.pv_done(g - 1), ((g - 1) >> 2) & 1, abort, kRoleSoftmax)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o[16];
          tmem_ld16_nw(tO + 16 * c, o);
          tmem_wait_ld();
          reg_fence16(o);
          float2* of = reinterpret_cast<float2*>(o);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int t = 0; t < 8; ++t) of[t] = __fmul2_rn(of[t], a2);
          tmem_st16_nw(tO + 16 * c, o);
        }
      }
      pf.lap(6);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(buf));
      tr.ev(4);
      pf.lap(8);
    }
    if (!ok) break;

    // ---- epilogue: O / l -> bf16 (32 columns at a time) -> global
    tr.ev(5);
    // every P.V of the item: the last one's completion implies the others'
    if (!warp_wait(sm.pv_done(g - 1), ((g - 1) >> 2) & 1, abort, kRoleSoftmax)) { ok = false; break; }
    pf.lap(9);
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
    if (lane == 0) mbar_arrive(sm.o_empty());
    if (write_row) {
      // padded rows (inv = 0) are written as zeros; O is finite there since
      // every value row such a row could meet is finite or zeroed
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        orow[c] = row_valid ? make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3])
                            : make_uint4(0, 0, 0, 0);
    }
    tr.ev(7);
    pf.lap(10);
  }
  tr.done();
  pf.flush(wq, lane == 0);
}

constexpr int kBandThreads = 256;

template <int D, bool kG, bool kB, bool kW>
__global__ void __launch_bounds__(kBandThreads, BandCfg<D>::kCtaPerSm)
    band_tc_kernel(const __grid_constant__ BandParams p) {
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
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.pv_done(s), 1);
    }
    mbar_init(sm.v_land(), 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(sm.s_full(b), 1);
      mbar_init(sm.p_full(b), 4);  // the four softmax warps
    }
    mbar_init(sm.o_empty(), 4);
    mbar_init(sm.fin(), 1);
    *sm.abort_flag() = 0;
    *cta_wait_limit(sm.abort_flag()) = wait_limit_ns();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  for (int i = threadIdx.x; i < p.nseg; i += blockDim.x) sm.segs()[i] = p.seg[i];
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) sm.pad()[i] = p.pad[i];
  for (int i = threadIdx.x; i < min(max(p.G, p.nrow_g), kGSmem); i += blockDim.x) sm.gidx()[i] = p.gidx[i];
  if (warp == 0) {
    tmem_alloc(smem_u32(sm.tmem_holder()), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder();

  if (warp >= 4) {
    band_softmax<D, kG, kB, kW>(p, sm, tmem, warp & 3, lane);
  } else if (warp == 0) {
    band_mma<D, kG>(p, sm, tmem);
  } else if (warp == 1) {
    band_producer<D, false, kG>(p, sm, lane);
  } else if (warp == 2) {
    band_producer<D, true, kG>(p, sm, lane);
  }  // warp 3: no role (the P.V products read V as loaded)

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kG, bool kB, bool kW>
static lf_status launch_band_tc_d(const BandParams& p, int grid, cudaStream_t s) {
  using C = BandCfg<D>;
  static std::atomic<uint64_t> attr_done{0};
  lf_status st = smem_attr_once((const void*)band_tc_kernel<D, kG, kB, kW>, C::kSmem, attr_done, "band kernel");
  if (st != LF_OK) return st;
  band_tc_kernel<D, kG, kB, kW><<<grid, kBandThreads, C::kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("band kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

// D = 64 only (D = 128 runs the pair kernel of band_pair.cuh).
// Global-row mode (p.gmode) is a separate instantiation, so that the band
// path carries none of its code.
inline lf_status launch(const BandParams& p, int grid, cudaStream_t s) {
  if (p.gmode) return launch_band_tc_d<64, true, false, false>(p, grid, s);
  if (p.rel_bias) return launch_band_tc_d<64, false, true, false>(p, grid, s);
  return p.varwin ? launch_band_tc_d<64, false, false, true>(p, grid, s)
                  : launch_band_tc_d<64, false, false, false>(p, grid, s);
}

}  // namespace ringk
}  // namespace lf
