// band_duo.cuh -- bf16 band-attention kernel for D = 64 on the sm_103a tensor
// cores: two consecutive 128-row query tiles per work item, sharing the
// 96-key K/V loads that cover their windows, each tile with its own MMA
// issuer, softmax warpgroup and TMEM.
//
// Computes the sliding / dilated / look-back-only window part of Longformer
// attention (velog.io/@lainshower/Longformer, section 3-1 "Sliding Window",
// "Dilated Sliding Window"; section 4.1 for the look-back-only pattern) plus
// the global tokens' key columns ("Global Attention"), for every row except
// the rows at global tokens' positions, which the global-row pass writes (it
// may run at the same time).
//
// Dilation is handled by residue classes: with dilation delta, row
// i = r + delta*m only ever attends rows of the same residue r, and in the
// coordinate m the window is a plain band of `half` steps back and `right`
// steps ahead.  A TMA tensor map whose row stride is delta rows presents a
// residue class as a dense matrix.
//
// Work item: tiles A (rows m0 .. m0+127) and B (rows m0+128 .. m0+255) of one
// (batch, head, residue).  Their key ranges overlap in all but 128 keys, so the
// item streams the union once as "loads" of kLK = 96 keys (K and V), then the
// gathered keys of the global tokens; each load is used by one or both tiles.
// A tile's use of a load is an "entry": S = Q K^T into TMEM, softmax, then
// O += P V.
//
// CTA (one per SM, persistent), 12 warps:
//   warp 0     Q and K producer (TMA; the global tokens' rows gathered with
//              plain loads)
//   warp 1     allocates TMEM; issues tile A's tcgen05.mma products
//   warp 2     V producer (zeroes value rows no row of the item attends, so
//              that 0 * whatever they hold cannot reach an output)
//   warp 3     issues tile B's tcgen05.mma products
//   warps 4-7  softmax and epilogue of tile A, warps 8-11 of tile B: one
//              query row per thread (TMEM lane)
//
// Why two issuers: a tcgen05.mma costs its issuing warp about 40-57 cycles
// (measured), and one 96-key entry needs 4 S products (N = 96) and 6 P.V
// products (N = 64, the tensor core finishes one in about 32 cycles).  One
// warp issuing for both tiles would be slower than the tensor core; one per
// tile keeps up.  Each tile's S products go to its own two TMEM slots, which
// its own issuer reuses only after the P.V that read the previous P there
// (one thread's MMAs execute in order), so no hand-off between issuers is
// needed.
//
// The P.V product reads P from TMEM (A operand) and V straight from the TMA
// tile in shared memory as an MN-major B operand (measured as fast as a
// K-major one), so no transposition is needed.  It multiplies only the
// 16-key steps that hold keys of its own tile; pairing is used only when the
// tiles' key ranges start and end on 16-key steps of the shared loads (window
// reach a multiple of 16), so a key one tile does not attend never meets
// that tile's rows, not even with weight 0.
//
// TMEM (512 columns): S slot s of tile x at columns 96 (2x + s) (P, two bf16
// per column, over its first 48), then O of tile A and of tile B (64 each).
//
// Every wait is bounded; a timeout sets the device error word and all roles
// leave their loops, drain their in-flight copies and free TMEM.
#pragma once

#include "lf_internal.cuh"

namespace lf {
namespace duok {

// Launched at 168 registers per thread (384 x 168 = 64512 of the SM's
// 65536); the first warpgroup (producers, issuers) gives registers back
// (setmaxnreg.dec to kRegsOther) and the softmax warpgroups take them
// (setmaxnreg.inc to kRegsSoftmax): 256 x 192 + 128 x 112 = 63488 <= 64512.
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 112;
constexpr int kRegsAtLaunchMin = (256 * kRegsSoftmax + 128 * kRegsOther + kThreads - 1) / kThreads;
constexpr int kGSmem = 1024;  // global positions kept in shared memory
constexpr int kLK = 96;       // keys per K/V load (and per S product)
constexpr int kLC = kLK / 32; // 32-column chunks per S slot
constexpr int kLS = kLK / 16; // 16-key steps per load
// Lazy rescaling: a row's running maximum is raised only when a new score
// exceeds it by more than kLazy in the exp2 domain, so that O is rescaled
// rarely; P values stay below 2^kLazy.
constexpr float kLazy = 8.0f;

template <int D>
struct Cfg {
  static_assert(D == 64, "the duo kernel is built for D = 64");
  static constexpr int kSt = 5;                  // K and V ring slots
  static constexpr int kQBuf = 2;                // Q buffers (two tiles each)
  static constexpr int kTileQ = 128 * D * 2;     // bytes of a [128, D] bf16 query tile
  static constexpr int kTileKV = kLK * D * 2;    // bytes of a [96, D] bf16 key or value load
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBuf * 2 * kTileQ;
  static constexpr int kOffV = kOffK + kSt * kTileKV;
  static constexpr int kOffBar = kOffV + kSt * kTileKV;
  // q_full[2] q_empty[2] k_full[5] k_empty[5] v_full[5] v_empty[5] v_land
  // s_full[2][2] p_full[2][2] o_bar[2] fin
  static constexpr int kNumBar = 2 + 2 + 4 * kSt + 1 + 4 + 4 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kOffSeg = kOffMisc + 16;
  static constexpr int kOffPad = kOffSeg + kMaxSeg * (int)sizeof(BandSeg);
  static constexpr int kOffGidx = kOffPad + kMaxBatch * 4;
  static constexpr int kSmem = kOffGidx + kGSmem * 4 + 1024;  // + slack to align the base
  static constexpr uint32_t kColO = 4 * kLK;
  static_assert(kColO + 2 * D <= 512, "TMEM budget");
  static_assert(kTileKV % 1024 == 0, "swizzle atoms");
  static_assert(kSmem <= 232448, "shared memory");
};

template <int D>
struct Smem {
  using C = Cfg<D>;
  uint8_t* base;
  uint32_t sbase;
  __device__ __forceinline__ uint32_t q(int qb, int x) const { return sbase + C::kOffQ + (2 * qb + x) * C::kTileQ; }
  __device__ __forceinline__ uint32_t k(int s) const { return sbase + C::kOffK + s * C::kTileKV; }
  __device__ __forceinline__ uint32_t v(int s) const { return sbase + C::kOffV + s * C::kTileKV; }
  __device__ __forceinline__ uint8_t* q_ptr(int qb, int x) const { return base + C::kOffQ + (2 * qb + x) * C::kTileQ; }
  __device__ __forceinline__ uint8_t* k_ptr(int s) const { return base + C::kOffK + s * C::kTileKV; }
  __device__ __forceinline__ uint8_t* v_ptr(int s) const { return base + C::kOffV + s * C::kTileKV; }
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + C::kOffBar + 8 * i; }
  // k_empty and v_empty complete after two arrivals: the commit of each
  // tile's issuer once its products that read the buffer are done; a buffer
  // only one tile uses gets the second arrival from that tile's issuer as a
  // plain arrive (the phase still waits for its commit).  A Q buffer is free
  // again after its item's epilogues, which stage the output tiles in it:
  // q_empty takes one arrival from each of the eight softmax warps.
  __device__ __forceinline__ uint32_t q_full(int b) const { return bar(0 + b); }
  __device__ __forceinline__ uint32_t q_empty(int b) const { return bar(2 + b); }
  __device__ __forceinline__ uint32_t k_full(int s) const { return bar(4 + s); }
  __device__ __forceinline__ uint32_t k_empty(int s) const { return bar(4 + C::kSt + s); }
  __device__ __forceinline__ uint32_t v_full(int s) const { return bar(4 + 2 * C::kSt + s); }
  __device__ __forceinline__ uint32_t v_empty(int s) const { return bar(4 + 3 * C::kSt + s); }
  __device__ __forceinline__ uint32_t v_land() const { return bar(4 + 4 * C::kSt); }
  __device__ __forceinline__ uint32_t s_full(int x, int s) const { return bar(5 + 4 * C::kSt + 2 * x + s); }
  __device__ __forceinline__ uint32_t p_full(int x, int s) const { return bar(9 + 4 * C::kSt + 2 * x + s); }
  // Completion of the last P.V of tile x in an item arrives on o_bar(x):
  // one phase per item of the tile, waited for once by its epilogue (the
  // next phase needs that softmax's P of the next item).
  __device__ __forceinline__ uint32_t o_bar(int x) const { return bar(13 + 4 * C::kSt + x); }
  __device__ __forceinline__ uint32_t fin() const { return bar(15 + 4 * C::kSt); }
  __device__ __forceinline__ uint32_t* tmem_holder() const { return reinterpret_cast<uint32_t*>(base + C::kOffMisc); }
  __device__ __forceinline__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + C::kOffMisc + 4); }
  __device__ __forceinline__ BandSeg* segs() const { return reinterpret_cast<BandSeg*>(base + C::kOffSeg); }
  __device__ __forceinline__ int32_t* pad() const { return reinterpret_cast<int32_t*>(base + C::kOffPad); }
  __device__ __forceinline__ int32_t* gidx() const { return reinterpret_cast<int32_t*>(base + C::kOffGidx); }
};

// The launch's lookup tables in shared memory (a data-dependent read of the
// kernel parameters would miss the constant cache).
struct Tables {
  const BandSeg* seg;
  const int32_t* pad;   // [B] trailing padding of each batch row
  const int32_t* gidx;  // [min(G, kGSmem)] global positions
};

__device__ __forceinline__ int gidx_at(const BandParams& p, const Tables& tb, int i) {
  return i < kGSmem ? tb.gidx[i] : p.gidx[i];
}

// number of global positions <= lim (gidx is strictly increasing)
__device__ __forceinline__ int upper_bound_gidx(const BandParams& p, const Tables& tb, int lim) {
  int lo = 0, hi = p.G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (gidx_at(p, tb, mid) <= lim) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ------------------------------------------------------------------ work items
// Fields come in pairs, one per tile (x = 0: A, x = 1: B), read through the
// accessors: the roles index them with a run-time tile number, and an array
// indexed that way would live in local memory.
struct Item {
  int r, delta, n_r, set, bh, Lb, Lm, m0;
  int nt;                  // tiles whose rows exist (1, or 2 when pairing)
  int act;                 // bit x: tile x has a valid row
  int klo0, klo1, khi0, khi1;  // keys (m coordinate) any valid row of tile x attends
  int gcnt0, gcnt1;        // global tokens visible to tile x (a prefix of the sorted list)
  int ng0, ng1;            // ... and the loads that hold them
  int U0, nb;              // band load L holds keys [U0 + kLK L, U0 + kLK L + kLK - 1], L < nb
  int lb1_0, lb0_1, lb1_1; // band loads tile A uses: [0, lb1_0]; tile B: [lb0_1, lb1_1]
  int gshare;              // both tiles use the same global loads
  int nload;               // band loads, then global loads
  int last0, last1;        // the last load tile A / B uses
  __device__ __forceinline__ int klo(int x) const { return x ? klo1 : klo0; }
  __device__ __forceinline__ int khi(int x) const { return x ? khi1 : khi0; }
};

struct Load {
  int glob;   // 0: band load, 1: global tokens' rows
  int base;   // first key (band) or first global token (global)
  int cnt;    // keys held
  int users;  // bit x: tile x uses it
};

// Every role decodes each item once, the same way.
__device__ __forceinline__ Item decode_item(const BandParams& p, const Tables& tb, int item) {
  Item it;
  const int b = item / p.items_per_b;
  const int rem = item - b * p.items_per_b;
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.seg[mid].begin <= rem) lo = mid; else hi = mid - 1;
  }
  const BandSeg sg = tb.seg[lo];
  it.r = sg.r;
  it.delta = sg.delta;
  it.n_r = sg.n_r;
  it.set = sg.set;
  it.m0 = (rem - sg.begin) * (p.pair ? 256 : 128);
  it.bh = b * p.H + sg.h;
  it.Lb = p.n - tb.pad[b];
  const int Lm = (it.Lb > it.r) ? (it.Lb - it.r + it.delta - 1) / it.delta : 0;
  it.Lm = min(Lm, it.n_r);
  it.nt = (p.pair && it.m0 + 128 < it.n_r) ? 2 : 1;
  it.act = 0;
  int klo[2], khi[2], gcnt[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    klo[x] = 0;
    khi[x] = -1;
    gcnt[x] = 0;
    const int mx = it.m0 + 128 * x;
    if (x >= it.nt || mx >= it.Lm) continue;
    it.act |= 1 << x;
    const int qlast = min(mx + 127, it.Lm - 1);
    klo[x] = max(0, mx - p.half);
    khi[x] = min(it.Lm - 1, qlast + p.right);
    int glim = it.Lb - 1;
    if (p.causal) glim = min(glim, it.r + it.delta * qlast);
    gcnt[x] = (p.G > 0) ? upper_bound_gidx(p, tb, glim) : 0;
  }
  it.klo0 = klo[0];
  it.klo1 = klo[1];
  it.khi0 = khi[0];
  it.khi1 = khi[1];
  it.gcnt0 = gcnt[0];
  it.gcnt1 = gcnt[1];
  it.ng0 = (gcnt[0] + kLK - 1) / kLK;
  it.ng1 = (gcnt[1] + kLK - 1) / kLK;
  it.U0 = klo[0];
  it.nb = 0;
  it.lb1_0 = -1;
  it.lb0_1 = 1;
  it.lb1_1 = 0;
  it.gshare = 1;
  it.nload = 0;
  it.last0 = it.last1 = -1;
  if (!(it.act & 1)) return it;  // every row of the item is padding
  const int last = (it.act & 2) ? khi[1] : khi[0];
  it.nb = (last - it.U0) / kLK + 1;
  it.lb1_0 = (khi[0] - it.U0) / kLK;
  if (it.act & 2) {
    it.lb0_1 = (klo[1] - it.U0) / kLK;
    it.lb1_1 = (khi[1] - it.U0) / kLK;
  }
  it.gshare = !(it.act & 2) || gcnt[0] == gcnt[1];
  it.nload = it.nb + (it.gshare ? it.ng0 : it.ng0 + it.ng1);
  it.last0 = it.ng0 > 0 ? it.nb + it.ng0 - 1 : it.lb1_0;
  if (it.act & 2) it.last1 = it.ng1 > 0 ? it.nload - 1 : it.lb1_1;
  return it;
}

__device__ __forceinline__ Load load_info(const Item& it, int L) {
  Load ld;
  if (L < it.nb) {
    ld.glob = 0;
    ld.base = it.U0 + kLK * L;
    ld.cnt = kLK;
    ld.users = ((L <= it.lb1_0) ? 1 : 0) | ((L >= it.lb0_1 && L <= it.lb1_1) ? 2 : 0);
  } else {
    int j = L - it.nb, gc = it.gcnt0;
    ld.glob = 1;
    if (it.gshare) {
      ld.users = it.act & 3;
    } else if (j < it.ng0) {
      ld.users = 1;
    } else {
      j -= it.ng0;
      gc = it.gcnt1;
      ld.users = 2;
    }
    ld.base = kLK * j;
    ld.cnt = min(kLK, gc - kLK * j);
  }
  return ld;
}

// The 16-key steps of load `ld` that hold keys tile x attends: [s0, s1].
__device__ __forceinline__ void kstep_range(const Item& it, const Load& ld, int x, int& s0, int& s1) {
  if (ld.glob) {
    s0 = 0;
    s1 = (ld.cnt - 1) >> 4;
  } else {
    const int lo = max(it.klo(x), ld.base), hi = min(it.khi(x), ld.base + kLK - 1);
    s0 = (lo - ld.base) >> 4;
    s1 = (hi - ld.base) >> 4;
  }
}

// Walks the entries of one tile over this CTA's items, in order, keeping the
// ring positions of every load (used by this tile or not) and of the items.
struct TileCursor {
  Item it;
  Load ld;
  int X;          // the tile
  int item, L;    // current item and load
  uint32_t lc;    // loads filled before the current one (K/V ring position)
  uint32_t ic;    // items with loads before the current one (Q buffer)
  uint32_t seen;  // entries of this tile already passed in the current item
  bool valid;

  // From load L on, the next load this tile uses; counts the loads passed.
  __device__ __forceinline__ bool seek_load() {
    for (; L < it.nload; ++L, ++lc) {
      ld = load_info(it, L);
      if ((ld.users >> X) & 1) return true;
    }
    return false;
  }
  // From `item` on, the first item with an entry of this tile.
  __device__ __forceinline__ void seek_item(const BandParams& p, const Tables& tb) {
    for (; item < p.total_items; item += gridDim.x) {
      it = decode_item(p, tb, item);
      L = 0;
      seen = 0;
      if (it.nload == 0) continue;
      if (seek_load()) {
        valid = true;
        return;
      }
      ++ic;  // an item with loads, none of them this tile's
    }
    valid = false;
  }
  __device__ __forceinline__ void start(const BandParams& p, const Tables& tb, int x) {
    X = x;
    item = blockIdx.x;
    lc = ic = 0;
    seek_item(p, tb);
  }
  // no later load of the item is this tile's
  __device__ __forceinline__ bool last_of_item() const { return L == (X ? it.last1 : it.last0); }
  // Moves to the next entry of the tile.
  __device__ __forceinline__ void next(const BandParams& p, const Tables& tb) {
    ++seen;
    ++L;
    ++lc;
    if (seek_load()) return;
    ++ic;
    item += gridDim.x;
    seek_item(p, tb);
  }
};

// 16-byte chunk `ch` of row `row` inside a [rows, 64] bf16 tile stored with
// the 128-byte swizzle TMA uses.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
  return (uint32_t)(row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// ------------------------------------------------------------------ producers
// kIsV = false: Q and K; kIsV = true: V.  Loads go into a ring of kSt slots.
template <int D, bool kIsV>
__device__ void producer(const BandParams& p, const Smem<D>& sm, const Tables& tb, int lane) {
  using C = Cfg<D>;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  volatile int* abort = sm.abort_flag();
  uint32_t lc = 0, ic = 0, land = 0;
  int last_fill[C::kSt], last_q[C::kQBuf];
#pragma unroll
  for (int s = 0; s < C::kSt; ++s) last_fill[s] = -1;
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s) last_q[s] = -1;
  int land_pending = -1;
  bool ok = true;
  Tracer tr;  // diagnostic timeline (LF_TRACE builds only)
  if (blockIdx.x == 0 && lane == 0) tr.track = kIsV ? 4 : 3;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const Item it = decode_item(p, tb, item);
    if (it.nload == 0) continue;
    if (!kIsV) {
      const int qb = ic % C::kQBuf;
      if (!warp_wait(sm.q_empty(qb), ((ic / C::kQBuf) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(sm.q_full(qb), __popc(it.act) * C::kTileQ);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (it.act & (1 << x)) tma_load_3d(sm.q(qb, x), &p.tq[it.set], 0, it.m0 + 128 * x, it.bh, sm.q_full(qb));
      }
      last_q[qb] = (int)ic;
    }
    ++ic;
    const __nv_bfloat16* src = (kIsV ? p.v : p.k) + (size_t)it.bh * p.n * D;
    const CUtensorMap* map = kIsV ? &p.tv[it.set] : &p.tk[it.set];
    const int klast = (it.act & 2) ? it.khi1 : it.khi0;  // last key any row of the item attends
    for (int L = 0; L < it.nload; ++L) {
      const Load ld = load_info(it, L);
      const int slot = lc % C::kSt;
      const uint32_t full = kIsV ? sm.v_full(slot) : sm.k_full(slot);
      const uint32_t empty = kIsV ? sm.v_empty(slot) : sm.k_empty(slot);
      const uint32_t dst = kIsV ? sm.v(slot) : sm.k(slot);
      uint8_t* dst_ptr = kIsV ? sm.v_ptr(slot) : sm.k_ptr(slot);
      tr.ev(20);
      if (!warp_wait(empty, ((lc / C::kSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      tr.ev(21);
      if (!ld.glob) {
        // value rows past the item's last attended key but inside the tensor
        // are zeroed after the copy lands
        const int z0 = klast - ld.base + 1, z1 = min(kLK, it.n_r - ld.base);
        if (kIsV && z0 < z1) {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_land(), C::kTileKV);
            tma_load_3d(dst, map, 0, ld.base, it.bh, sm.v_land());
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
            mbar_arrive_expect_tx(full, C::kTileKV);
            tma_load_3d(dst, map, 0, ld.base, it.bh, full);
          }
          last_fill[slot] = (int)lc;
        }
      } else {
        // rows of the global tokens [base, base + cnt), zeros up to the next 16
        const int nrow = (ld.cnt + 15) & ~15;
        for (int idx = lane; idx < nrow * CH; idx += 32) {
          const int row = idx / CH, ch = idx - (idx / CH) * CH;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (row < ld.cnt)
            x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)gidx_at(p, tb, ld.base + row) * D) + ch);
          *reinterpret_cast<uint4*>(dst_ptr + sw128_offset(row, ch)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
        last_fill[slot] = -1;  // completed synchronously
      }
      ++lc;
    }
  }
  tr.done();
  // Let every TMA copy this warp issued land before the CTA can exit.
  int dummy = 0;
#pragma unroll
  for (int s = 0; s < C::kSt; ++s)
    if (last_fill[s] >= 0)
      mbar_wait(kIsV ? sm.v_full(s) : sm.k_full(s), ((uint32_t)last_fill[s] / C::kSt) & 1, &dummy, kRoleDrain,
                kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s)
    if (last_q[s] >= 0) mbar_wait(sm.q_full(s), ((uint32_t)last_q[s] / C::kQBuf) & 1, &dummy, kRoleDrain, kDrainLimitNs);
  if (land_pending >= 0) mbar_wait(sm.v_land(), (uint32_t)land_pending & 1, &dummy, kRoleDrain, kDrainLimitNs);
}

// ------------------------------------------------------------------ MMA issuer (one warp per tile)
// Two queues per tile: S products run up to two entries ahead (the tile's two
// S slots) and leave behind packed records of what each entry's P.V product
// needs; a P.V product goes once the softmax has written its P.  The warp
// polls both queues and issues whichever is ready, so that a P.V never waits
// behind an S whose K or Q load is late.  The one ordering kept: the S of
// tile entry j + 2 is issued only after the P.V of entry j, which read the P
// in the slot it overwrites (one thread's MMAs execute in order).  The
// completion of that S therefore also tells the softmax that P.V j is done
// (before a rescale of O); when the tile has no entry j + 2, a commit with no
// new product stands in.  The whole warp keeps the bookkeeping; one elected
// lane issues.
//   record bits: 0 S slot, 1-3 V ring slot, 4 v_full parity, 5 p_full parity,
//   6-8 first 16-key step, 9-11 last 16-key step, 12 first product of the
//   tile in its item, 13 last product of the tile in its item, 14 the load's
//   only user
template <int D>
__device__ void mma_issuer(const BandParams& p, const Smem<D>& sm, const Tables& tb, uint32_t tmem, int X) {
  using C = Cfg<D>;
  static_assert(C::kSt <= 8 && kLS <= 8, "record fields");
  volatile int* abort = sm.abort_flag();
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);  // V: MN-major (D contiguous)
  // descriptors of Q tile 0, K slot 0 and V slot 0; the address field counts 16 bytes
  const uint64_t qdesc0 = smem_desc_sw128(sm.q(0, 0), 16, 1024);
  const uint64_t kdesc0 = smem_desc_sw128(sm.k(0), 16, 1024);
  const uint64_t vdesc0 = smem_desc_sw128(sm.v(0), 16, 1024);
  TileCursor cs;
  cs.start(p, tb, X);
  uint32_t ns = 0, np = 0;  // S and P.V products issued by this warp
  uint32_t f0 = 0, f1 = 0;  // records of the P.V products not yet issued, oldest first
  int nf = 0;
  bool ok = true;
  Tracer tr;  // diagnostic timeline (LF_TRACE builds only)
  if (blockIdx.x == 0 && (threadIdx.x & 31) == 0) tr.track = 5 + X;
  Prof pf;    // diagnostic phase counters (LF_PROF builds only)
  uint64_t idle_since = 0;  // start of the current stretch without progress (0: none)
  uint32_t spins = 0;

  while (ok && (nf > 0 || cs.valid)) {
    bool progress = false;
    // ---- the oldest P.V, if its P and V are there
    if (nf > 0) {
      const uint32_t rec = f0;
      const uint32_t slot = rec & 1, vs = (rec >> 1) & 7;
      if (__shfl_sync(0xffffffffu, (int)(mbar_test_wait(sm.p_full(X, slot), (rec >> 5) & 1) &&
                                         mbar_test_wait(sm.v_full(vs), (rec >> 4) & 1)), 0)) {
        tc_fence_after();
        const int s0 = (rec >> 6) & 7, s1 = (rec >> 9) & 7;
        const uint32_t o = tmem + C::kColO + D * X, pt = tmem + kLK * (2 * X + slot);
        const uint64_t vd = vdesc0 + (uint64_t)((vs * C::kTileKV) >> 4);
        const uint32_t acc0 = ((rec >> 12) & 1) ? 0u : 1u;  // O starts over with the tile's first product
        if (s0 == 0 && s1 == kLS - 1) {
#pragma unroll
          for (int kk = 0; kk < kLS; ++kk)
            mma_bf16_ts_w(o, pt + 8 * kk, vd + kk * (2048 >> 4), idesc_pv, kk > 0 ? 1u : acc0);
        } else {
          for (int kk = s0; kk <= s1; ++kk)
            mma_bf16_ts_w(o, pt + 8 * kk, vd + kk * (2048 >> 4), idesc_pv, kk > s0 ? 1u : acc0);
        }
        if ((rec >> 13) & 1) mma_commit_w(sm.o_bar(X));
        mma_commit_w(sm.v_empty(vs));
        if (((rec >> 14) & 1) && elect_one()) mbar_arrive(sm.v_empty(vs));
        if (!cs.valid) mma_commit_w(sm.s_full(X, slot));  // no entry np + 2: stands in for its S
        f0 = f1;
        --nf;
        ++np;
        tr.ev(3);
        progress = true;
      }
    }
    // ---- the next S, if its slot's previous P.V is issued and its K (and Q) are there
    if (cs.valid && ns < np + 2) {
      const uint32_t ks = cs.lc % C::kSt;
      const uint32_t qb = cs.ic % C::kQBuf;
      if (__shfl_sync(0xffffffffu, (int)(mbar_test_wait(sm.k_full(ks), (cs.lc / C::kSt) & 1) &&
                                         (cs.seen != 0 || mbar_test_wait(sm.q_full(qb), (cs.ic / C::kQBuf) & 1))), 0)) {
        tc_fence_after();
        const uint32_t slot = ns & 1;
        const uint32_t d = tmem + kLK * (2 * X + slot);
        const uint32_t idesc = idesc_bf16_f32(128, cs.ld.glob ? (cs.ld.cnt + 15) & ~15 : kLK, 0);
        const uint64_t qd = qdesc0 + (uint64_t)(((2 * qb + X) * C::kTileQ) >> 4);
        const uint64_t kd = kdesc0 + (uint64_t)((ks * C::kTileKV) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_bf16_ss_w(d, qd + 2 * kk, kd + 2 * kk, idesc, kk > 0);
        mma_commit_w(sm.s_full(X, slot));
        const bool only = cs.ld.users != 3;
        mma_commit_w(sm.k_empty(ks));
        if (only && elect_one()) mbar_arrive(sm.k_empty(ks));
        int s0, s1;
        kstep_range(cs.it, cs.ld, X, s0, s1);
        const bool last = cs.last_of_item();
        const uint32_t rec = slot | (ks << 1) | (((cs.lc / C::kSt) & 1) << 4) | (((ns >> 1) & 1) << 5) |
                             ((uint32_t)s0 << 6) | ((uint32_t)s1 << 9) | ((uint32_t)(cs.seen == 0) << 12) |
                             ((uint32_t)last << 13) | ((uint32_t)only << 14);
        if (nf == 0) f0 = rec; else f1 = rec;
        ++nf;
        ++ns;
        cs.next(p, tb);
        if (!cs.valid) {
          // the stream of S products ended: P.V products already issued that
          // have no entry two on get their stand-in commits now
          for (uint32_t j = (ns >= 2 ? ns - 2 : 0); j < np; ++j) mma_commit_w(sm.s_full(X, j & 1));
        }
        tr.ev(1);
        progress = true;
      }
    }
    if (progress) {
      spins = 0;
      idle_since = 0;
      continue;
    }
    // Nothing to issue: sleep in the barrier this warp most likely needs
    // next (the oldest P.V's P, else the next S's K), so that the softmax
    // warps sharing this warp's sub-partition keep its issue slots.  The
    // wake-up is the phase completing or the time hint running out.
    // (both queues may be waiting: short sleeps, alternating between them)
    const bool s_wait = cs.valid && ns < np + 2;
    if (nf > 0 && (!s_wait || (spins & 1) == 0)) {
      const uint32_t rec = f0;
      mbar_try_wait(sm.p_full(X, rec & 1), (rec >> 5) & 1, 128);
    } else if (s_wait) {
      mbar_try_wait(sm.k_full(cs.lc % C::kSt), (cs.lc / C::kSt) & 1, 128);
    }
    __syncwarp();
    // bounded: the wait limit without progress is a timeout
    if (++spins >= 16) {
      spins = 0;
      // lane 0 decides for the warp, which must stay converged
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
      // (SM cycles at two per ns, as in mbar_wait)
      const uint64_t now = __shfl_sync(0xffffffffu, (unsigned long long)clock64(), 0);
      if (idle_since == 0) {
        idle_since = now;
      } else if (now - idle_since > 2 * *cta_wait_limit(abort)) {
        if ((threadIdx.x & 31) == 0) atomicCAS(&g_device_error, 0u, (uint32_t)LF_ERR_TIMEOUT | ((uint32_t)kRoleMma << 8));
        *abort = 1;
        break;
      }
    }
  }
  tr.done();
  pf.flush(2 + X, (threadIdx.x & 31) == 0);
  // Every MMA this warp issued must finish before TMEM is freed.
  mma_commit_w(sm.fin());
  __syncwarp();
  int dummy = 0;
  mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, kDrainLimitNs);
  __syncwarp();
}

// ------------------------------------------------------------------ softmax / epilogue
// Bits [lo, hi] of a 32-bit word (empty when hi < lo); lo, hi may lie outside [0, 31].
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  const uint32_t from = lo <= 0 ? 0xffffffffu : (lo >= 32 ? 0u : (0xffffffffu << lo));
  const uint32_t upto = hi >= 31 ? 0xffffffffu : (hi < 0 ? 0u : (0xffffffffu >> (31 - hi)));
  return from & upto;
}

// m coordinate of position g in residue class r, or a value that is never
// inside a band when g is not in the class
__device__ __forceinline__ int residue_coord(int g, int r, int delta) {
  if (delta == 1) return g;
  const int d = g - r;
  return (d >= 0 && d % delta == 0) ? d / delta : -(1 << 29);
}

// Columns of a 32-column chunk whose keep bit is clear become -inf.
__device__ __forceinline__ void mask32(uint32_t* x, uint32_t keep) {
  const uint32_t kNegInf = 0xff800000u;
#pragma unroll
  for (int t = 0; t < 32; ++t) x[t] = ((keep >> t) & 1u) ? x[t] : kNegInf;
}

// Maximum of 32 raw scores (two independent max3 chains).
__device__ __forceinline__ float max32(const uint32_t* x) {
#define LF_V(i) __uint_as_float(x[i])
  float a = max3f(LF_V(0), LF_V(1), LF_V(2)), b = max3f(LF_V(3), LF_V(4), LF_V(5));
#pragma unroll
  for (int t = 6; t < 30; t += 4) {
    a = max3f(a, LF_V(t), LF_V(t + 1));
    b = max3f(b, LF_V(t + 2), LF_V(t + 3));
  }
  a = max3f(a, LF_V(30), LF_V(31));
#undef LF_V
  return fmaxf(a, b);
}

// P for 32 columns: p = exp2(s * sl2 - m), packed to bf16 pairs (pk[t] holds
// columns 2t, 2t + 1); returns the sum of the p values.  Masked columns hold
// -inf and give p = 0.
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

// Per-row running state of the online softmax.
struct RowState {
  float m_run, l_run;
};

// P of the chunks in cm (bits 0-2: computed; bits 4-6: written as zeros)
// from the scores in x against reference m; returns the sum of the p values,
// and in pmax the largest bf16 P bit pattern (P >= 0, so the bit patterns
// order like the values).
__device__ __forceinline__ float p_chunks(uint32_t tS, uint32_t cm, int mode, const uint32_t* x, float sl2, float m,
                                          uint32_t& pmax) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float mneg = (m == NEG_INF) ? 0.f : -m;
  uint32_t pk[16];
  float l = 0.f;
  uint32_t mp = 0u;
#pragma unroll
  for (int c = 0; c < kLC; ++c) {
    if (mode != 0 && ((cm >> c) & 1)) {
      l += exp32(x + 32 * c, sl2, mneg, pk);
      tmem_st16_nw(tS + 16 * c, pk);  // P chunk c over columns [16c, 16c + 16) (already read)
#pragma unroll
      for (int t = 0; t < 16; ++t) mp = max_u16x2(mp, pk[t]);
    } else if ((cm >> (4 + c)) & 1) {
#pragma unroll
      for (int t = 0; t < 16; ++t) pk[t] = 0u;
      tmem_st16_nw(tS + 16 * c, pk);
    }
  }
  pmax = max(mp & 0xffffu, mp >> 16);
  return l;
}

// One entry: the 32-column chunks c with bit c of cm set (the same bits in
// every lane of the warp) are read from TMEM and masked (mode 2); chunks
// with bit 4 + c set, which no row of the warp attends, get P = 0 without
// being read.  P (bf16) goes over the slot's columns [16c, 16c + 16).
// While every row of the warp has a reference maximum from earlier entries,
// P is computed against it at once and the entry's own maximum only checks
// it afterwards: P is recomputed, against a raised maximum, only if some
// score exceeds the reference by more than kLazy (so P <= 2^kLazy always).
// Returns the factor O must be scaled by (1 = none).
__device__ __forceinline__ float softmax_entry(uint32_t tS, uint32_t cm, int mode, const uint32_t (&keep)[kLC],
                                               float sl2, RowState& st, bool row_valid, Tracer& tr) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  uint32_t x[kLK];
  if (mode != 0) {
#pragma unroll
    for (int c = 0; c < kLC; ++c)
      if ((cm >> c) & 1) tmem_ld32_nw(tS + 32 * c, x + 32 * c);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < kLC; ++c) reg_fence32(x + 32 * c);
    tr.ev(15);
    if (mode == 2) {
#pragma unroll
      for (int c = 0; c < kLC; ++c)
        if ((cm >> c) & 1) mask32(x + 32 * c, keep[c]);
    }
  }
  // a row whose reference is still -inf (no score yet) needs its maximum first
  const bool need = mode != 0 && row_valid && st.m_run == NEG_INF;
  float alpha = 1.f, l;
  uint32_t pmax;
  // the entry's own maximum of the scaled scores
  auto row_max = [&]() -> float {
    float mx = NEG_INF;
    if (mode != 0) {
#pragma unroll
      for (int c = 0; c < kLC; ++c)
        if ((cm >> c) & 1) mx = fmaxf(mx, max32(x + 32 * c));
    }
    return mx * sl2;  // the scale is positive
  };
  if (__any_sync(0xffffffffu, need)) {
    const float mt = row_max();
    if (mt > st.m_run + kLazy) {
      alpha = ex2_approx(st.m_run - mt);  // 0 while m_run is -inf
      st.m_run = mt;
    }
    tr.ev(16);
    l = p_chunks(tS, cm, mode, x, sl2, st.m_run, pmax);
  } else {
    tr.ev(16);
    l = p_chunks(tS, cm, mode, x, sl2, st.m_run, pmax);
    // P above 2^kLazy (bf16 0x4380 is 256) means a score beyond the lazy bound
    const bool over = pmax > 0x4380u;
    if (__any_sync(0xffffffffu, over)) {
      // rare: raise the maximum and write P again over the first version
      const float mt = row_max();
      if (mt > st.m_run + kLazy) {
        alpha = ex2_approx(st.m_run - mt);
        st.m_run = mt;
      }
      l = p_chunks(tS, cm, mode, x, sl2, st.m_run, pmax);
    }
  }
  st.l_run = st.l_run * alpha + l;
  tr.ev(17);
  return alpha;
}

template <int D>
__device__ void softmax_wg(const BandParams& p, const Smem<D>& sm, const Tables& tb, uint32_t tmem, int X,
                           int wq, int lane) {
  using C = Cfg<D>;
  volatile int* abort = sm.abort_flag();
  const int row = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tO = tmem + lane_base + C::kColO + D * X;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float sl2 = p.sl2;
  uint32_t jx = 0;     // entries of this tile passed (S slot j & 1, phase j >> 1)
  uint32_t nitem = 0;  // items in which this tile had entries (o_bar phase)
  uint32_t nq = 0;     // items with loads passed (Q buffer)
  bool ok = true;
  Tracer tr;  // diagnostic timeline (LF_TRACE builds only)
  if (blockIdx.x == 0 && wq == 0 && lane == 0) tr.track = 1 + X;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const Item it = decode_item(p, tb, item);
    const uint32_t qb = nq % C::kQBuf;  // the item's Q buffer, if it has loads
    if (it.nload > 0) ++nq;
    if (X >= it.nt) continue;  // no such tile in this item
    const int m_q = it.m0 + 128 * X + row;
    const int i_q = it.r + it.delta * m_q;
    // rows at the positions of global tokens are written by the global-row
    // pass, which may run at the same time: this kernel leaves them alone
    bool write_row = m_q < it.n_r;
    if (p.G > 0 && write_row) {
      const int mt0 = it.m0 + 128 * X;
      const int i_lo = it.r + it.delta * mt0;
      const int i_hi = it.r + it.delta * min(mt0 + 127, it.n_r - 1);
      if (upper_bound_gidx(p, tb, i_hi) > upper_bound_gidx(p, tb, i_lo - 1) &&
          upper_bound_gidx(p, tb, i_q) > upper_bound_gidx(p, tb, i_q - 1))
        write_row = false;
    }
    const bool row_valid = m_q < it.Lm;
    uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + (size_t)i_q) * D);
    if (!(it.act & (1 << X))) {
      if (write_row) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
      }
      continue;  // (tile A's warps release the Q buffer for this tile too)
    }
    RowState st;
    st.m_run = NEG_INF;
    st.l_run = 0.f;
    int nmine = 0;
    // the rows of this warp: [mw, mw_last]
    const int mw = it.m0 + 128 * X + 32 * wq;
    const int mw_last = min(mw + 31, it.Lm - 1);
    const int clo_row = m_q - p.half, chi_row = row_valid ? min(m_q + p.right, it.Lm - 1) : m_q - p.half - 1;

    for (int L = 0; ok && L < it.nload; ++L) {
      const Load ld = load_info(it, L);
      if (!((ld.users >> X) & 1)) continue;
      tr.ev(9);
      // ---- keep[c]: bit t set where this row attends column 32c + t
      // mode 0: no row of the warp attends a column of the entry; 1: every
      // row attends every column; 2: masked
      uint32_t keep[kLC];
#pragma unroll
      for (int c = 0; c < kLC; ++c) keep[c] = ~0u;
      int mode;
      uint32_t ncm;  // chunks the P.V reads
      uint32_t cm;   // chunks to compute
      if (!ld.glob) {
        ncm = (1u << kLC) - 1u;
        const int kb = ld.base;
        const bool all = (mw + 31 < it.Lm) && kb >= mw + 31 - p.half && kb + kLK - 1 <= min(mw + p.right, it.Lm - 1);
        const int u0 = mw - p.half - kb, u1 = min(mw_last + p.right, it.Lm - 1) - kb;  // the warp's keys, relative
        cm = 0;
        if (mw < it.Lm) {
#pragma unroll
          for (int c = 0; c < kLC; ++c)
            if (u0 <= 32 * c + 31 && u1 >= 32 * c) cm |= 1u << c;
        }
        mode = all ? 1 : (cm ? 2 : 0);
        if (mode == 2) {
#pragma unroll
          for (int c = 0; c < kLC; ++c) keep[c] = bit_range(clo_row - kb - 32 * c, min(chi_row - kb, kLK - 1) - 32 * c);
        }
      } else {
        const int nc = (ld.cnt + 31) >> 5;
        ncm = (1u << nc) - 1u;
        // tokens [base, base + cnt): every one is visible to every valid row
        // unless one lies within reach of the warp's windows (counted in the
        // band, or after a row when causal)
        const int g_first = gidx_at(p, tb, ld.base), g_last = gidx_at(p, tb, ld.base + ld.cnt - 1);
        const int iw_lo = it.r + it.delta * (mw - p.half), iw_hi = it.r + it.delta * (mw_last + p.right);
        const int iw_first = it.r + it.delta * mw;
        const bool simple = mw + 31 < it.Lm && (g_last < iw_lo || g_first > iw_hi) &&
                            (!p.causal || g_last <= iw_first);
        if (simple) {
#pragma unroll
          for (int c = 0; c < kLC; ++c) keep[c] = bit_range(0 - 32 * c, ld.cnt - 1 - 32 * c);
        } else {
#pragma unroll
          for (int c = 0; c < kLC; ++c) {
            uint32_t k = 0;
            const int tend = max(0, min(32, ld.cnt - 32 * c));
#pragma unroll 1
            for (int t = 0; t < tend; ++t) {
              const int g = gidx_at(p, tb, ld.base + 32 * c + t);
              const int mg = residue_coord(g, it.r, it.delta);
              const bool in_band = (m_q - mg <= p.half) && (mg - m_q <= p.right) && mg < it.Lm;
              k |= (uint32_t)((!p.causal || g <= i_q) && !in_band) << t;
            }
            keep[c] = row_valid ? k : 0u;
          }
        }
        uint32_t all_bits = ~0u;
        cm = 0;
#pragma unroll
        for (int c = 0; c < kLC; ++c) {
          if (c < nc) {
            all_bits &= keep[c];
            if (__any_sync(0xffffffffu, keep[c] != 0u)) cm |= 1u << c;
          }
        }
        const bool all = __all_sync(0xffffffffu, all_bits == ~0u) && (ld.cnt & 31) == 0;
        mode = !cm ? 0 : (all ? 1 : 2);
      }
      cm &= ncm;
      if (mode == 0) cm = 0;
      cm |= (ncm & ~cm) << 4;

      const uint32_t slot = jx & 1;
      const uint32_t tS = tmem + lane_base + kLK * (2 * X + slot);
      tr.ev(10);
      if (!__all_sync(0xffffffffu, mbar_test_wait(sm.s_full(X, slot), (jx >> 1) & 1)) &&
          !warp_wait(sm.s_full(X, slot), (jx >> 1) & 1, abort, kRoleSoftmax)) {
        ok = false;
        break;
      }
      tr.ev(11);
      tc_fence_after();
      const float alpha = softmax_entry(tS, cm, mode, keep, sl2, st, row_valid, tr);
      // ---- O *= alpha before this entry's P.V adds to it; the tile's
      // previous P.V must be done: the S of this tile's next entry was issued
      // after it, so the completion of that S (in the other slot) tells
      if (nmine > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const uint32_t j2 = jx + 1;
        if (!warp_wait(sm.s_full(X, j2 & 1), (j2 >> 1) & 1, abort, kRoleSoftmax)) { ok = false; break; }
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
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(X, slot));
      tr.ev(12);
      ++jx;
      ++nmine;
    }
    if (!ok) break;

    tr.ev(13);
    // ---- epilogue: O / l -> bf16 -> global, after the tile's last P.V
    if (!warp_wait(sm.o_bar(X), nitem & 1, abort, kRoleSoftmax)) { ok = false; break; }
    ++nitem;
    tc_fence_after();
    const float inv = (row_valid && st.l_run > 0.f) ? 1.0f / st.l_run : 0.f;
    // The tile's Q tile (dead: every S of the item is done) holds this
    // warp's 32 output rows, 128-byte swizzled, so that each store below
    // writes four whole rows instead of one 16-byte piece of 32 rows.
    uint8_t* stage = sm.q_ptr(qb, X) + 32 * wq * 128;
    fence_proxy_async_smem();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32_nw(tO + 32 * c, o);
      tmem_wait_ld();
      reg_fence32(o);
      const float* of = reinterpret_cast<const float*>(o);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_valid)
          v = make_uint4(pack_bf16x2(of[8 * q4 + 0] * inv, of[8 * q4 + 1] * inv),
                         pack_bf16x2(of[8 * q4 + 2] * inv, of[8 * q4 + 3] * inv),
                         pack_bf16x2(of[8 * q4 + 4] * inv, of[8 * q4 + 5] * inv),
                         pack_bf16x2(of[8 * q4 + 6] * inv, of[8 * q4 + 7] * inv));
        const int ch = 4 * c + q4;  // 16-byte chunk of the row
        *reinterpret_cast<uint4*>(stage + lane * 128 + ((ch ^ (lane & 7)) << 4)) = v;
      }
    }
    tc_fence_before();  // the next item's first P.V overwrites O after this read
    __syncwarp();
    {
      const int ch = lane & 7;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int rr = 4 * k + (lane >> 3);  // row of the warp this lane copies
        const bool wr = __shfl_sync(0xffffffffu, (int)write_row, rr) != 0;
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((ch ^ (rr & 7)) << 4));
        if (wr) {
          const size_t ir = (size_t)it.r + (size_t)it.delta * (mw + rr);
          reinterpret_cast<uint4*>(p.out + ((size_t)it.bh * p.n + ir) * D)[ch] = v;
        }
      }
    }
    __syncwarp();
    // release the Q buffer (for both tiles when tile B has no rows here)
    if (lane == 0) mbar_arrive_cnt(sm.q_empty(qb), (X == 0 && !(it.act & 2)) ? 2u : 1u);
    tr.ev(14);
  }
  tr.done();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) band_duo_kernel(const __grid_constant__ BandParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem<D> sm;
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
      mbar_init(sm.q_empty(b), 8);  // the eight softmax warps, after their epilogues
      mbar_init(sm.o_bar(b), 1);
      for (int s = 0; s < 2; ++s) {
        mbar_init(sm.s_full(b, s), 1);
        mbar_init(sm.p_full(b, s), 4);  // the four warps of the tile's softmax warpgroup
      }
    }
    for (int s = 0; s < C::kSt; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 2);
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 2);
    }
    mbar_init(sm.v_land(), 1);
    mbar_init(sm.fin(), 2);  // both issuers
    *sm.abort_flag() = 0;
    *cta_wait_limit(sm.abort_flag()) = wait_limit_ns();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  for (int i = threadIdx.x; i < p.nseg; i += blockDim.x) sm.segs()[i] = p.seg[i];
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) sm.pad()[i] = p.pad[i];
  for (int i = threadIdx.x; i < min(p.G, kGSmem); i += blockDim.x) sm.gidx()[i] = p.gidx[i];
  if (warp == 1) {
    tmem_alloc(smem_u32(sm.tmem_holder()), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder();
  const Tables tb{sm.segs(), sm.pad(), sm.gidx()};

  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax_wg<D>(p, sm, tb, tmem, (warp >> 2) - 1, warp & 3, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == 0) {
      producer<D, false>(p, sm, tb, lane);
    } else if (warp == 2) {
      producer<D, true>(p, sm, tb, lane);
    } else {
      mma_issuer<D>(p, sm, tb, tmem, warp >> 1);  // warp 1: tile A, warp 3: tile B
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static lf_status launch_duo(const BandParams& p, int grid, cudaStream_t s) {
  using C = Cfg<D>;
  static std::atomic<uint64_t> attr_done{0};
  static std::atomic<bool> regs_checked{false};
  lf_status st = smem_attr_once((const void*)band_duo_kernel<D>, C::kSmem, attr_done, "band kernel");
  if (st != LF_OK) return st;
  if (!regs_checked.load(std::memory_order_acquire)) {
    // The register hand-over between warpgroups needs the launch allocation
    // it was planned for; with fewer registers setmaxnreg.inc could never be
    // satisfied, so refuse to launch rather than wait.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, band_duo_kernel<D>);
    if (e != cudaSuccess) {
      set_error("cudaFuncGetAttributes(band kernel): %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
    if (fa.numRegs < kRegsAtLaunchMin || fa.numRegs * kThreads > 65536) {
      set_error("band kernel built with %d registers per thread; its register split needs %d..%d", fa.numRegs,
                kRegsAtLaunchMin, 65536 / kThreads);
      return LF_ERR_UNSUPPORTED;
    }
    regs_checked.store(true, std::memory_order_release);
  }
  band_duo_kernel<D><<<grid, kThreads, C::kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("band kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

// Band launches with D = 64 (not the global-row mode).
inline lf_status launch(const BandParams& p, int grid, cudaStream_t s) { return launch_duo<64>(p, grid, s); }

}  // namespace duok
}  // namespace lf
