// band_duo.cuh -- bf16 band-attention kernel on the sm_103a tensor cores:
// two consecutive 128-row query tiles per work item, sharing the 128-key
// K/V blocks that cover their windows.
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
// item streams the union once as "loads" of 128 keys (K and V), then the
// gathered keys of the global tokens; each load is used by one or both tiles,
// and every (load, tile) use is an "entry": S = Q K^T into TMEM, softmax, then
// O += P V.  Entries are ordered by load, A before B, so the tensor core
// alternates between the tiles and each softmax warpgroup works while the
// other tile's products run.
//
// CTA (one per SM, persistent), 12 warps:
//   warp 0     Q and K producer (TMA; the global tokens' rows gathered with
//              plain loads)
//   warp 1     allocates TMEM; issues every tcgen05.mma from one elected lane:
//              the S of entry g + kSBuf after the P.V of entry g, which frees
//              the S slot it reuses (one thread's MMAs execute in order)
//   warp 2     V producer (zeroes value rows no row of the item attends, so
//              that 0 * whatever they hold cannot reach an output)
//   warp 3     idle
//   warps 4-7  softmax and epilogue of tile A, warps 8-11 of tile B: one
//              query row per thread (TMEM lane)
//
// The P.V product reads P from TMEM (A operand) and V straight from the TMA
// tile in shared memory as an MN-major B operand (measured as fast as a
// K-major one), so no transposition is needed.  It multiplies only the
// 16-key steps that hold keys of its own tile; pairing is used only when the
// tiles' key ranges start and end on 16-key steps of the shared loads (window
// reach a multiple of 16), so a key one tile does not attend never meets
// that tile's rows, not even with weight 0.
//
// TMEM (512 columns): kSBuf S slots of 128 columns (P, two bf16 per column,
// over the first 64 of its slot), then O of tile A and of tile B (D columns each).
//
// Every wait is bounded; a timeout sets the device error word and all roles
// leave their loops, drain their in-flight copies and free TMEM.
#pragma once

#include "lf_internal.cuh"

namespace lf {
namespace duok {

// Launched at 168 registers per thread (384 x 168 = 64512 of the SM's
// 65536); the first warpgroup (producers, MMA) gives registers back
// (setmaxnreg.dec to kRegsOther) and the softmax warpgroups take them
// (setmaxnreg.inc to kRegsSoftmax): 256 x 208 + 128 x 80 = 63488 <= 64512.
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 80;
constexpr int kRegsAtLaunchMin = (256 * kRegsSoftmax + 128 * kRegsOther + kThreads - 1) / kThreads;
constexpr int kGSmem = 1024;  // global positions kept in shared memory
// Lazy rescaling: a row's running maximum is raised only when a new score
// exceeds it by more than kLazy in the exp2 domain, so that O is rescaled
// rarely; P values stay below 2^kLazy.
constexpr float kLazy = 8.0f;

template <int D>
struct Cfg {
  static constexpr int kSBuf = (D == 64) ? 3 : 2;  // S slots (128 TMEM columns each)
  static constexpr int kSt = (D == 64) ? 4 : 2;    // K and V ring slots
  static constexpr int kQBuf = (D == 64) ? 2 : 1;  // Q buffers (two tiles each)
  static constexpr int kTile = 128 * D * 2;        // bytes of a [128, D] bf16 tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBuf * 2 * kTile;
  static constexpr int kOffV = kOffK + kSt * kTile;
  static constexpr int kOffBar = kOffV + kSt * kTile;
  // q_full[2] q_empty[2] k_full[4] k_empty[4] v_full[4] v_empty[4] v_land
  // s_full[3] p_full[3] o_bar[2][2] fin
  static constexpr int kNumBar = 32;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kOffSeg = kOffMisc + 16;
  static constexpr int kOffPad = kOffSeg + kMaxSeg * (int)sizeof(BandSeg);
  static constexpr int kOffGidx = kOffPad + kMaxBatch * 4;
  static constexpr int kSmem = kOffGidx + kGSmem * 4 + 1024;  // + slack to align the base
  static constexpr uint32_t kColO = 128 * kSBuf;
  static_assert(kColO + 2 * D <= 512, "TMEM budget");
  static_assert(kSBuf <= 3 && kSt <= 4 && kQBuf <= 2, "barrier arrays");
  static_assert(kSmem <= 232448, "shared memory");
};

template <int D>
struct Smem {
  using C = Cfg<D>;
  uint8_t* base;
  uint32_t sbase;
  __device__ __forceinline__ uint32_t q(int qb, int x) const { return sbase + C::kOffQ + (2 * qb + x) * C::kTile; }
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
  __device__ __forceinline__ uint32_t s_full(int b) const { return bar(21 + b); }
  __device__ __forceinline__ uint32_t p_full(int b) const { return bar(24 + b); }
  // Completion of P.V number j of tile x (counted over the CTA's life)
  // arrives on o_bar(x, j & 1).  The softmax of tile x waits only when it
  // must: for its previous P.V before rescaling O, for its last two before
  // the epilogue.  A phase parity names a phase unambiguously only while the
  // barrier is within one phase of it, and two alternating barriers keep it
  // so: when the softmax handles entry e, whose S it has seen complete, every
  // P.V issued before that S -- so every P.V of entries e - 3 and older --
  // is complete, so at most the tile's last two P.V products are pending,
  // one per barrier; and none of its later P.V products can start before it
  // publishes their P.
  __device__ __forceinline__ uint32_t o_bar(int x, uint32_t j) const { return bar(27 + 2 * x + (j & 1)); }
  __device__ __forceinline__ uint32_t fin() const { return bar(31); }
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
  int U0, nb;              // band load L holds keys [U0 + 128 L, U0 + 128 L + 127], L < nb
  int lb1_0, lb0_1, lb1_1; // band loads tile A uses: [0, lb1_0]; tile B: [lb0_1, lb1_1]
  int gshare;              // both tiles use the same global loads
  int nload;               // band loads, then global loads
  __device__ __forceinline__ int klo(int x) const { return x ? klo1 : klo0; }
  __device__ __forceinline__ int khi(int x) const { return x ? khi1 : khi0; }
  __device__ __forceinline__ int gcnt(int x) const { return x ? gcnt1 : gcnt0; }
};

struct Load {
  int glob;   // 0: band load, 1: global tokens' rows
  int base;   // first key (band) or first global token (global)
  int cnt;    // keys held (128 for band loads)
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
  it.ng0 = (gcnt[0] + 127) >> 7;
  it.ng1 = (gcnt[1] + 127) >> 7;
  it.U0 = klo[0];
  it.nb = 0;
  it.lb1_0 = -1;
  it.lb0_1 = 1;
  it.lb1_1 = 0;
  it.gshare = 1;
  it.nload = 0;
  if (!(it.act & 1)) return it;  // every row of the item is padding
  const int last = (it.act & 2) ? khi[1] : khi[0];
  it.nb = (last - it.U0) / 128 + 1;
  it.lb1_0 = (khi[0] - it.U0) / 128;
  if (it.act & 2) {
    it.lb0_1 = (klo[1] - it.U0) / 128;
    it.lb1_1 = (khi[1] - it.U0) / 128;
  }
  it.gshare = !(it.act & 2) || gcnt[0] == gcnt[1];
  it.nload = it.nb + (it.gshare ? it.ng0 : it.ng0 + it.ng1);
  return it;
}

__device__ __forceinline__ Load load_info(const Item& it, int L) {
  Load ld;
  if (L < it.nb) {
    ld.glob = 0;
    ld.base = it.U0 + 128 * L;
    ld.cnt = 128;
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
    ld.base = 128 * j;
    ld.cnt = min(128, gc - 128 * j);
  }
  return ld;
}

// The 16-key steps of load `ld` that hold keys tile x attends: [s0, s1].
__device__ __forceinline__ void kstep_range(const Item& it, const Load& ld, int x, int& s0, int& s1) {
  if (ld.glob) {
    s0 = 0;
    s1 = (ld.cnt - 1) >> 4;
  } else {
    const int lo = max(it.klo(x), ld.base), hi = min(it.khi(x), ld.base + 127);
    s0 = (lo - ld.base) >> 4;
    s1 = (hi - ld.base) >> 4;
  }
}

// Walks the entries (load, tile) of this CTA's items in order.
struct Cursor {
  Item it;
  Load ld;
  int item, L, x;
  int seen0, seen1;  // entries of tile A / B already passed in the current item
  uint32_t lc;       // loads filled before the current one (ring position)
  uint32_t ec;       // entries before the current one (S slot)
  uint32_t ic;       // items with loads before the current one (Q buffer)
  bool valid;

  __device__ __forceinline__ bool seek_load() {
    for (; L < it.nload; ++L) {
      ld = load_info(it, L);
      if (ld.users) return true;
    }
    return false;
  }
  __device__ __forceinline__ void seek_item(const BandParams& p, const Tables& tb) {
    for (; item < p.total_items; item += gridDim.x) {
      it = decode_item(p, tb, item);
      L = 0;
      seen0 = seen1 = 0;
      if (it.nload > 0 && seek_load()) {
        x = (ld.users & 1) ? 0 : 1;
        valid = true;
        return;
      }
    }
    valid = false;
  }
  __device__ __forceinline__ void start(const BandParams& p, const Tables& tb) {
    item = blockIdx.x;
    lc = ec = ic = 0;
    seek_item(p, tb);
  }
  __device__ __forceinline__ bool last_user() const { return x == 1 || !(ld.users & 2); }
  __device__ __forceinline__ bool first_of_item() const { return seen0 + seen1 == 0; }
  __device__ __forceinline__ bool first_of_tile() const { return (x ? seen1 : seen0) == 0; }
  // Moves to the next entry; returns true when that leaves the item.
  __device__ __forceinline__ bool next(const BandParams& p, const Tables& tb) {
    ++ec;
    if (x) ++seen1; else ++seen0;
    if (x == 0 && (ld.users & 2)) {
      x = 1;
      return false;
    }
    ++lc;
    ++L;
    if (seek_load()) {
      x = (ld.users & 1) ? 0 : 1;
      return false;
    }
    ++ic;
    item += gridDim.x;
    seek_item(p, tb);
    return true;
  }
};

// 16-byte chunk `ch` of row `row` inside a [128, D] bf16 tile stored as D/64
// blocks of [128, 64] with the 128-byte swizzle TMA uses.
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
  return (uint32_t)((ch >> 3) * 128 * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
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

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const Item it = decode_item(p, tb, item);
    if (it.nload == 0) continue;
    if (!kIsV) {
      const int qb = ic % C::kQBuf;
      if (!warp_wait(sm.q_empty(qb), ((ic / C::kQBuf) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(sm.q_full(qb), __popc(it.act) * C::kTile);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (it.act & (1 << x))
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sm.q(qb, x) + c * 16384, &p.tq[it.set], c * 64, it.m0 + 128 * x, it.bh, sm.q_full(qb));
      }
      last_q[qb] = (int)ic;
    }
    ++ic;
    const __nv_bfloat16* src = (kIsV ? p.v : p.k) + (size_t)it.bh * p.n * D;
    const CUtensorMap* map = kIsV ? &p.tv[it.set] : &p.tk[it.set];
    const int klast = (it.act & 2) ? it.khi1 : it.khi0;  // last key any row of the item attends
    for (int L = 0; L < it.nload; ++L) {
      const Load ld = load_info(it, L);
      if (!ld.users) continue;
      const int slot = lc % C::kSt;
      const uint32_t full = kIsV ? sm.v_full(slot) : sm.k_full(slot);
      const uint32_t empty = kIsV ? sm.v_empty(slot) : sm.k_empty(slot);
      const uint32_t dst = kIsV ? sm.v(slot) : sm.k(slot);
      uint8_t* dst_ptr = kIsV ? sm.v_ptr(slot) : sm.k_ptr(slot);
      if (!warp_wait(empty, ((lc / C::kSt) & 1) ^ 1, abort, kRoleProducer)) { ok = false; break; }
      if (!ld.glob) {
        // value rows past the item's last attended key but inside the tensor
        // are zeroed after the copy lands
        const int z0 = klast - ld.base + 1, z1 = min(128, it.n_r - ld.base);
        if (kIsV && z0 < z1) {
          if (lane == 0) {
            mbar_arrive_expect_tx(sm.v_land(), C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * 16384, map, c * 64, ld.base, it.bh, sm.v_land());
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
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * 16384, map, c * 64, ld.base, it.bh, full);
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
  // Let every TMA copy this warp issued land before the CTA can exit.
  int dummy = 0;
#pragma unroll
  for (int s = 0; s < C::kSt; ++s)
    if (last_fill[s] >= 0)
      mbar_wait(kIsV ? sm.v_full(s) : sm.k_full(s), ((uint32_t)last_fill[s] / C::kSt) & 1, &dummy, kRoleDrain,
                200000000ull);
#pragma unroll
  for (int s = 0; s < C::kQBuf; ++s)
    if (last_q[s] >= 0) mbar_wait(sm.q_full(s), ((uint32_t)last_q[s] / C::kQBuf) & 1, &dummy, kRoleDrain, 200000000ull);
  if (land_pending >= 0) mbar_wait(sm.v_land(), (uint32_t)land_pending & 1, &dummy, kRoleDrain, 200000000ull);
}

// ------------------------------------------------------------------ MMA issuer (one warp)
// Two cursors over the same entry sequence: S products run kSBuf entries
// ahead of the P.V products.  The whole warp keeps the bookkeeping; one
// elected lane issues.
template <int D>
__device__ void mma_issuer(const BandParams& p, const Smem<D>& sm, const Tables& tb, uint32_t tmem) {
  using C = Cfg<D>;
  volatile int* abort = sm.abort_flag();
  const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);  // V: MN-major (D contiguous)
  Cursor cs, cp;
  cs.start(p, tb);
  cp.start(p, tb);
  uint32_t npv0 = 0, npv1 = 0;  // P.V products issued per tile (o_bar barrier and phase)
  bool ok = true;

  // S = Q K^T of the entry under cs into its S slot
  auto issue_s = [&]() -> bool {
    const int ks = cs.lc % C::kSt;
    if (!warp_wait(sm.k_full(ks), (cs.lc / C::kSt) & 1, abort, kRoleMma)) return false;
    const int qb = cs.ic % C::kQBuf;
    if (cs.first_of_item() &&
        !warp_wait(sm.q_full(qb), (cs.ic / C::kQBuf) & 1, abort, kRoleMma))
      return false;
    tc_fence_after();
    const uint32_t slot = cs.ec % C::kSBuf;
    const uint32_t d = tmem + 128 * slot;
    const uint32_t idesc = cs.ld.glob ? idesc_bf16_f32(128, (cs.ld.cnt + 15) & ~15, 0) : idesc_s;
    const uint32_t qa = sm.q(qb, cs.x), kb = sm.k(ks);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_bf16_ss_w(d, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024), idesc, kk > 0);
    }
    mma_commit_w(sm.s_full(slot));
    if (cs.last_user()) mma_commit_w(sm.k_empty(ks));
    return true;
  };

  for (int i = 0; i < C::kSBuf && cs.valid; ++i) {
    if (!issue_s()) { ok = false; break; }
    if (cs.next(p, tb)) mma_commit_w(sm.q_empty((cs.ic - 1) % C::kQBuf));
  }
  while (ok && cp.valid) {
    const uint32_t slot = cp.ec % C::kSBuf;
    const int vs = cp.lc % C::kSt;
    ok = warp_wait(sm.p_full(slot), (cp.ec / C::kSBuf) & 1, abort, kRoleMma) &&
         warp_wait(sm.v_full(vs), (cp.lc / C::kSt) & 1, abort, kRoleMma);
    if (!ok) break;
    tc_fence_after();
    {
      int s0, s1;
      kstep_range(cp.it, cp.ld, cp.x, s0, s1);
      const uint32_t o = tmem + C::kColO + D * cp.x, pt = tmem + 128 * slot, vb = sm.v(vs);
      const uint32_t first = cp.first_of_tile();  // O starts over with the tile's first product
      for (int kk = s0; kk <= s1; ++kk)
        mma_bf16_ts_w(o, pt + 8 * kk, smem_desc_sw128(vb + kk * 2048, 16384, 1024), idesc_pv,
                      (kk > s0 || !first) ? 1u : 0u);
      mma_commit_w(sm.o_bar(cp.x, cp.x ? npv1++ : npv0++));
      if (cp.last_user()) mma_commit_w(sm.v_empty(vs));
    }
    cp.next(p, tb);
    if (cs.valid) {
      if (!issue_s()) { ok = false; break; }
      if (cs.next(p, tb)) mma_commit_w(sm.q_empty((cs.ic - 1) % C::kQBuf));
    }
  }
  // Every MMA this warp issued must finish before TMEM is freed.
  mma_commit_w(sm.fin());
  __syncwarp();
  int dummy = 0;
  mbar_wait(sm.fin(), 0, &dummy, kRoleDrain, 200000000ull);
  __syncwarp();
}

// ------------------------------------------------------------------ softmax / epilogue
// Bits [lo, hi] of a 32-bit word (empty when hi < lo); lo, hi may lie outside [0, 31].
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 31);
  if (hi < lo) return 0u;
  const uint32_t upto = (hi == 31) ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
  return upto & ~((1u << lo) - 1u);
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

// One entry of nc (1..4) 32-column chunks: read S from TMEM (mode != 0),
// mask (mode 2), update the running maximum, write P (bf16) over the slot's
// first 16*nc columns, and return the factor O must be scaled by (1 = none).
__device__ __forceinline__ float softmax_entry(uint32_t tS, int nc, int mode, const uint32_t (&keep)[4], float sl2,
                                               RowState& st) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  uint32_t x[128];
  float mx = NEG_INF;
  if (mode != 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < nc) tmem_ld32_nw(tS + 32 * c, x + 32 * c);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 4; ++c) reg_fence32(x + 32 * c);
    if (mode == 2) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < nc) mask32(x + 32 * c, keep[c]);
    }
    mx = max32(x);
#pragma unroll
    for (int c = 1; c < 4; ++c)
      if (c < nc) mx = fmaxf(mx, max32(x + 32 * c));
  }
  const float mt = mx * sl2;  // the scale is positive
  float alpha = 1.f;
  if (mt > st.m_run + kLazy) {
    alpha = ex2_approx(st.m_run - mt);  // 0 while m_run is -inf
    st.m_run = mt;
  }
  uint32_t pk[16];
  if (mode != 0) {
    const float mneg = (st.m_run == NEG_INF) ? 0.f : -st.m_run;
    float l = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c < nc) {
        l += exp32(x + 32 * c, sl2, mneg, pk);
        tmem_st16_nw(tS + 16 * c, pk);  // P chunk c over columns [16c, 16c + 16) (already read)
      }
    }
    st.l_run = st.l_run * alpha + l;
  } else {
#pragma unroll
    for (int t = 0; t < 16; ++t) pk[t] = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < nc) tmem_st16_nw(tS + 16 * c, pk);
    st.l_run = st.l_run * alpha;
  }
  return alpha;
}

__device__ __forceinline__ int floor_div_i(int a, int b) {  // b > 0
  const int q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
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
  uint32_t ec = 0;   // entries of both tiles passed (S slot)
  uint32_t npv = 0;  // P.V products of this tile published (P.V j: o_bar(X, j), phase j >> 1)
  bool ok = true;

  for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
    const Item it = decode_item(p, tb, item);
    if (X >= it.nt) {
      // no such tile in this item: only count the other tile's entries
      for (int L = 0; L < it.nload; ++L) ec += __popc(load_info(it, L).users);
      continue;
    }
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
      for (int L = 0; L < it.nload; ++L) ec += __popc(load_info(it, L).users);
      continue;
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
      if (!ld.users) continue;
      if (!(ld.users & (1 << X))) {
        ++ec;  // the other tile's entry
        continue;
      }
      // entries of a load: tile A's, then tile B's
      const uint32_t after = (X == 0 && (ld.users & 2)) ? 1u : 0u;
      if (X == 1 && (ld.users & 1)) ++ec;
      // ---- keep[c]: bit t set where this row attends column 32c + t
      // mode 0: no row of the warp attends a column of the entry; 1: every
      // row attends every column; 2: masked
      uint32_t keep[4] = {~0u, ~0u, ~0u, ~0u};
      int mode, nc;
      if (!ld.glob) {
        nc = 4;
        const int kb = ld.base;
        // keys every row of the warp attends: [mw_last - half, mw + right] (clipped to Lm - 1)
        const bool all = (mw + 31 < it.Lm) && kb >= mw + 31 - p.half && kb + 127 <= min(mw + p.right, it.Lm - 1);
        const bool any = mw < it.Lm && kb + 127 >= mw - p.half && kb <= min(mw_last + p.right, it.Lm - 1);
        mode = all ? 1 : (any ? 2 : 0);
        if (mode == 2) {
#pragma unroll
          for (int c = 0; c < 4; ++c) keep[c] = bit_range(clo_row - kb - 32 * c, min(chi_row - kb, 127) - 32 * c);
        }
      } else {
        nc = (ld.cnt + 31) >> 5;
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
          for (int c = 0; c < 4; ++c) keep[c] = bit_range(0 - 32 * c, ld.cnt - 1 - 32 * c);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
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
        uint32_t any_bits = 0u, all_bits = ~0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < nc) {
            any_bits |= keep[c];
            all_bits &= (c == nc - 1 && (ld.cnt & 31)) ? (keep[c] | ~bit_range(0, (ld.cnt & 31) - 1)) : keep[c];
          }
        }
        const bool any = __any_sync(0xffffffffu, any_bits != 0u);
        const bool all = __all_sync(0xffffffffu, all_bits == ~0u) && (ld.cnt & 31) == 0;
        mode = !any ? 0 : (all ? 1 : 2);
      }

      const uint32_t slot = ec % C::kSBuf;
      const uint32_t tS = tmem + lane_base + 128 * slot;
      if (!warp_wait(sm.s_full(slot), (ec / C::kSBuf) & 1, abort, kRoleSoftmax)) { ok = false; break; }
      tc_fence_after();
      const float alpha = softmax_entry(tS, nc, mode, keep, sl2, st);
      // ---- O *= alpha before this entry's P.V adds to it; the tile's
      // previous P.V must be done (they complete in order)
      if (nmine > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!warp_wait(sm.o_bar(X, npv - 1), ((npv - 1) >> 1) & 1, abort, kRoleSoftmax)) { ok = false; break; }
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
      if (lane == 0) mbar_arrive(sm.p_full(slot));
      ec += 1 + after;
      ++nmine;
      ++npv;
    }
    if (!ok) break;

    // ---- epilogue: O / l -> bf16 -> global, after the tile's last P.V (the
    // one before it first, so that each wait finds its barrier within a phase)
    if (npv >= 2 && !warp_wait(sm.o_bar(X, npv - 2), ((npv - 2) >> 1) & 1, abort, kRoleSoftmax)) { ok = false; break; }
    if (!warp_wait(sm.o_bar(X, npv - 1), ((npv - 1) >> 1) & 1, abort, kRoleSoftmax)) { ok = false; break; }
    tc_fence_after();
    const float inv = (row_valid && st.l_run > 0.f) ? 1.0f / st.l_run : 0.f;
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
    tc_fence_before();  // the next item's first P.V overwrites O after this read
    if (write_row) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        orow[c] = row_valid ? make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3])
                            : make_uint4(0, 0, 0, 0);
    }
  }
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
      mbar_init(sm.q_empty(b), 1);
      mbar_init(sm.o_bar(b, 0), 1);
      mbar_init(sm.o_bar(b, 1), 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 1);
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 1);
    }
    mbar_init(sm.v_land(), 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(sm.s_full(b), 1);
      mbar_init(sm.p_full(b), 4);  // the four warps of one softmax warpgroup
    }
    mbar_init(sm.fin(), 1);
    *sm.abort_flag() = 0;
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
    } else if (warp == 1) {
      mma_issuer<D>(p, sm, tb, tmem);
    } else if (warp == 2) {
      producer<D, true>(p, sm, tb, lane);
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
