// band_bwd.cuh -- backward of the band attention (bf16 or fp32 inputs, fp32
// gradients), on the CUDA cores.
//
// The gradient of L = sum(dout * out) through each row's softmax
// (velog.io/@lainshower/Longformer, section 3-1 "Attention Pattern": the same
// attended sets as the forward): with p_t the row's softmax weights over its
// keys t, dp_t = <dout_row, v_t> and D_row = sum_t p_t dp_t,
//   ds_t = p_t (dp_t - D_row),   dq_row = scale * sum_t ds_t k_t,
//   dk_t += scale * ds_t q_row,  dv_t += p_t dout_row.
// Rows of global tokens use qg, kg, vg ("Linear Projections for Global
// Attention") and write dqg, dkg, dvg.
//
// Two kernels, both one warp per row or key, fixed summation orders and no
// atomics (bitwise reproducible):
//   row pass  per row: its log-sum-exp and D_row (one sweep over its keys
//             with an online maximum), then dq (a second sweep); the row's
//             two statistics go to a scratch array for the key pass
//   key pass  per key position j: dk_j and dv_j over the rows that attend
//             key j (the band rows whose window holds it; every row for a
//             global token), then dkg_j and dvg_j over the global rows
// In a sweep the lanes take one key (or row) each and compute its two dot
// products over d in full; the accumulations into dq, dk, dv are then done
// with the lanes split over d, reading the operand rows coalesced.
#pragma once

#include <type_traits>

#include "lf_internal.cuh"

namespace lf {
namespace bwdk {

constexpr int kWarps = 8;  // warps per CTA (one row or key each)

struct BwdParams {
  int32_t B, H, n, d;    // this launch's batch rows and heads; sequence, head size
  int32_t Htot, b0, h0;  // the launch's block within the [B, H] tensors
  int32_t half, right, causal, G;
  float scale, sl2;      // 1/sqrt(d) and that times log2(e)
  int32_t pad[kMaxBatch];
  int32_t gidx[kMaxGlobal];
  int32_t dil[kMaxHeadsSimt];
};

__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// <row[0..d), sv[0..d)> with row in global memory and sv in shared memory
// (every lane of the warp reads the same sv: a broadcast).
template <typename T, int D>
__device__ __forceinline__ float dot_row(const T* row, const float* sv, int d) {
  float acc = 0.f;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
      const uint4 x = __ldg(r4 + c8);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(w[e] << 16), sv[8 * c8 + 2 * e], acc);
        acc = fmaf(__uint_as_float(w[e] & 0xffff0000u), sv[8 * c8 + 2 * e + 1], acc);
      }
    }
  } else {
#pragma unroll 4
    for (int c = 0; c < d; ++c) acc = fmaf(__ldg(row + c), sv[c], acc);
  }
  return acc;
}

// row[0..d) into shared memory as floats (lanes split over d)
template <typename T>
__device__ __forceinline__ void row_to_smem(float* sv, const T* row, int d, int lane) {
  for (int c = lane; c < d; c += 32) sv[c] = ldf(row + c);
}

// rank of position i in the sorted global list, or -1
__device__ __forceinline__ int grank(const BwdParams& p, int i) {
  int lo = 0, hi = p.G - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int g = p.gidx[mid];
    if (g == i) return mid;
    if (g < i) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

// the position of one row (or key) of this launch
struct Pos {
  int b, h, i;       // batch row and head within the launch, position
  int64_t bh;        // (b0 + b) * Htot + h0 + h: the plane in the tensors
  int L;             // valid length of the batch row
  int delta, r, m;   // dilation, residue class and class coordinate of i
  int n_r;           // positions in the class
};

__device__ __forceinline__ Pos pos_of(const BwdParams& p, int64_t id) {
  Pos s;
  s.i = (int)(id % p.n);
  const int64_t bhl = id / p.n;
  s.h = (int)(bhl % p.H);
  s.b = (int)(bhl / p.H);
  s.bh = (int64_t)(p.b0 + s.b) * p.Htot + p.h0 + s.h;
  s.L = p.n - p.pad[s.b];
  s.delta = p.dil[s.h];
  s.r = s.i % s.delta;
  s.m = s.i / s.delta;
  s.n_r = (p.n - s.r + s.delta - 1) / s.delta;
  return s;
}

// Is key j in row i's band (same class, within the window)?
__device__ __forceinline__ bool in_band(const BwdParams& p, int i, int j, int delta) {
  const int off = j - i;
  if (off % delta != 0) return false;
  const int steps = off / delta;
  return steps >= -p.half && steps <= p.right;
}

// A sweep's list of keys for an ordinary row: band keys (class coordinates
// [lo, lo + nb)) then the global tokens not in the band.
struct RowKeys {
  int lo, nb, cnt;
};

__device__ __forceinline__ RowKeys row_keys(const BwdParams& p, const Pos& s) {
  RowKeys rk;
  rk.lo = max(0, s.m - p.half);
  int hi = min(s.m + p.right, s.n_r - 1);
  // keys must be valid positions: r + delta * m' < L
  const int mlast = s.L > s.r ? (s.L - 1 - s.r) / s.delta : -1;
  hi = min(hi, mlast);
  rk.nb = max(0, hi - rk.lo + 1);
  rk.cnt = rk.nb + p.G;
  return rk;
}

// key index of list entry t, or -1 if entry t is a global token that this
// row does not attend as a global column (padding, later than the row when
// causal, or already in the band)
__device__ __forceinline__ int row_key_at(const BwdParams& p, const Pos& s, const RowKeys& rk, int t) {
  if (t < rk.nb) return s.r + s.delta * (rk.lo + t);
  const int g = p.gidx[t - rk.nb];
  if (g >= s.L || (p.causal && g > s.i) || in_band(p, s.i, g, s.delta)) return -1;
  return g;
}

// ---------------------------------------------------------------- row pass
// One warp per row: statistics (log2-sum-exp of the scaled scores and D),
// then dq (or dqg for a global token's row).  Padding rows get zeros.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_row_kernel(BwdParams p, const T* __restrict__ q,
                                                             const T* __restrict__ k, const T* __restrict__ v,
                                                             const T* __restrict__ qg, const T* __restrict__ kg,
                                                             const T* __restrict__ vg, const T* __restrict__ dout,
                                                             float* __restrict__ dq, float* __restrict__ dqg,
                                                             float2* __restrict__ stats) {
  __shared__ float s_q[kWarps][D], s_do[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = (int64_t)blockIdx.x * kWarps + warp;
  if (id >= (int64_t)p.B * p.H * p.n) return;
  const Pos s = pos_of(p, id);
  const int d = p.d;
  const int64_t orow = s.bh * p.n + s.i;  // out / dout row
  const int gr = p.G > 0 ? grank(p, s.i) : -1;
  float* dq_row = gr >= 0 ? dqg + (s.bh * p.G + gr) * d : dq + orow * d;
  float2* st = stats + ((int64_t)s.b * p.H + s.h) * p.n + s.i;
  // a global token's q row takes part in nothing (its row scores with qg)
  if (gr >= 0)
    for (int c = lane; c < d; c += 32) dq[orow * d + c] = 0.f;
  if (s.i >= s.L) {
    for (int c = lane; c < d; c += 32) dq_row[c] = 0.f;
    if (lane == 0) *st = make_float2(-INFINITY, 0.f);
    return;
  }
  const T* qrow = gr >= 0 ? qg + (s.bh * p.G + gr) * d : q + orow * d;
  const T* ks = (gr >= 0 ? kg : k) + s.bh * p.n * d;
  const T* vs = (gr >= 0 ? vg : v) + s.bh * p.n * d;
  row_to_smem(s_q[warp], qrow, d, lane);
  row_to_smem(s_do[warp], dout + orow * d, d, lane);
  __syncwarp();

  // the row's keys: every valid key up to the row (causal) for a global
  // token's row, else the band and the global columns
  RowKeys rk;
  if (gr >= 0) {
    rk.lo = 0;
    rk.nb = p.causal ? min(s.L, s.i + 1) : s.L;
    rk.cnt = rk.nb;
  } else {
    rk = row_keys(p, s);
  }
  auto key_at = [&](int t) -> int { return gr >= 0 ? t : row_key_at(p, s, rk, t); };

  // sweep 1: running maximum mx, l = sum 2^(s - mx), a = sum 2^(s - mx) dp
  float mx = -INFINITY, l = 0.f, a = 0.f;
  for (int t = lane; t < rk.cnt; t += 32) {
    const int j = key_at(t);
    if (j < 0) continue;
    const float s2 = dot_row<T, D>(ks + (int64_t)j * d, s_q[warp], d) * p.sl2;
    const float dp = dot_row<T, D>(vs + (int64_t)j * d, s_do[warp], d);
    if (s2 > mx) {
      const float f = exp2f(mx - s2);  // 0 while mx is -inf
      l *= f;
      a *= f;
      mx = s2;
    }
    const float e = exp2f(s2 - mx);
    l += e;
    a = fmaf(e, dp, a);
  }
  float M = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f = (mx == -INFINITY) ? 0.f : exp2f(mx - M);
  l *= f;
  a *= f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, o);
    a += __shfl_xor_sync(0xffffffffu, a, o);
  }
  const float lse2 = M + log2f(l);
  const float Drow = a / l;
  if (lane == 0) *st = make_float2(lse2, Drow);

  // sweep 2: dq = scale * sum_t p_t (dp_t - D) k_t, lanes split over d
  constexpr int kC = D / 32;
  float acc[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) acc[c] = 0.f;
  for (int t0 = 0; t0 < rk.cnt; t0 += 32) {
    const int t = t0 + lane;
    const int j = t < rk.cnt ? key_at(t) : -1;
    float ds = 0.f;
    if (j >= 0) {
      const float s2 = dot_row<T, D>(ks + (int64_t)j * d, s_q[warp], d) * p.sl2;
      const float dp = dot_row<T, D>(vs + (int64_t)j * d, s_do[warp], d);
      ds = exp2f(s2 - lse2) * (dp - Drow);
    }
    const int nu = min(32, rk.cnt - t0);
    for (int u = 0; u < nu; ++u) {
      const float dsu = __shfl_sync(0xffffffffu, ds, u);
      const int ju = __shfl_sync(0xffffffffu, j, u);
      if (ju < 0) continue;
      const T* kr = ks + (int64_t)ju * d;
#pragma unroll
      for (int c = 0; c < kC; ++c)
        if (lane + 32 * c < d) acc[c] = fmaf(dsu, ldf(kr + lane + 32 * c), acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < kC; ++c)
    if (lane + 32 * c < d) dq_row[lane + 32 * c] = acc[c] * p.scale;
}

// ---------------------------------------------------------------- key pass
// One warp per key position j: dk_j, dv_j over the ordinary rows that attend
// key j, then (with global tokens) dkg_j, dvg_j over the global rows.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_key_kernel(BwdParams p, const T* __restrict__ q,
                                                             const T* __restrict__ k, const T* __restrict__ v,
                                                             const T* __restrict__ qg, const T* __restrict__ kg,
                                                             const T* __restrict__ vg, const T* __restrict__ dout,
                                                             float* __restrict__ dk, float* __restrict__ dv,
                                                             float* __restrict__ dkg, float* __restrict__ dvg,
                                                             const float2* __restrict__ stats) {
  __shared__ float s_k[kWarps][D], s_v[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = (int64_t)blockIdx.x * kWarps + warp;
  if (id >= (int64_t)p.B * p.H * p.n) return;
  const Pos s = pos_of(p, id);  // here i is the key position j
  const int d = p.d;
  const int j = s.i;
  const int64_t krow = s.bh * p.n + j;
  const float2* st = stats + ((int64_t)s.b * p.H + s.h) * p.n;
  constexpr int kC = D / 32;
  float ak[kC], av[kC];

  // ---- ordinary rows: dk_j, dv_j
#pragma unroll
  for (int c = 0; c < kC; ++c) ak[c] = av[c] = 0.f;
  if (j < s.L) {
    row_to_smem(s_k[warp], k + krow * d, d, lane);
    row_to_smem(s_v[warp], v + krow * d, d, lane);
    __syncwarp();
    // rows attending key j: every valid row (from j on when causal) for a
    // global token; else the class rows whose window holds j
    const bool jg = p.G > 0 && grank(p, j) >= 0;
    int lo, cnt;  // positions lo + t (global key) or class coordinates lo + t
    if (jg) {
      lo = p.causal ? j : 0;
      cnt = s.L - lo;
    } else {
      lo = max(0, s.m - p.right);
      int hi = min(s.m + p.half, s.n_r - 1);
      const int mlast = s.L > s.r ? (s.L - 1 - s.r) / s.delta : -1;
      hi = min(hi, mlast);
      cnt = max(0, hi - lo + 1);
    }
    for (int t0 = 0; t0 < cnt; t0 += 32) {
      const int t = t0 + lane;
      int i = -1;
      if (t < cnt) {
        i = jg ? lo + t : s.r + s.delta * (lo + t);
        if (p.G > 0 && grank(p, i) >= 0) i = -1;  // a global token's row uses kg, vg
      }
      float pr = 0.f, ds = 0.f;
      if (i >= 0) {
        const float2 sd = st[i];
        const int64_t orow = s.bh * p.n + i;
        const float s2 = dot_row<T, D>(q + orow * d, s_k[warp], d) * p.sl2;
        const float dp = dot_row<T, D>(dout + orow * d, s_v[warp], d);
        pr = exp2f(s2 - sd.x);
        ds = pr * (dp - sd.y);
      }
      const int nu = min(32, cnt - t0);
      for (int u = 0; u < nu; ++u) {
        const int iu = __shfl_sync(0xffffffffu, i, u);
        const float pu = __shfl_sync(0xffffffffu, pr, u);
        const float dsu = __shfl_sync(0xffffffffu, ds, u);
        if (iu < 0) continue;
        const int64_t orow = s.bh * p.n + iu;
        const T* qr = q + orow * d;
        const T* dr = dout + orow * d;
#pragma unroll
        for (int c = 0; c < kC; ++c) {
          if (lane + 32 * c < d) {
            av[c] = fmaf(pu, ldf(dr + lane + 32 * c), av[c]);
            ak[c] = fmaf(dsu, ldf(qr + lane + 32 * c), ak[c]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    if (lane + 32 * c < d) {
      dk[krow * d + lane + 32 * c] = ak[c] * p.scale;
      dv[krow * d + lane + 32 * c] = av[c];
    }
  }
  if (p.G == 0) return;

  // ---- global rows: dkg_j, dvg_j (the global row of g attends every valid
  // key, those up to g when causal)
#pragma unroll
  for (int c = 0; c < kC; ++c) ak[c] = av[c] = 0.f;
  if (j < s.L) {
    __syncwarp();
    row_to_smem(s_k[warp], kg + krow * d, d, lane);
    row_to_smem(s_v[warp], vg + krow * d, d, lane);
    __syncwarp();
    for (int t0 = 0; t0 < p.G; t0 += 32) {
      const int t = t0 + lane;
      int g = -1;
      if (t < p.G) {
        g = p.gidx[t];
        if (g >= s.L || (p.causal && j > g)) g = -1;
      }
      float pr = 0.f, ds = 0.f;
      if (g >= 0) {
        const float2 sd = st[g];
        const float s2 = dot_row<T, D>(qg + (s.bh * p.G + t) * d, s_k[warp], d) * p.sl2;
        const float dp = dot_row<T, D>(dout + (s.bh * p.n + g) * d, s_v[warp], d);
        pr = exp2f(s2 - sd.x);
        ds = pr * (dp - sd.y);
      }
      const int nu = min(32, p.G - t0);
      for (int u = 0; u < nu; ++u) {
        const int gu = __shfl_sync(0xffffffffu, g, u);
        const float pu = __shfl_sync(0xffffffffu, pr, u);
        const float dsu = __shfl_sync(0xffffffffu, ds, u);
        if (gu < 0) continue;
        const T* qr = qg + (s.bh * p.G + t0 + u) * d;
        const T* dr = dout + (s.bh * p.n + gu) * d;
#pragma unroll
        for (int c = 0; c < kC; ++c) {
          if (lane + 32 * c < d) {
            av[c] = fmaf(pu, ldf(dr + lane + 32 * c), av[c]);
            ak[c] = fmaf(dsu, ldf(qr + lane + 32 * c), ak[c]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    if (lane + 32 * c < d) {
      dkg[krow * d + lane + 32 * c] = ak[c] * p.scale;
      dvg[krow * d + lane + 32 * c] = av[c];
    }
  }
}

}  // namespace bwdk
}  // namespace lf
