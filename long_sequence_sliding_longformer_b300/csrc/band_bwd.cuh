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
// Five kernels, in stream order, fixed summation orders and no atomics
// (bitwise reproducible):
//   rows_tiled   per 64 consecutive rows of one residue class, one sweep
//                over 32-key chunks of the band and of the global columns
//                staged in shared memory, with an online row maximum: the
//                rows' statistics (log2-sum-exp of the scaled scores and
//                D_row) and dq = scale (sum e dp k - D_row sum e k) / sum e
//   grows        per global token's row (one CTA, 8 warps over its keys):
//                its statistics and dqg
//   keys_tiled   per 64 consecutive keys of one residue class: dk, dv from
//                the ordinary rows whose band holds them, over 32-row chunks
//   gkeys        per global token's key (one CTA, 8 warps over the rows):
//                adds the rows that attend it as a global column
//   kgvg         per key position: dkg, dvg from the global rows
// In the tiled kernels 256 threads compute a 64 x 32 block of scores and of
// dout.v products with 4 x 2 register blocks, then accumulate the gradient
// rows from the block staged in shared memory.
#pragma once

#include <type_traits>

#include "lf_internal.cuh"

namespace lf {
namespace bwdk {

constexpr int kTR = 64;        // rows (or keys) per tile
constexpr int kKC = 32;        // keys (or rows) per chunk
constexpr int kThreads = 256;  // tiled kernels
constexpr int kWarps = 8;      // warp kernels: warps per CTA

struct BwdParams {
  int32_t B, H, n, d;    // this launch's batch rows and heads; sequence, head size
  int32_t Htot, b0, h0;  // the launch's block within the [B, H] tensors
  int32_t causal, G;
  float scale, sl2;      // 1/sqrt(d) and that times log2(e)
  int32_t tiles_b;       // tiles of 64 class positions per batch row (all heads, classes)
  int32_t head_tile_off[kMaxHeadsSimt + 1];
  int32_t pad[kMaxBatch];
  int32_t gidx[kMaxGlobal];
  int32_t dil[kMaxHeadsSimt];
  int32_t half_h[kMaxHeadsSimt];  // window reach per head in class steps: back half_h, ahead causal ? 0 : half_h
  // Relative position bias: rel_bias[(h0 + h) * rb_stride + rb_half + t] is
  // added to the scaled score of a band key at window step t (nullptr: none).
  // drb_part (nullptr: no bias gradient): per tile of the keys pass, the
  // rb_stride sums of ds by window step.
  const float* rel_bias;
  int32_t rb_stride, rb_half;
  float* drb_part;
};

// Largest window whose bias gradient the keys pass accumulates in shared memory.
constexpr int kMaxBiasW = 4096;

__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

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

// Is key j in row i's band (same class, within head h's window)?
__device__ __forceinline__ bool in_band(const BwdParams& p, int h, int i, int j, int delta) {
  const int off = j - i;
  if (off % delta != 0) return false;
  const int steps = off / delta;
  return steps >= -p.half_h[h] && steps <= (p.causal ? 0 : p.half_h[h]);
}

// One tile of a tiled kernel: batch row, head, residue class and the class
// coordinates [m0, m0 + 64) it covers.
struct Tile {
  int b, h, delta, r, n_r, m0, L;
  int half, right;  // the head's window reach in class steps (back, ahead)
  int64_t bh;  // the (b, h) plane in the tensors
  int mlast;   // last class coordinate whose position is valid (< L), or -1
};

__device__ __forceinline__ Tile tile_of(const BwdParams& p, int blk) {
  Tile t;
  t.b = blk / p.tiles_b;
  int local = blk - t.b * p.tiles_b;
  int lo = 0, hi = p.H;  // the head: head_tile_off[h] <= local < head_tile_off[h + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.head_tile_off[mid] <= local) lo = mid; else hi = mid;
  }
  t.h = lo;
  local -= p.head_tile_off[lo];
  t.delta = p.dil[t.h];
  t.half = p.half_h[t.h];
  t.right = p.causal ? 0 : t.half;
  // classes r < rem hold q + 1 positions, the others q
  const int q = p.n / t.delta, rem = p.n % t.delta;
  const int c1 = (q + 1 + kTR - 1) / kTR, c0 = (q + kTR - 1) / kTR;
  if (local < rem * c1) {
    t.r = local / c1;
    t.m0 = (local - t.r * c1) * kTR;
  } else {
    const int l2 = local - rem * c1;
    t.r = rem + l2 / c0;
    t.m0 = (l2 - (t.r - rem) * c0) * kTR;
  }
  t.n_r = (p.n - t.r + t.delta - 1) / t.delta;
  t.bh = (int64_t)(p.b0 + t.b) * p.Htot + p.h0 + t.h;
  t.L = p.n - p.pad[t.b];
  t.mlast = t.L > t.r ? min(t.n_r - 1, (t.L - 1 - t.r) / t.delta) : -1;
  return t;
}

// rows of src (row indices given by rowid(k), -1 for a zero row) into
// dst[kRows][SD] as floats, d columns then zeros up to D
template <typename T, int D, int kRows, typename F>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int d, F rowid) {
  constexpr int SD = D + 4;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    // bf16 rows (d == D, a multiple of 8): 16-byte loads of 8 values
    constexpr int CH = D / 8;
    for (int idx = threadIdx.x; idx < kRows * CH; idx += kThreads) {
      const int k = idx / CH, c8 = idx % CH;
      const int row = rowid(k);
      uint4 x = make_uint4(0, 0, 0, 0);
      if (row >= 0) x = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)row * D) + c8);
      const float4 lo = make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u),
                                    __uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
      const float4 hi = make_float4(__uint_as_float(x.z << 16), __uint_as_float(x.z & 0xffff0000u),
                                    __uint_as_float(x.w << 16), __uint_as_float(x.w & 0xffff0000u));
      *reinterpret_cast<float4*>(dst + k * SD + 8 * c8) = lo;
      *reinterpret_cast<float4*>(dst + k * SD + 8 * c8 + 4) = hi;
    }
  } else {
    for (int idx = threadIdx.x; idx < kRows * D; idx += kThreads) {
      const int k = idx / D, c = idx % D;
      const int row = rowid(k);
      dst[k * SD + c] = (row >= 0 && c < d) ? ldf(src + (int64_t)row * d + c) : 0.f;
    }
  }
}

// 4 x 2 block of <A[ra + i], B[rb + j]> over D columns (A, B row stride D + 4),
// for two pairs of operands at once: (a1, b1) and (a2, b2)
template <int D>
__device__ __forceinline__ void dot_block(const float* a1, const float* b1, const float* a2, const float* b2,
                                          int ra, int rb0, int rb1, float (&x)[4][2], float (&y)[4][2]) {
  constexpr int SD = D + 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i][0] = x[i][1] = y[i][0] = y[i][1] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    float4 av[4], cv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      av[i] = *reinterpret_cast<const float4*>(a1 + (ra + i) * SD + c);
      cv[i] = *reinterpret_cast<const float4*>(a2 + (ra + i) * SD + c);
    }
    const float4 b0 = *reinterpret_cast<const float4*>(b1 + rb0 * SD + c);
    const float4 b1v = *reinterpret_cast<const float4*>(b1 + rb1 * SD + c);
    const float4 d0 = *reinterpret_cast<const float4*>(b2 + rb0 * SD + c);
    const float4 d1 = *reinterpret_cast<const float4*>(b2 + rb1 * SD + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i][0] = fmaf(av[i].x, b0.x, fmaf(av[i].y, b0.y, fmaf(av[i].z, b0.z, fmaf(av[i].w, b0.w, x[i][0]))));
      x[i][1] = fmaf(av[i].x, b1v.x, fmaf(av[i].y, b1v.y, fmaf(av[i].z, b1v.z, fmaf(av[i].w, b1v.w, x[i][1]))));
      y[i][0] = fmaf(cv[i].x, d0.x, fmaf(cv[i].y, d0.y, fmaf(cv[i].z, d0.z, fmaf(cv[i].w, d0.w, y[i][0]))));
      y[i][1] = fmaf(cv[i].x, d1.x, fmaf(cv[i].y, d1.y, fmaf(cv[i].z, d1.z, fmaf(cv[i].w, d1.w, y[i][1]))));
    }
  }
}

// Shared-memory bytes of the tiled kernels (fp32 operand tiles, row stride D + 4).
template <int D>
constexpr int rows_smem_bytes() {
  return (2 * kTR + 2 * kKC) * (D + 4) * 4 + 2 * kTR * (kKC + 1) * 4 + 4 * kTR * 4;
}
template <int D>
constexpr int keys_smem_bytes() {
  return (2 * kTR + 2 * kKC) * (D + 4) * 4 + 2 * kTR * (kKC + 1) * 4 + (3 * kKC + kTR) * 4;
}

// ---------------------------------------------------------------- rows_tiled
// 64 class rows [m0, m0 + 64): thread (ty, tx) = (tid / 16, tid % 16) holds
// rows 4ty..4ty+3 and keys tx, tx + 16 of every 32-key chunk; for dq it owns
// rows 4ty..4ty+3 and columns [tx * D/16, (tx + 1) * D/16).  At d = 128 the
// accumulators need more than half the register file per thread: one CTA
// per SM.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, D == 128 ? 1 : 2) bwd_rows_tiled(BwdParams p, const T* __restrict__ q,
                                                          const T* __restrict__ k, const T* __restrict__ v,
                                                          const T* __restrict__ dout, float* __restrict__ dq,
                                                          float2* __restrict__ stats) {
  constexpr int SD = D + 4, CPT = D / 16;
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                 // [64][SD]
  float* Ds = Qs + kTR * SD;      // dout rows [64][SD]
  float* Ks = Ds + kTR * SD;      // [32][SD]
  float* Vs = Ks + kKC * SD;      // [32][SD]
  float* dS = Vs + kKC * SD;      // [64][33]: e dp of the chunk
  float* rl = dS + 2 * kTR * (kKC + 1);  // (e of the chunk in the [64][33] before rl)
  float* rD = rl + kTR;              // per row: D
  int* rpos = reinterpret_cast<int*>(rD + kTR);  // per row: position, -1 if not an ordinary valid row
  int* rzero = rpos + kTR;                      // per row: position whose dq row is written as zeros, or -1

  const Tile t = tile_of(p, blockIdx.x);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int d = p.d;
  const T* qb = q + t.bh * p.n * d;
  const T* kb = k + t.bh * p.n * d;
  const T* vb = v + t.bh * p.n * d;
  const T* db = dout + t.bh * p.n * d;
  if (tid < kTR) {
    const int m = t.m0 + tid;
    int pos = -1, zero = -1;
    if (m < t.n_r) {
      const int i = t.r + t.delta * m;
      if (i >= t.L || (p.G > 0 && grank(p, i) >= 0)) zero = i;  // padding, or a global token's position
      else pos = i;
    }
    rpos[tid] = pos;
    rzero[tid] = zero;
  }
  __syncthreads();
  stage_rows<T, D, kTR>(Qs, qb, d, [&](int a) { return rpos[a]; });
  stage_rows<T, D, kTR>(Ds, db, d, [&](int a) { return rpos[a]; });

  // keys: band class coordinates [klo, khi], then the global list in chunks
  const int klo = max(0, t.m0 - t.half);
  const int khi = min(t.m0 + kTR - 1 + t.right, t.mlast);
  const int nband = khi >= klo ? (khi - klo + 1 + kKC - 1) / kKC : 0;
  const int nglob = (p.G + kKC - 1) / kKC;
  const int nchunks = nband + nglob;
  // the bias of this head, indexed by window step
  const float* brow = p.rel_bias ? p.rel_bias + (int64_t)(p.h0 + t.h) * p.rb_stride + p.rb_half : nullptr;

  // the key (position) of chunk column kk, or -1 (also for a global token in
  // the padding: it is staged as zeros, so that whatever it holds cannot reach
  // dq through a zero weight)
  auto key_at = [&](int c, int kk) -> int {
    if (c < nband) {
      const int mk = klo + c * kKC + kk;
      return mk <= khi ? t.r + t.delta * mk : -1;
    }
    const int gi = (c - nband) * kKC + kk;
    return (gi < p.G && p.gidx[gi] < t.L) ? p.gidx[gi] : -1;
  };
  // is key j (chunk c) attended by row a?
  auto attends = [&](int a, int c, int j) -> bool {
    const int i = rpos[a];
    if (i < 0 || j < 0) return false;
    if (c < nband) {
      const int off = (j - i) / t.delta;  // same class: exact
      return off >= -t.half && off <= t.right;
    }
    return j < t.L && (!p.causal || j <= i) && !in_band(p, t.h, i, j, t.delta);
  };

  // One sweep over the chunks with a running row maximum mx (shared by the 16
  // threads of a row group): e = 2^(s - mx), ls = sum e, as = sum e dp, and
  // the dq accumulators A = sum (e dp) k and Bk = sum e k, rescaled when mx
  // rises; at the end D = as / ls and dq = scale (A - D Bk) / ls.
  float mx[4], ls[4], as[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mx[i] = -INFINITY;
    ls[i] = as[i] = 0.f;
  }
  float accA[4][CPT], accB[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) accA[i][cc] = accB[i][cc] = 0.f;
  float* Es = rl - kTR * (kKC + 1);  // e of the chunk [64][33] (just below rl)
  float s[4][2], dp[4][2];
  for (int c = 0; c < nchunks; ++c) {
    __syncthreads();  // the previous chunk's K, V, e and e dp are no longer read
    stage_rows<T, D, kKC>(Ks, kb, d, [&](int kk) { return key_at(c, kk); });
    stage_rows<T, D, kKC>(Vs, vb, d, [&](int kk) { return key_at(c, kk); });
    __syncthreads();
    dot_block<D>(Qs, Ks, Ds, Vs, 4 * ty, tx, tx + 16, s, dp);
    bool att[4][2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int key = key_at(c, tx + 16 * j);
#pragma unroll
      for (int i = 0; i < 4; ++i) att[i][j] = attends(4 * ty + i, c, key);
    }
    // scores in the exp2 domain, with the bias on the band keys
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        s[i][j] *= p.sl2;
        if (p.rel_bias && c < nband && att[i][j])
          s[i][j] += __ldg(brow + (klo + c * kKC + tx + 16 * j) - (t.m0 + 4 * ty + i)) * kLog2e;
      }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (att[i][j]) cm = fmaxf(cm, s[i][j]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      if (cm > mx[i]) {
        const float f = exp2f(mx[i] - cm);  // 0 while mx is -inf
        ls[i] *= f;
        as[i] *= f;
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) {
          accA[i][cc] *= f;
          accB[i][cc] *= f;
        }
        mx[i] = cm;
      }
      const int row = 4 * ty + i;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float e = 0.f;
        if (att[i][j]) e = exp2f(s[i][j] - mx[i]);
        ls[i] += e;
        as[i] = fmaf(e, dp[i][j], as[i]);
        Es[row * (kKC + 1) + tx + 16 * j] = e;
        dS[row * (kKC + 1) + tx + 16 * j] = e * dp[i][j];
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kKC; ++kk) {
      float kv[CPT];
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) kv[cc] = Ks[kk * SD + tx * CPT + cc];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float xe = Es[(4 * ty + i) * (kKC + 1) + kk];
        const float xd = dS[(4 * ty + i) * (kKC + 1) + kk];
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) {
          accB[i][cc] = fmaf(xe, kv[cc], accB[i][cc]);
          accA[i][cc] = fmaf(xd, kv[cc], accA[i][cc]);
        }
      }
    }
  }
  // the row group's totals (the 16 threads share mx)
  float acc[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float l = ls[i], a = as[i];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, o);
      a += __shfl_xor_sync(0xffffffffu, a, o);
    }
    const int row = 4 * ty + i;
    const bool ok = rpos[row] >= 0 && l > 0.f;
    const float Drow = ok ? a / l : 0.f, inv = ok ? 1.f / l : 0.f;
    if (tx == 0 && ok) stats[((int64_t)t.b * p.H + t.h) * p.n + rpos[row]] = make_float2(mx[i] + log2f(l), Drow);
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) acc[i][cc] = (accA[i][cc] - Drow * accB[i][cc]) * inv;
  }
  // write dq rows (zeros at padding and global tokens' positions)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 4 * ty + i;
    const int pos = rpos[row] >= 0 ? rpos[row] : rzero[row];
    if (pos < 0) continue;
    float* out = dq + (t.bh * p.n + pos) * d;
    const bool zero = rpos[row] < 0;
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      const int col = tx * CPT + cc;
      if (col < d) out[col] = zero ? 0.f : acc[i][cc] * p.scale;
    }
  }
}

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

// ---------------------------------------------------------------- keys_tiled
// 64 class keys [m0, m0 + 64): dk, dv from the ordinary rows whose band holds
// them (rows of global tokens excluded; the global columns' other rows are
// added by bwd_gkeys).  Thread (ty, tx) holds keys 4ty..4ty+3 and rows tx,
// tx + 16 of every 32-row chunk; for the accumulation keys 4ty..4ty+3 and
// columns [tx * D/16, (tx + 1) * D/16).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, D == 128 ? 1 : 2) bwd_keys_tiled(BwdParams p, const T* __restrict__ q,
                                                          const T* __restrict__ k, const T* __restrict__ v,
                                                          const T* __restrict__ dout, float* __restrict__ dk,
                                                          float* __restrict__ dv, const float2* __restrict__ stats) {
  constexpr int SD = D + 4, CPT = D / 16;
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                    // [64][SD]
  float* Vs = Ks + kTR * SD;         // [64][SD]
  float* Qs = Vs + kTR * SD;         // [32][SD]
  float* Ds = Qs + kKC * SD;         // dout rows [32][SD]
  float* Ps = Ds + kKC * SD;         // [64][33]
  float* dSs = Ps + kTR * (kKC + 1);  // [64][33]
  float* cl = dSs + kTR * (kKC + 1);  // per chunk row: log2-sum-exp
  float* cD = cl + kKC;               // per chunk row: D
  int* crow = reinterpret_cast<int*>(cD + kKC);  // per chunk row: position or -1
  int* kpos = crow + kKC;                       // per key: position if valid (< L), else -1
  float* bacc = reinterpret_cast<float*>(kpos + kTR);  // bias gradient by window step (drb_part only)

  const Tile t = tile_of(p, blockIdx.x);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int d = p.d;
  const T* qb = q + t.bh * p.n * d;
  const T* kb = k + t.bh * p.n * d;
  const T* vb = v + t.bh * p.n * d;
  const T* db = dout + t.bh * p.n * d;
  const float2* st = stats + ((int64_t)t.b * p.H + t.h) * p.n;
  for (int a = tid; a < kTR; a += kThreads) {
    const int m = t.m0 + a;
    kpos[a] = (m <= t.mlast) ? t.r + t.delta * m : -1;
  }
  if (p.drb_part)
    for (int u = tid; u < p.rb_stride; u += kThreads) bacc[u] = 0.f;
  const float* brow = p.rel_bias ? p.rel_bias + (int64_t)(p.h0 + t.h) * p.rb_stride + p.rb_half : nullptr;
  __syncthreads();
  stage_rows<T, D, kTR>(Ks, kb, d, [&](int a) { return kpos[a]; });
  stage_rows<T, D, kTR>(Vs, vb, d, [&](int a) { return kpos[a]; });

  // rows whose band can hold a key of the tile: class coordinates [rlo, rhi]
  const int rlo = max(0, t.m0 - t.right);
  const int rhi = min(t.m0 + kTR - 1 + t.half, t.mlast);
  const int nchunks = rhi >= rlo ? (rhi - rlo + 1 + kKC - 1) / kKC : 0;

  float accv[4][CPT], acck[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) accv[i][cc] = acck[i][cc] = 0.f;
  float s[4][2], dp[4][2];
  for (int c = 0; c < nchunks; ++c) {
    __syncthreads();  // the previous chunk's rows are no longer read
    if (tid < kKC) {
      const int mr = rlo + c * kKC + tid;
      int i = -1;
      if (mr <= rhi) {
        i = t.r + t.delta * mr;
        if (p.G > 0 && grank(p, i) >= 0) i = -1;  // a global token's row uses kg, vg
      }
      crow[tid] = i;
      const float2 x = i >= 0 ? st[i] : make_float2(INFINITY, 0.f);
      cl[tid] = x.x;
      cD[tid] = x.y;
    }
    __syncthreads();
    stage_rows<T, D, kKC>(Qs, qb, d, [&](int kk) { return crow[kk]; });
    stage_rows<T, D, kKC>(Ds, db, d, [&](int kk) { return crow[kk]; });
    __syncthreads();
    dot_block<D>(Ks, Qs, Vs, Ds, 4 * ty, tx, tx + 16, s, dp);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int rr = tx + 16 * j;
      const int i = crow[rr];
      const int mr = rlo + c * kKC + rr;
#pragma unroll
      for (int a4 = 0; a4 < 4; ++a4) {
        const int a = 4 * ty + a4;
        const int off = (t.m0 + a) - mr;  // key offset from the row, in class steps
        float pv = 0.f, ds = 0.f;
        if (i >= 0 && kpos[a] >= 0 && off >= -t.half && off <= t.right) {
          float s2 = s[a4][j] * p.sl2;
          if (brow) s2 += __ldg(brow + off) * kLog2e;
          pv = exp2f(s2 - cl[rr]);
          ds = pv * (dp[a4][j] - cD[rr]);
        }
        Ps[a * (kKC + 1) + rr] = pv;
        dSs[a * (kKC + 1) + rr] = ds;
      }
    }
    __syncthreads();
    if (p.drb_part) {
      // the bias gradient: ds summed along the chunk's diagonals, on which
      // the window step (key - row) is constant; one thread per diagonal,
      // rows in order
      const int o0 = t.m0 - (rlo + c * kKC);  // the step at key 0, chunk row 0
      for (int u = tid; u < kTR + kKC - 1; u += kThreads) {
        const int dl = u - (kKC - 1);  // key - chunk row
        const int o = o0 + dl;
        if (o < -t.half || o > t.right) continue;
        float sum = 0.f;
        for (int rr = max(0, -dl); rr < kKC && rr + dl < kTR; ++rr) sum += dSs[(rr + dl) * (kKC + 1) + rr];
        bacc[o + p.rb_half] += sum;
      }
    }
#pragma unroll 4
    for (int rr = 0; rr < kKC; ++rr) {
      float dov[CPT], qv[CPT];
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) {
        dov[cc] = Ds[rr * SD + tx * CPT + cc];
        qv[cc] = Qs[rr * SD + tx * CPT + cc];
      }
#pragma unroll
      for (int a4 = 0; a4 < 4; ++a4) {
        const float pv = Ps[(4 * ty + a4) * (kKC + 1) + rr];
        const float ds = dSs[(4 * ty + a4) * (kKC + 1) + rr];
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) {
          accv[a4][cc] = fmaf(pv, dov[cc], accv[a4][cc]);
          acck[a4][cc] = fmaf(ds, qv[cc], acck[a4][cc]);
        }
      }
    }
  }
  if (p.drb_part) {
    __syncthreads();
    for (int u = tid; u < p.rb_stride; u += kThreads) p.drb_part[(int64_t)blockIdx.x * p.rb_stride + u] = bacc[u];
  }
  // write dk, dv for every class position of the tile (zeros past the valid length)
#pragma unroll
  for (int a4 = 0; a4 < 4; ++a4) {
    const int m = t.m0 + 4 * ty + a4;
    if (m >= t.n_r) continue;
    const int pos = t.r + t.delta * m;
    const bool ok = kpos[4 * ty + a4] >= 0;
    float* okr = dk + (t.bh * p.n + pos) * d;
    float* ovr = dv + (t.bh * p.n + pos) * d;
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      const int col = tx * CPT + cc;
      if (col < d) {
        okr[col] = ok ? acck[a4][cc] * p.scale : 0.f;
        ovr[col] = ok ? accv[a4][cc] : 0.f;
      }
    }
  }
}

// ---------------------------------------------------------------- bias_reduce
// drb[h0 + h][o] += the keys pass's partial sums of head h at step entry o,
// over the launch's batch rows and the head's tiles, in order (block y = h).
__global__ void bwd_bias_reduce(BwdParams p, float* __restrict__ drb) {
  const int h = blockIdx.y;
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.rb_stride) return;
  float sum = 0.f;
  for (int b = 0; b < p.B; ++b)
    for (int tl = p.head_tile_off[h]; tl < p.head_tile_off[h + 1]; ++tl)
      sum += p.drb_part[((int64_t)b * p.tiles_b + tl) * p.rb_stride + o];
  drb[(int64_t)(p.h0 + h) * p.rb_stride + o] += sum;
}

// ---------------------------------------------------------------- grows
// One CTA (8 warps) per global token's row: statistics over its keys (kg,
// every valid key, those up to the token when causal), then dqg.  The warps
// take interleaved 32-key chunks and their partial results are combined in
// warp order.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_grows(BwdParams p, const T* __restrict__ qg,
                                                        const T* __restrict__ kg, const T* __restrict__ vg,
                                                        const T* __restrict__ dout, float* __restrict__ dqg,
                                                        float2* __restrict__ stats) {
  __shared__ float s_q[D], s_do[D];
  __shared__ float wm[kWarps], wl[kWarps], wa[kWarps], fin[2];
  __shared__ float wacc[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = blockIdx.x % p.G;
  const int bhl = blockIdx.x / p.G;
  const int h = bhl % p.H, b = bhl / p.H;
  const int64_t bh = (int64_t)(p.b0 + b) * p.Htot + p.h0 + h;
  const int d = p.d;
  const int g = p.gidx[rg];
  const int L = p.n - p.pad[b];
  float* dqrow = dqg + (bh * p.G + rg) * d;
  if (g >= L) {
    for (int c = threadIdx.x; c < d; c += kWarps * 32) dqrow[c] = 0.f;
    return;
  }
  const int Lg = p.causal ? min(L, g + 1) : L;
  const T* ks = kg + bh * p.n * d;
  const T* vs = vg + bh * p.n * d;
  for (int c = threadIdx.x; c < D; c += kWarps * 32) {
    s_q[c] = c < d ? ldf(qg + (bh * p.G + rg) * d + c) : 0.f;
    s_do[c] = c < d ? ldf(dout + (bh * p.n + g) * d + c) : 0.f;
  }
  __syncthreads();
  // sweep 1
  float mx = -INFINITY, l = 0.f, a = 0.f;
  for (int j = warp * 32 + lane; j < Lg; j += kWarps * 32) {
    const float s2 = dot_row<T, D>(ks + (int64_t)j * d, s_q, d) * p.sl2;
    const float dp = dot_row<T, D>(vs + (int64_t)j * d, s_do, d);
    if (s2 > mx) {
      const float f = exp2f(mx - s2);
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
  if (lane == 0) {
    wm[warp] = M;
    wl[warp] = l;
    wa[warp] = a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float MM = -INFINITY;
    for (int w = 0; w < kWarps; ++w) MM = fmaxf(MM, wm[w]);
    float LL = 0.f, AA = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float ff = (wm[w] == -INFINITY) ? 0.f : exp2f(wm[w] - MM);
      LL += wl[w] * ff;
      AA += wa[w] * ff;
    }
    fin[0] = MM + log2f(LL);
    fin[1] = AA / LL;
    stats[((int64_t)b * p.H + h) * p.n + g] = make_float2(fin[0], fin[1]);
  }
  __syncthreads();
  const float lse2 = fin[0], Drow = fin[1];
  // sweep 2: per warp partial dqg over its chunks
  constexpr int kC = (D + 31) / 32;
  float acc[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) acc[c] = 0.f;
  for (int j0 = warp * 32; j0 < Lg; j0 += kWarps * 32) {
    const int j = j0 + lane;
    float ds = 0.f;
    if (j < Lg) {
      const float s2 = dot_row<T, D>(ks + (int64_t)j * d, s_q, d) * p.sl2;
      const float dp = dot_row<T, D>(vs + (int64_t)j * d, s_do, d);
      ds = exp2f(s2 - lse2) * (dp - Drow);
    }
    const int nu = min(32, Lg - j0);
    for (int u = 0; u < nu; ++u) {
      const float dsu = __shfl_sync(0xffffffffu, ds, u);
      const T* kr = ks + (int64_t)(j0 + u) * d;
#pragma unroll
      for (int c = 0; c < kC; ++c)
        if (lane + 32 * c < d) acc[c] = fmaf(dsu, ldf(kr + lane + 32 * c), acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < kC; ++c)
    if (lane + 32 * c < D) wacc[warp][lane + 32 * c] = acc[c];
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += kWarps * 32) {
    float x = 0.f;
    for (int w = 0; w < kWarps; ++w) x += wacc[w][c];
    dqrow[c] = x * p.scale;
  }
}

// ---------------------------------------------------------------- gkeys
// One CTA (8 warps) per global token's key g: adds to dk[g], dv[g] (written by
// bwd_keys_tiled for the rows whose band holds g) the ordinary rows that
// attend g only as a global column.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_gkeys(BwdParams p, const T* __restrict__ q,
                                                        const T* __restrict__ k, const T* __restrict__ v,
                                                        const T* __restrict__ dout, float* __restrict__ dk,
                                                        float* __restrict__ dv, const float2* __restrict__ stats) {
  __shared__ float s_k[D], s_v[D];
  __shared__ float wk[kWarps][D], wv[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = blockIdx.x % p.G;
  const int bhl = blockIdx.x / p.G;
  const int h = bhl % p.H, b = bhl / p.H;
  const int64_t bh = (int64_t)(p.b0 + b) * p.Htot + p.h0 + h;
  const int d = p.d;
  const int g = p.gidx[rg];
  const int L = p.n - p.pad[b];
  if (g >= L) return;  // padding: bwd_keys_tiled wrote zeros
  const int delta = p.dil[h];
  const float2* st = stats + ((int64_t)b * p.H + h) * p.n;
  for (int c = threadIdx.x; c < D; c += kWarps * 32) {
    s_k[c] = c < d ? ldf(k + (bh * p.n + g) * d + c) : 0.f;
    s_v[c] = c < d ? ldf(v + (bh * p.n + g) * d + c) : 0.f;
  }
  __syncthreads();
  constexpr int kC = (D + 31) / 32;
  float ak[kC], av[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) ak[c] = av[c] = 0.f;
  const int lo = p.causal ? g : 0;
  for (int i0 = lo + warp * 32; i0 < L; i0 += kWarps * 32) {
    const int i = i0 + lane;
    float pr = 0.f, ds = 0.f;
    bool use = i < L && !in_band(p, h, i, g, delta) && !(p.G > 0 && grank(p, i) >= 0);
    if (use) {
      const float2 sd = st[i];
      const int64_t orow = bh * p.n + i;
      const float s2 = dot_row<T, D>(q + orow * d, s_k, d) * p.sl2;
      const float dp = dot_row<T, D>(dout + orow * d, s_v, d);
      pr = exp2f(s2 - sd.x);
      ds = pr * (dp - sd.y);
    }
    const int nu = min(32, L - i0);
    for (int u = 0; u < nu; ++u) {
      const float pu = __shfl_sync(0xffffffffu, pr, u);
      const float dsu = __shfl_sync(0xffffffffu, ds, u);
      if (pu == 0.f && dsu == 0.f) continue;
      const int64_t orow = bh * p.n + i0 + u;
#pragma unroll
      for (int c = 0; c < kC; ++c) {
        if (lane + 32 * c < d) {
          av[c] = fmaf(pu, ldf(dout + orow * d + lane + 32 * c), av[c]);
          ak[c] = fmaf(dsu, ldf(q + orow * d + lane + 32 * c), ak[c]);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kC; ++c)
    if (lane + 32 * c < D) {
      wk[warp][lane + 32 * c] = ak[c];
      wv[warp][lane + 32 * c] = av[c];
    }
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += kWarps * 32) {
    float xk = 0.f, xv = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      xk += wk[w][c];
      xv += wv[w][c];
    }
    dk[(bh * p.n + g) * d + c] += xk * p.scale;
    dv[(bh * p.n + g) * d + c] += xv;
  }
}

// ---------------------------------------------------------------- kgvg
// One warp per key position j: dkg_j, dvg_j from the global rows (the row of
// global token g attends every valid key, those up to g when causal).
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_kgvg(BwdParams p, const T* __restrict__ qg,
                                                       const T* __restrict__ kg, const T* __restrict__ vg,
                                                       const T* __restrict__ dout, float* __restrict__ dkg,
                                                       float* __restrict__ dvg, const float2* __restrict__ stats) {
  __shared__ float s_k[kWarps][D], s_v[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = (int64_t)blockIdx.x * kWarps + warp;
  if (id >= (int64_t)p.B * p.H * p.n) return;
  const int j = (int)(id % p.n);
  const int64_t bhl = id / p.n;
  const int h = (int)(bhl % p.H), b = (int)(bhl / p.H);
  const int64_t bh = (int64_t)(p.b0 + b) * p.Htot + p.h0 + h;
  const int d = p.d;
  const int L = p.n - p.pad[b];
  const int64_t krow = bh * p.n + j;
  const float2* st = stats + ((int64_t)b * p.H + h) * p.n;
  constexpr int kC = (D + 31) / 32;
  float ak[kC], av[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) ak[c] = av[c] = 0.f;
  if (j < L) {
    for (int c = lane; c < D; c += 32) {
      s_k[warp][c] = c < d ? ldf(kg + krow * d + c) : 0.f;
      s_v[warp][c] = c < d ? ldf(vg + krow * d + c) : 0.f;
    }
    __syncwarp();
    for (int t0 = 0; t0 < p.G; t0 += 32) {
      const int tt = t0 + lane;
      int g = -1;
      if (tt < p.G) {
        g = p.gidx[tt];
        if (g >= L || (p.causal && j > g)) g = -1;
      }
      float pr = 0.f, ds = 0.f;
      if (g >= 0) {
        const float2 sd = st[g];
        const float s2 = dot_row<T, D>(qg + (bh * p.G + tt) * d, s_k[warp], d) * p.sl2;
        const float dp = dot_row<T, D>(dout + (bh * p.n + g) * d, s_v[warp], d);
        pr = exp2f(s2 - sd.x);
        ds = pr * (dp - sd.y);
      }
      const int nu = min(32, p.G - t0);
      for (int u = 0; u < nu; ++u) {
        const int gu = __shfl_sync(0xffffffffu, g, u);
        const float pu = __shfl_sync(0xffffffffu, pr, u);
        const float dsu = __shfl_sync(0xffffffffu, ds, u);
        if (gu < 0) continue;
        const T* qr = qg + (bh * p.G + t0 + u) * d;
        const T* dr = dout + (bh * p.n + gu) * d;
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
