// global_rows.cuh -- rows of the global tokens (velog.io/@lainshower/Longformer,
// section 3-1 "Global Attention" and "Linear Projections for Global Attention").
//
// A global token g attends to every valid key j (j <= g when causal) using
// its own projections: softmax(qg[g] . kg[j] / sqrt(d)) averaged over vg[j].
// These few rows are long (n keys each), so the keys are split across CTAs:
//
//   global_partial_kernel  grid (key chunks, query blocks, B*H).  Each CTA
//       scores up to 8 global queries against its chunk of keys, keeps a
//       running (max, sum, weighted value sum) over its sub-chunks of 128 keys
//       and writes that partial state to a scratch buffer.
//   global_merge_kernel    grid (G, B*H).  Merges the partials of one row in
//       increasing chunk order (a fixed order: results are deterministic),
//       normalises and writes the row of `out` at the token's position.
//
// Scores are kept in the exp2 domain (scaled by log2(e)/sqrt(d)).
#pragma once

#include "band_simt.cuh"
#include "lf_internal.cuh"

namespace lf {

constexpr int kGThreads = 128;
constexpr int kGSub = kGThreads;  // keys per sub-chunk (one per thread)
constexpr int kGQ = 8;            // global queries per CTA

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ void from_f(T* dst, float x);
template <>
__device__ __forceinline__ void from_f<float>(float* dst, float x) { *dst = x; }
template <>
__device__ __forceinline__ void from_f<__nv_bfloat16>(__nv_bfloat16* dst, float x) { *dst = __float2bfloat16_rn(x); }

// Scratch layout: per (bh, chunk, g): [m, l, acc[0..d)] as fp32, d + 2 floats.
template <typename T>
__global__ void __launch_bounds__(kGThreads)
global_partial_kernel(const __grid_constant__ PatternParams p, const T* __restrict__ qg,
                      const T* __restrict__ kg, const T* __restrict__ vg, float* __restrict__ ws,
                      int nchunks, int chunk) {
  __shared__ float qs[kGQ][128];
  __shared__ float sc[kGQ][kGSub];
  __shared__ float red[kGThreads / 32][kGQ][128];
  __shared__ float run_m[kGQ], run_l[kGQ], sub_m[kGQ], sub_l[kGQ];
  __shared__ float run_acc[kGQ][128];

  const int D = p.d;
  const int c_idx = blockIdx.x;
  const int g0 = blockIdx.y * kGQ;
  const int gq = min(kGQ, p.G - g0);
  const int64_t bh = blockIdx.z;
  const int b = (int)(bh / p.H);
  const int L = p.n - p.pad[b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float sl2 = p.scale * 1.4426950408889634f;
  const float NEG_INF = -__int_as_float(0x7f800000);

  for (int idx = tid; idx < kGQ * 128; idx += kGThreads) {
    const int g = idx / 128, c = idx % 128;
    qs[g][c] = (g < gq && c < D) ? to_f<T>(qg[((bh * p.G) + g0 + g) * D + c]) : 0.f;
    run_acc[g][c] = 0.f;
  }
  if (tid < kGQ) {
    run_m[tid] = NEG_INF;
    run_l[tid] = 0.f;
  }
  __syncthreads();

  const T* kb = kg + bh * (int64_t)p.n * D;
  const T* vb = vg + bh * (int64_t)p.n * D;
  const int k_begin = c_idx * chunk;
  const int k_end = min(k_begin + chunk, L);

  for (int j0 = k_begin; j0 < k_end; j0 += kGSub) {
    // ---- scores: one key per thread
    {
      const int j = j0 + tid;
      float s[kGQ];
#pragma unroll
      for (int g = 0; g < kGQ; ++g) s[g] = 0.f;
      if (j < k_end) {
        const T* kr = kb + (int64_t)j * D;
        for (int c = 0; c < D; ++c) {
          const float kv = to_f<T>(kr[c]);
#pragma unroll
          for (int g = 0; g < kGQ; ++g) s[g] = fmaf(qs[g][c], kv, s[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < kGQ; ++g) {
        bool ok = j < k_end && g < gq;
        if (ok && p.causal) ok = j <= p.gidx[g0 + g];
        sc[g][tid] = ok ? s[g] * sl2 : NEG_INF;
      }
    }
    __syncthreads();
    // ---- per query: sub-chunk maximum (warp w reduces queries w, w+4)
    for (int g = warp; g < kGQ; g += kGThreads / 32) {
      float mx = NEG_INF;
      for (int t = lane; t < kGSub; t += 32) mx = fmaxf(mx, sc[g][t]);
      mx = warp_max(mx);
      if (lane == 0) sub_m[g] = mx;
    }
    __syncthreads();
    // ---- weights
    for (int idx = tid; idx < kGQ * kGSub; idx += kGThreads) {
      const int g = idx / kGSub, t = idx % kGSub;
      const float m = sub_m[g];
      sc[g][t] = (m == NEG_INF) ? 0.f : ex2_approx(sc[g][t] - m);
    }
    __syncthreads();
    for (int g = warp; g < kGQ; g += kGThreads / 32) {
      float sm = 0.f;
      for (int t = lane; t < kGSub; t += 32) sm += sc[g][t];
      sm = warp_sum(sm);
      if (lane == 0) sub_l[g] = sm;
    }
    // ---- weighted values: warp w takes keys [32w, 32w+32) of the sub-chunk
    {
      float acc[kGQ][4];
#pragma unroll
      for (int g = 0; g < kGQ; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[g][u] = 0.f;
      for (int t = warp * 32; t < warp * 32 + 32; ++t) {
        const int j = j0 + t;
        if (j >= k_end) break;
        const T* vr = vb + (int64_t)j * D;
        float vv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = lane + 32 * u;
          vv[u] = (c < D) ? to_f<T>(vr[c]) : 0.f;
        }
#pragma unroll
        for (int g = 0; g < kGQ; ++g) {
          const float w = sc[g][t];
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[g][u] = fmaf(w, vv[u], acc[g][u]);
        }
      }
#pragma unroll
      for (int g = 0; g < kGQ; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = lane + 32 * u;
          if (c < 128) red[warp][g][c] = acc[g][u];
        }
    }
    __syncthreads();
    // ---- fold the sub-chunk into the running state (fixed warp order)
    for (int idx = tid; idx < kGQ * 128; idx += kGThreads) {
      const int g = idx / 128, c = idx % 128;
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kGThreads / 32; ++w) a += red[w][g][c];
      const float mo = run_m[g], ms = sub_m[g];
      const float mn = fmaxf(mo, ms);
      const float fo = (mo == NEG_INF) ? 0.f : ex2_approx(mo - mn);
      const float fs = (ms == NEG_INF) ? 0.f : ex2_approx(ms - mn);
      run_acc[g][c] = run_acc[g][c] * fo + a * fs;
    }
    __syncthreads();
    if (tid < kGQ) {
      const float mo = run_m[tid], ms = sub_m[tid];
      const float mn = fmaxf(mo, ms);
      const float fo = (mo == NEG_INF) ? 0.f : ex2_approx(mo - mn);
      const float fs = (ms == NEG_INF) ? 0.f : ex2_approx(ms - mn);
      run_l[tid] = run_l[tid] * fo + sub_l[tid] * fs;
      run_m[tid] = mn;
    }
    __syncthreads();
  }
  // ---- write this chunk's partial state
  for (int idx = tid; idx < gq * (D + 2); idx += kGThreads) {
    const int g = idx / (D + 2), c = idx % (D + 2);
    float val;
    if (c == 0) val = run_m[g];
    else if (c == 1) val = run_l[g];
    else val = run_acc[g][c - 2];
    ws[((bh * nchunks + c_idx) * p.G + g0 + g) * (D + 2) + c] = val;
  }
}

template <typename T>
__global__ void __launch_bounds__(128)
global_merge_kernel(const __grid_constant__ PatternParams p, const float* __restrict__ ws,
                    T* __restrict__ out, int nchunks) {
  const int g = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / p.H);
  const int D = p.d;
  const int L = p.n - p.pad[b];
  const int pos = p.gidx[g];
  const float NEG_INF = -__int_as_float(0x7f800000);
  T* orow = out + (bh * p.n + pos) * D;
  const int c = threadIdx.x;
  if (c >= D) return;
  if (pos >= L) {
    from_f<T>(orow + c, 0.f);
    return;
  }
  float M = NEG_INF;
  for (int ch = 0; ch < nchunks; ++ch) M = fmaxf(M, ws[((bh * nchunks + ch) * p.G + g) * (D + 2)]);
  float l = 0.f, a = 0.f;
  if (M != NEG_INF) {
    for (int ch = 0; ch < nchunks; ++ch) {
      const float* e = ws + ((bh * nchunks + ch) * p.G + g) * (D + 2);
      if (e[0] == NEG_INF) continue;
      const float f = ex2_approx(e[0] - M);
      l = fmaf(e[1], f, l);
      a = fmaf(e[2 + c], f, a);
    }
  }
  from_f<T>(orow + c, l > 0.f ? a / l : 0.f);
}

template <typename T>
lf_status launch_global_rows(const PatternParams& p, const T* qg, const T* kg, const T* vg, T* out,
                             float* ws, int nchunks, int chunk, cudaStream_t s) {
  const int64_t bhs = (int64_t)p.B * p.H;
  if (bhs > 65535 || nchunks > 0x7fffffff) {
    set_error("global-row kernels: B*H = %lld exceeds the grid limit", (long long)bhs);
    return LF_ERR_UNSUPPORTED;
  }
  dim3 g1(nchunks, (p.G + kGQ - 1) / kGQ, (unsigned)bhs);
  global_partial_kernel<T><<<g1, kGThreads, 0, s>>>(p, qg, kg, vg, ws, nchunks, chunk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("global partial kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  dim3 g2(p.G, (unsigned)bhs);
  global_merge_kernel<T><<<g2, 128, 0, s>>>(p, ws, out, nchunks);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("global merge kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

template lf_status launch_global_rows<float>(const PatternParams&, const float*, const float*,
                                             const float*, float*, float*, int, int, cudaStream_t);
template lf_status launch_global_rows<__nv_bfloat16>(const PatternParams&, const __nv_bfloat16*,
                                                     const __nv_bfloat16*, const __nv_bfloat16*,
                                                     __nv_bfloat16*, float*, int, int, cudaStream_t);

}  // namespace lf
