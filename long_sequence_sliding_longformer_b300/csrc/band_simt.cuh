// band_simt.cuh -- fp32 band attention on CUDA cores (one warp per query row).
//
// Same pattern as the tensor-core kernel (velog.io/@lainshower/Longformer,
// section 3-1: sliding / dilated window and global columns; section 4.1:
// look-back-only window), with fp32 inputs, fp32 arithmetic and the accurate
// expf.  Lanes take 32 keys at a time: each lane scores one key, the warp
// updates a running maximum and sum, and each lane accumulates d/32 output
// columns.  Rows of global tokens are left to the global-row kernels.
#pragma once

#include "lf_internal.cuh"

namespace lf {

constexpr int kSimtWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// rank of position i in the sorted global list, or -1
__device__ __forceinline__ int global_rank(const PatternParams& p, int i) {
  int lo = 0, hi = p.G - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int g = p.gidx[mid];
    if (g == i) return mid;
    if (g < i) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

__global__ void __launch_bounds__(kSimtWarps * 32)
band_simt_f32_kernel(const __grid_constant__ SimtParams sp, const float* __restrict__ q,
                     const float* __restrict__ k, const float* __restrict__ v,
                     float* __restrict__ out) {
  const PatternParams& p = sp.pat;
  __shared__ float qs[kSimtWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t flat = (int64_t)blockIdx.x * kSimtWarps + warp;
  const int64_t total = (int64_t)p.B * p.H * p.n;
  if (flat >= total) return;
  const int D = p.d;
  const int i = (int)(flat % p.n);
  const int64_t bh = flat / p.n;
  const int h = (int)(bh % p.H);
  const int b = (int)(bh / p.H);
  const int L = p.n - p.pad[b];
  float* orow = out + flat * D;
  if (i >= L) {
    for (int c = lane; c < D; c += 32) orow[c] = 0.f;
    return;
  }
  if (p.G > 0 && global_rank(p, i) >= 0) return;

  const float* qrow = q + flat * D;
  for (int c = lane; c < D; c += 32) qs[warp][c] = qrow[c];
  __syncwarp();
  const int delta = sp.dil[h];
  const int half = sp.half_h[h], right = p.causal ? 0 : half;
  // window steps t with key j = i + delta*t inside [0, L)
  const int tlo = max(-half, -(i / delta));
  const int thi = min(right, (L - 1 - i) / delta);
  const float* kb = k + bh * (int64_t)p.n * D;
  const float* vb = v + bh * (int64_t)p.n * D;
  const float NEG_INF = -__int_as_float(0x7f800000);
  float m = NEG_INF, l = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  auto update = [&](float s, int j, bool valid) {
    const float cmax = warp_max(valid ? s : NEG_INF);
    const float m_new = fmaxf(m, cmax);
    if (m_new == NEG_INF) return;  // nothing valid yet (warp-uniform)
    const float alpha = expf(m - m_new);
    const float pj = valid ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] *= alpha;
    for (int kk = 0; kk < 32; ++kk) {
      const float pk = __shfl_sync(0xffffffffu, pj, kk);
      const int jk = __shfl_sync(0xffffffffu, j, kk);
      if (pk != 0.f) {
        const float* vr = vb + (int64_t)jk * D;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = lane + 32 * u;
          if (c < D) acc[u] += pk * vr[c];
        }
      }
    }
    m = m_new;
  };

  for (int t0 = tlo; t0 <= thi; t0 += 32) {
    const int t = t0 + lane;
    const bool valid = t <= thi;
    const int j = valid ? i + delta * t : 0;
    float s = NEG_INF;
    if (valid) {
      const float* kr = kb + (int64_t)j * D;
      float a = 0.f;
      for (int c = 0; c < D; ++c) a = fmaf(qs[warp][c], kr[c], a);
      s = a * p.scale;
      if (sp.rel_bias) s += __ldg(sp.rel_bias + (int64_t)h * sp.rb_stride + sp.rb_half + t);
    }
    update(s, j, valid);
  }
  for (int g0 = 0; g0 < p.G; g0 += 32) {
    const int r = g0 + lane;
    bool valid = r < p.G;
    const int g = valid ? p.gidx[r] : 0;
    if (valid) valid = g < L && (!p.causal || g <= i);
    if (valid) {  // a global key already inside the window is counted there
      const int off = g - i;
      if (off % delta == 0) {
        const int st = off / delta;
        if (st >= -half && st <= right) valid = false;
      }
    }
    float s = NEG_INF;
    if (valid) {
      const float* kr = kb + (int64_t)g * D;
      float a = 0.f;
      for (int c = 0; c < D; ++c) a = fmaf(qs[warp][c], kr[c], a);
      s = a * p.scale;
    }
    update(s, g, valid);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = lane + 32 * u;
    if (c < D) orow[c] = acc[u] * inv;
  }
}

lf_status launch_band_simt_f32(const SimtParams& p, const float* q, const float* k, const float* v,
                               float* out, cudaStream_t s) {
  const int64_t rows = (int64_t)p.pat.B * p.pat.H * p.pat.n;
  const int64_t blocks = (rows + kSimtWarps - 1) / kSimtWarps;
  if (blocks > 0x7fffffff) {
    set_error("fp32 band kernel: too many rows (%lld)", (long long)rows);
    return LF_ERR_UNSUPPORTED;
  }
  band_simt_f32_kernel<<<(unsigned)blocks, kSimtWarps * 32, 0, s>>>(p, q, k, v, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("fp32 band kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

}  // namespace lf
