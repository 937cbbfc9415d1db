// global_rows.cuh -- rows of the global tokens (velog.io/@lainshower/Longformer,
// section 3-1 "Global Attention" and "Linear Projections for Global Attention").
//
// A global token g attends to every valid key j (j <= g when causal) using
// its own projections: softmax(qg[g] . kg[j] / sqrt(d)) averaged over vg[j].
// These few rows are long (n keys each), so the keys are split across CTAs:
//
//   partial pass  grid (key chunks, query blocks, B*H).  Each CTA scores a
//       block of global queries against its chunk of keys, keeps a running
//       (max, sum, weighted value sum) and writes that partial state to a
//       scratch buffer.
//   merge         done by the last CTA of each (query block, B*H) pair to
//       finish (a counter per pair): it merges the partials of its rows in
//       increasing chunk order (a fixed order: results are deterministic),
//       normalises and writes the rows of `out` at the tokens' positions.
//       The band kernels leave those rows alone, so the whole pass may run
//       beside them.
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
//
// Called by every thread of a partial-pass CTA once its partial state is
// written.  The last CTA of query block `qblk` of row set `bh` to get here
// (counters[bh * nqb + qblk] counts them; zero before the pass) merges the
// chunks of rows g0 .. g0 + gq - 1 and writes them to `out`.
template <typename T>
__device__ void merge_if_last(const PatternParams& p, const float* ws, T* __restrict__ out,
                              unsigned* counters, int nchunks, int nqb, int qblk, int g0, int gq,
                              int64_t bh) {
  __shared__ unsigned s_last;
  __threadfence();  // this CTA's partial state is visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&counters[bh * nqb + qblk], 1u) == (unsigned)nchunks - 1u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // and every other CTA's is visible to this one
  const int D = p.d;
  const int b = (int)(bh / p.H);
  const int L = p.n - p.pad[b];
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int64_t cstride = (int64_t)p.G * (D + 2);
  // each thread one (row, column); the chunks are read 16 at a time (all
  // loads of a block in flight together) and added in chunk order
  constexpr int kBlk = 16;
  for (int idx = threadIdx.x; idx < gq * D; idx += blockDim.x) {
    const int g = idx / D, c = idx - (idx / D) * D;
    const float* base = ws + ((bh * nchunks) * p.G + g0 + g) * (D + 2);
    float M = NEG_INF;
    for (int ch0 = 0; ch0 < nchunks; ch0 += kBlk) {
      float mv[kBlk];
#pragma unroll
      for (int u = 0; u < kBlk; ++u) mv[u] = (ch0 + u < nchunks) ? __ldcg(base + (ch0 + u) * cstride) : NEG_INF;
#pragma unroll
      for (int u = 0; u < kBlk; ++u) M = fmaxf(M, mv[u]);
    }
    float l = 0.f, a = 0.f;
    if (M != NEG_INF) {
      for (int ch0 = 0; ch0 < nchunks; ch0 += kBlk) {
        float mv[kBlk], lv[kBlk], av[kBlk];
#pragma unroll
        for (int u = 0; u < kBlk; ++u) {
          const bool in = ch0 + u < nchunks;
          const float* e = base + (ch0 + u) * cstride;
          mv[u] = in ? __ldcg(e) : NEG_INF;
          lv[u] = in ? __ldcg(e + 1) : 0.f;
          av[u] = in ? __ldcg(e + 2 + c) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBlk; ++u) {
          if (mv[u] == NEG_INF) continue;  // nothing attended in this chunk: skip, never scale by 0
          const float f = ex2_approx(mv[u] - M);
          l = fmaf(lv[u], f, l);
          a = fmaf(av[u], f, a);
        }
      }
    }
    const int pos = p.gidx[g0 + g];
    from_f<T>(out + (bh * p.n + pos) * D + c, (pos < L && l > 0.f) ? a / l : 0.f);
  }
}

template <typename T>
__global__ void __launch_bounds__(kGThreads)
global_partial_kernel(const __grid_constant__ PatternParams p, const T* __restrict__ qg,
                      const T* __restrict__ kg, const T* __restrict__ vg, float* __restrict__ ws,
                      T* __restrict__ out, unsigned* counters, int nchunks, int chunk) {
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
          if (w == 0.f) continue;  // an unattended key's value never enters the sum
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
      if (ms != NEG_INF) run_acc[g][c] = run_acc[g][c] * fo + a * ex2_approx(ms - mn);
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
  merge_if_last<T>(p, ws, out, counters, nchunks, gridDim.y, blockIdx.y, g0, gq, bh);
}

// bf16 streaming variant for a few global queries (NQ <= 8 per CTA).  Each
// key row is split into 16-byte chunks across CH = D/8 lanes, so a warp reads
// 32/CH whole rows per step with coalesced 16-byte loads; a lane keeps the
// running (max, sum, weighted values) of its key slot for its 8 columns, and
// the slots and warps are merged in a fixed order at the end.
constexpr int kGsWarps = 4;

template <int D, int NQ>
__global__ void __launch_bounds__(kGsWarps * 32)
global_partial_stream_kernel(const __grid_constant__ PatternParams p,
                             const __nv_bfloat16* __restrict__ qg,
                             const __nv_bfloat16* __restrict__ kg,
                             const __nv_bfloat16* __restrict__ vg, float* __restrict__ ws,
                             __nv_bfloat16* __restrict__ out, unsigned* counters, int nchunks,
                             int chunk) {
  constexpr int CH = D / 8;       // 16-byte chunks per row
  constexpr int KPW = 32 / CH;    // key rows per warp step
  __shared__ float red[kGsWarps][NQ][D + 2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = lane / CH, c = lane % CH;
  const int g0 = blockIdx.x * NQ;
  const int c_idx = blockIdx.y;
  const int64_t bh = blockIdx.z;
  const int gq = min(NQ, p.G - g0);
  const int b = (int)(bh / p.H);
  const int L = p.n - p.pad[b];
  const float sl2 = p.scale * 1.4426950408889634f;
  const float NEG_INF = -__int_as_float(0x7f800000);

  float qv[NQ][8];
  int gpos[NQ];
#pragma unroll
  for (int g = 0; g < NQ; ++g) {
    gpos[g] = (g < gq) ? p.gidx[g0 + g] : -1;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (g < gq) x = __ldg(reinterpret_cast<const uint4*>(qg + ((bh * p.G) + g0 + g) * D) + c);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      qv[g][2 * e] = f.x * sl2;
      qv[g][2 * e + 1] = f.y * sl2;
    }
  }
  float m[NQ], l[NQ], acc[NQ][8];
#pragma unroll
  for (int g = 0; g < NQ; ++g) {
    m[g] = NEG_INF;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  }

  const int k_begin = c_idx * chunk;
  const int k_end = min(k_begin + chunk, L);
  const uint4* kb = reinterpret_cast<const uint4*>(kg + bh * (int64_t)p.n * D);
  const uint4* vb = reinterpret_cast<const uint4*>(vg + bh * (int64_t)p.n * D);
  constexpr int U = NQ <= 2 ? 8 : 4;  // key steps in flight per warp
  constexpr int STEP = kGsWarps * KPW;
  for (int j00 = k_begin + warp * KPW; j00 < k_end; j00 += U * STEP) {
   uint4 kxs[U], vxs[U];
#pragma unroll
   for (int u = 0; u < U; ++u) {
    const int j = j00 + u * STEP + ks;
    kxs[u] = make_uint4(0, 0, 0, 0);
    vxs[u] = make_uint4(0, 0, 0, 0);
    if (j < k_end) {
      kxs[u] = __ldg(kb + (int64_t)j * CH + c);
      vxs[u] = __ldg(vb + (int64_t)j * CH + c);
    }
   }
#pragma unroll
   for (int u = 0; u < U; ++u) {
    const int j = j00 + u * STEP + ks;
    const bool valid = j < k_end;
    float kf[8], vf[8];
    {
      const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kxs[u]);
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vxs[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = __bfloat1622float2(k2[e]);
        const float2 bb = __bfloat1622float2(v2[e]);
        kf[2 * e] = a.x;
        kf[2 * e + 1] = a.y;
        vf[2 * e] = bb.x;
        vf[2 * e + 1] = bb.y;
      }
    }
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(qv[g][e], kf[e], s);
#pragma unroll
      for (int off = CH / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const bool ok = valid && g < gq && (!p.causal || j <= gpos[g]);
      if (ok) {
        if (s > m[g]) {
          const float alpha = ex2_approx(m[g] - s);  // 0 when m was -inf
          l[g] *= alpha;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
          m[g] = s;
        }
        const float pw = ex2_approx(s - m[g]);
        l[g] += pw;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pw, vf[e], acc[g][e]);
      }
    }
   }
  }
  // merge the key slots of this warp (lanes c, c+CH, ...), in a fixed order
#pragma unroll
  for (int off = CH; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
      const float mn = fmaxf(m[g], m2);
      const float fa = (m[g] == NEG_INF) ? 0.f : ex2_approx(m[g] - mn);
      const float fb = (m2 == NEG_INF) ? 0.f : ex2_approx(m2 - mn);
      l[g] = l[g] * fa + l2 * fb;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float a2 = __shfl_xor_sync(0xffffffffu, acc[g][e], off);
        acc[g][e] = acc[g][e] * fa + a2 * fb;
      }
      m[g] = mn;
    }
  }
  if (ks == 0) {
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
#pragma unroll
      for (int e = 0; e < 8; ++e) red[warp][g][2 + c * 8 + e] = acc[g][e];
      if (c == 0) {
        red[warp][g][0] = m[g];
        red[warp][g][1] = l[g];
      }
    }
  }
  __syncthreads();
  // merge the warps in order and write the chunk's partial state
  for (int idx = tid; idx < gq * (D + 2); idx += kGsWarps * 32) {
    const int g = idx / (D + 2), col = idx - (idx / (D + 2)) * (D + 2);
    float mm = NEG_INF;
#pragma unroll
    for (int w = 0; w < kGsWarps; ++w) mm = fmaxf(mm, red[w][g][0]);
    float val = 0.f;
    if (col == 0) {
      val = mm;
    } else {
#pragma unroll
      for (int w = 0; w < kGsWarps; ++w) {
        const float mw = red[w][g][0];
        const float f = (mw == NEG_INF) ? 0.f : ex2_approx(mw - mm);
        val = fmaf(red[w][g][col], f, val);
      }
    }
    ws[((bh * nchunks + c_idx) * p.G + g0 + g) * (D + 2) + col] = val;
  }
  merge_if_last<__nv_bfloat16>(p, ws, out, counters, nchunks, gridDim.x, blockIdx.x, g0, gq, bh);
}

// Query-block size of the streaming kernel for a given number of global tokens.
inline int stream_nq(int G) { return G >= 8 ? 8 : (G >= 4 ? 4 : (G >= 2 ? 2 : 1)); }

template <typename T>
inline bool launch_partial_stream(const PatternParams&, const T*, const T*, const T*, float*, T*,
                                  unsigned*, int, int, cudaStream_t) {
  return false;  // fp32 inputs use the generic kernel
}

template <int D>
inline void launch_stream_d(const PatternParams& p, const __nv_bfloat16* qg, const __nv_bfloat16* kg,
                            const __nv_bfloat16* vg, float* ws, __nv_bfloat16* out,
                            unsigned* counters, int nchunks, int chunk, cudaStream_t s) {
  const int nq = stream_nq(p.G);
  dim3 grid((p.G + nq - 1) / nq, nchunks, (unsigned)((int64_t)p.B * p.H));
  switch (nq) {
    case 1: global_partial_stream_kernel<D, 1><<<grid, kGsWarps * 32, 0, s>>>(p, qg, kg, vg, ws, out, counters, nchunks, chunk); break;
    case 2: global_partial_stream_kernel<D, 2><<<grid, kGsWarps * 32, 0, s>>>(p, qg, kg, vg, ws, out, counters, nchunks, chunk); break;
    case 4: global_partial_stream_kernel<D, 4><<<grid, kGsWarps * 32, 0, s>>>(p, qg, kg, vg, ws, out, counters, nchunks, chunk); break;
    default: global_partial_stream_kernel<D, 8><<<grid, kGsWarps * 32, 0, s>>>(p, qg, kg, vg, ws, out, counters, nchunks, chunk); break;
  }
}

template <>
inline bool launch_partial_stream<__nv_bfloat16>(const PatternParams& p, const __nv_bfloat16* qg,
                                                 const __nv_bfloat16* kg, const __nv_bfloat16* vg,
                                                 float* ws, __nv_bfloat16* out, unsigned* counters,
                                                 int nchunks, int chunk, cudaStream_t s) {
  if (p.d == 64) launch_stream_d<64>(p, qg, kg, vg, ws, out, counters, nchunks, chunk, s);
  else if (p.d == 128) launch_stream_d<128>(p, qg, kg, vg, ws, out, counters, nchunks, chunk, s);
  else return false;
  return true;
}

// Counters the global-row pass needs for B*H rows sets of G global tokens
// (one per query block; at most one per token).
inline size_t global_counters(int64_t bh, int G) { return (size_t)bh * (size_t)G; }

// The whole global-row pass on stream s: clears the merge counters, then the
// partial kernel (whose last CTAs merge and write the rows of `out`).
template <typename T>
lf_status launch_global_rows(const PatternParams& p, const T* qg, const T* kg, const T* vg, T* out,
                             float* ws, unsigned* counters, int nchunks, int chunk, cudaStream_t s) {
  const int64_t bhs = (int64_t)p.B * p.H;
  if (bhs > 65535 || nchunks > 65535) {
    set_error("global-row kernels: B*H = %lld or %d key chunks exceed the grid limit", (long long)bhs, nchunks);
    return LF_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaMemsetAsync(counters, 0, global_counters(bhs, p.G) * sizeof(unsigned), s);
  if (e != cudaSuccess) {
    set_error("clearing the global-row counters: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  if (!launch_partial_stream(p, qg, kg, vg, ws, out, counters, nchunks, chunk, s)) {
    dim3 g1(nchunks, (p.G + kGQ - 1) / kGQ, (unsigned)bhs);
    global_partial_kernel<T><<<g1, kGThreads, 0, s>>>(p, qg, kg, vg, ws, out, counters, nchunks, chunk);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("global partial kernel launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

template lf_status launch_global_rows<float>(const PatternParams&, const float*, const float*,
                                             const float*, float*, float*, unsigned*, int, int,
                                             cudaStream_t);
template lf_status launch_global_rows<__nv_bfloat16>(const PatternParams&, const __nv_bfloat16*,
                                                     const __nv_bfloat16*, const __nv_bfloat16*,
                                                     __nv_bfloat16*, float*, unsigned*, int, int,
                                                     cudaStream_t);

}  // namespace lf
