// mem_combine.cuh -- the Memorizing-Transformer combine (lf_mem_combine):
// each query attends the km (key, value) pairs a kNN lookup retrieved from a
// memory of earlier segments, and the result is mixed with the local
// attention output by a per-head weight (Memorizing Transformer notes,
// section "Memorizing Transformer": local attention, attention over the k
// retrieved pairs, a weighted sum with one scalar per head).  The lookup
// itself is the caller's; this is the gather, the softmax over the retrieved
// pairs and the mix.  Included at the end of lf_attn.cu.
//
// One warp per query: lane j takes slot j (km <= 32), reads idx and the
// retrieved key row (16-byte loads) and scores it against the query (kept in
// shared memory); the softmax runs across the lanes; then the lanes split d
// and sum the retrieved value rows (coalesced row reads), mix with the local
// row and store bf16.  Bound by the gathers from HBM.
#pragma once

#include "lf_internal.cuh"

namespace lf {
namespace memk {

constexpr int kWarps = 8;
constexpr uint32_t kRoleMemIndex = 7;  // device error word: an index out of range

template <int D>
__global__ void __launch_bounds__(kWarps * 32) mem_combine_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* local, const __nv_bfloat16* __restrict__ mem_k,
    const __nv_bfloat16* __restrict__ mem_v, const int32_t* __restrict__ idx, const float* __restrict__ gate,
    __nv_bfloat16* out, int32_t H, int32_t n, int32_t M, int32_t km, int64_t rows, float sl2) {
  __shared__ float s_q[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= rows) return;
  const int64_t bh = row / n;
  const int h = (int)(bh % H);
  // the query row as floats
  {
    constexpr int PER = D / 32;
    const __nv_bfloat16* qr = q + row * D + lane * PER;
#pragma unroll
    for (int c = 0; c < PER; ++c) s_q[warp][lane * PER + c] = __bfloat162float(qr[c]);
  }
  __syncwarp();
  // slot `lane`: its memory position and score
  int ix = lane < km ? __ldg(idx + row * km + lane) : -1;
  if (ix < -1 || ix >= M) {
    atomicCAS(&g_device_error, 0u, (uint32_t)LF_ERR_INVALID_ARG | (kRoleMemIndex << 8));
    ix = -1;  // treated as an empty slot
  }
  float s = -INFINITY;
  if (ix >= 0) {
    const uint4* kr = reinterpret_cast<const uint4*>(mem_k + ((size_t)bh * M + ix) * D);
    float acc = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
      const uint4 x = __ldg(kr + c8);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(w[e] << 16), s_q[warp][8 * c8 + 2 * e], acc);
        acc = fmaf(__uint_as_float(w[e] & 0xffff0000u), s_q[warp][8 * c8 + 2 * e + 1], acc);
      }
    }
    s = acc * sl2;
  }
  float mx = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float e = (ix >= 0) ? exp2f(s - mx) : 0.f;
  float tot = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float p = tot > 0.f ? e / tot : 0.f;
  // o_mem over the slots, lanes split over d (D/32 columns each)
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = 0.f;
  for (int u = 0; u < km; ++u) {
    const int iu = __shfl_sync(0xffffffffu, ix, u);
    const float pu = __shfl_sync(0xffffffffu, p, u);
    if (iu < 0) continue;
    const __nv_bfloat16* vr = mem_v + ((size_t)bh * M + iu) * D + lane * PER;
    if constexpr (PER == 2) {
      const uint32_t x = __ldg(reinterpret_cast<const uint32_t*>(vr));
      acc[0] = fmaf(pu, __uint_as_float(x << 16), acc[0]);
      acc[1] = fmaf(pu, __uint_as_float(x & 0xffff0000u), acc[1]);
    } else {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(vr));
      acc[0] = fmaf(pu, __uint_as_float(x.x << 16), acc[0]);
      acc[1] = fmaf(pu, __uint_as_float(x.x & 0xffff0000u), acc[1]);
      acc[2] = fmaf(pu, __uint_as_float(x.y << 16), acc[2]);
      acc[3] = fmaf(pu, __uint_as_float(x.y & 0xffff0000u), acc[3]);
    }
  }
  // mix with the local row (read before the write: out may be local)
  const float g = __ldg(gate + h);
  const __nv_bfloat16* lr = local + row * D + lane * PER;
  __nv_bfloat16* orow = out + row * D + lane * PER;
  if constexpr (PER == 2) {
    const uint32_t x = *reinterpret_cast<const uint32_t*>(lr);
    const float l0 = __uint_as_float(x << 16), l1 = __uint_as_float(x & 0xffff0000u);
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(g * acc[0] + (1.f - g) * l0, g * acc[1] + (1.f - g) * l1);
  } else {
    const uint2 x = *reinterpret_cast<const uint2*>(lr);
    const float l0 = __uint_as_float(x.x << 16), l1 = __uint_as_float(x.x & 0xffff0000u);
    const float l2 = __uint_as_float(x.y << 16), l3 = __uint_as_float(x.y & 0xffff0000u);
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(g * acc[0] + (1.f - g) * l0, g * acc[1] + (1.f - g) * l1),
                                                 pack_bf16x2(g * acc[2] + (1.f - g) * l2, g * acc[3] + (1.f - g) * l3));
  }
}

}  // namespace memk

static lf_status mem_combine(const void* q, const void* local, const void* mem_k, const void* mem_v,
                             const int32_t* idx, const float* gate, void* out, int32_t B, int32_t H, int32_t n,
                             int32_t d, int32_t M, int32_t km, cudaStream_t stream) {
  t_msg[0] = 0;
  if (B < 0 || H < 1 || n < 0 || M < 0) {
    set_error("B, n, M must be >= 0 and H >= 1 (got %d, %d, %d, %d)", B, n, M, H);
    return LF_ERR_INVALID_ARG;
  }
  if (d != 64 && d != 128) {
    set_error("memory combine supports d = 64 or 128 (got %d)", d);
    return LF_ERR_UNSUPPORTED;
  }
  if (km < 1 || km > 32) {
    set_error("km (retrieved pairs per query) must be in [1, 32] (got %d)", km);
    return LF_ERR_UNSUPPORTED;
  }
  const int64_t rows = (int64_t)B * H * n;
  if (rows == 0) return LF_OK;
  const void* ptrs[7] = {q, local, mem_k, mem_v, idx, gate, out};
  const char* names[7] = {"q", "local", "mem_k", "mem_v", "idx", "gate", "out"};
  for (int t = 0; t < 7; ++t) {
    const bool may_be_null = (t == 2 || t == 3);  // no memory at all (M == 0)
    if (!ptrs[t] && !may_be_null) {
      set_error("%s must not be NULL", names[t]);
      return LF_ERR_INVALID_ARG;
    }
    const uintptr_t align = (t == 4 || t == 5) ? 3 : 15;  // idx, gate: 4 bytes; bf16 tensors: 16
    if (((uintptr_t)ptrs[t]) & align) {
      set_error("%s must be %d-byte aligned", names[t], (int)align + 1);
      return LF_ERR_INVALID_ARG;
    }
  }
  if (M > 0 && (!mem_k || !mem_v)) {
    set_error("mem_k and mem_v must not be NULL when M > 0");
    return LF_ERR_INVALID_ARG;
  }
  const size_t ob = (size_t)rows * d * 2;
  // out may be local itself, but must not overlap any other input
  if ((out != local && overlaps(out, ob, local, ob)) || overlaps(out, ob, q, ob) ||
      overlaps(out, ob, mem_k, (size_t)B * H * M * d * 2) || overlaps(out, ob, mem_v, (size_t)B * H * M * d * 2) ||
      overlaps(out, ob, idx, (size_t)rows * km * 4) || overlaps(out, ob, gate, (size_t)H * 4)) {
    set_error("out overlaps an input other than local");
    return LF_ERR_INVALID_ARG;
  }
  if (injected_fault("launch")) {
    set_error("memory combine launch: injected failure (LF_FAULT=launch)");
    return LF_ERR_CUDA;
  }
  cudaGetLastError();
  const int64_t blocks = (rows + memk::kWarps - 1) / memk::kWarps;
  if (blocks >= ((int64_t)1 << 31)) {
    set_error("memory combine too large");
    return LF_ERR_UNSUPPORTED;
  }
  const float sl2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  using bf = __nv_bfloat16;
  if (d == 64)
    memk::mem_combine_kernel<64><<<(unsigned)blocks, memk::kWarps * 32, 0, stream>>>(
        (const bf*)q, (const bf*)local, (const bf*)mem_k, (const bf*)mem_v, idx, gate, (bf*)out, H, n, M, km, rows, sl2);
  else
    memk::mem_combine_kernel<128><<<(unsigned)blocks, memk::kWarps * 32, 0, stream>>>(
        (const bf*)q, (const bf*)local, (const bf*)mem_k, (const bf*)mem_v, idx, gate, (bf*)out, H, n, M, km, rows, sl2);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("memory combine launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

}  // namespace lf

extern "C" {

lf_status lf_mem_combine(const void* q, const void* local, const void* mem_k, const void* mem_v,
                         const int32_t* idx, const float* gate, void* out, int32_t B, int32_t H, int32_t n,
                         int32_t d, int32_t M, int32_t km, cudaStream_t stream) {
  return lf::mem_combine(q, local, mem_k, mem_v, idx, gate, out, B, H, n, d, M, km, stream);
}

}  // extern "C"
