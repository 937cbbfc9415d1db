// lf_proj.cuh -- host side of the per-head projections (lf_proj_heads):
// validation, tensor maps and the launch of proj_gemm.cuh's kernel.
// Included at the end of lf_attn.cu (same translation unit: it uses that
// file's tensor-map builder and error helpers).
#pragma once

#include "proj_gemm.cuh"

namespace lf {

template <int BN>
static lf_status launch_proj(projk::ProjParams& pp, cudaStream_t s) {
  using C = projk::Cfg<BN>;
  static std::atomic<uint64_t> attr_done{0};
  lf_status st = smem_attr_once((const void*)projk::proj_gemm_kernel<BN>, C::kSmem, attr_done, "projection");
  if (st != LF_OK) return st;
  if (injected_fault("launch")) {
    set_error("projection launch: injected failure (LF_FAULT=launch)");
    return LF_ERR_CUDA;
  }
  const int grid = std::min(pp.tiles, sm_count());
  projk::proj_gemm_kernel<BN><<<grid, projk::kThreads, C::kSmem, s>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("projection launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch();
  return LF_OK;
}

static lf_status proj_heads(const void* x, const void* w, const float* bias, void* y, int32_t B, int32_t n,
                            int32_t K, int32_t n_out, int32_t H, int32_t d, cudaStream_t stream) {
  t_msg[0] = 0;
  if (B < 0 || n < 0 || K < 1 || n_out < 1 || H < 1 || d < 1) {
    set_error("B, n must be >= 0 and K, n_out, H, d >= 1 (got %d, %d, %d, %d, %d, %d)", B, n, K, n_out, H, d);
    return LF_ERR_INVALID_ARG;
  }
  if (K % 64 != 0) {
    set_error("K must be a multiple of 64 (got %d)", K);
    return LF_ERR_UNSUPPORTED;
  }
  if (d % 32 != 0) {
    set_error("d must be a multiple of 32 (got %d)", d);
    return LF_ERR_UNSUPPORTED;
  }
  const int64_t N = (int64_t)n_out * H * d, M = (int64_t)B * n;
  if (N % 128 != 0) {
    set_error("n_out * H * d must be a multiple of 128 (got %lld)", (long long)N);
    return LF_ERR_UNSUPPORTED;
  }
  if (M >= (int64_t)1 << 31 || N >= (int64_t)1 << 31 || M * K >= ((int64_t)1 << 40) || N * K >= ((int64_t)1 << 40)) {
    set_error("projection too large");
    return LF_ERR_UNSUPPORTED;
  }
  if (M == 0) return LF_OK;
  const void* ptrs[3] = {x, w, y};
  const char* names[3] = {"x", "w", "y"};
  for (int t = 0; t < 3; ++t) {
    if (!ptrs[t]) {
      set_error("%s must not be NULL", names[t]);
      return LF_ERR_INVALID_ARG;
    }
    if (((uintptr_t)ptrs[t]) & 15) {
      set_error("%s must be 16-byte aligned", names[t]);
      return LF_ERR_INVALID_ARG;
    }
  }
  if (overlaps(y, (size_t)(N * M * 2), x, (size_t)(M * K * 2)) || overlaps(y, (size_t)(N * M * 2), w, (size_t)(N * K * 2))) {
    set_error("y overlaps an input");
    return LF_ERR_INVALID_ARG;
  }
  if (!encode_fn()) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return LF_ERR_CUDA;
  }
  cudaGetLastError();
  const int BN = (N % 256 == 0) ? 256 : 128;
  static thread_local projk::ProjParams pp;
  memset(&pp, 0, sizeof pp);
  lf_status st;
  if ((st = make_map(&pp.tx, x, K, M, 1, K, M * K, projk::kBM)) != LF_OK) return st;
  if ((st = make_map(&pp.tw, w, K, N, 1, K, N * K, BN)) != LF_OK) return st;
  pp.bias = bias;
  pp.y = reinterpret_cast<__nv_bfloat16*>(y);
  pp.M = (int32_t)M;
  pp.N = (int32_t)N;
  pp.K = K;
  pp.B = B;
  pp.n = n;
  pp.H = H;
  pp.d = d;
  pp.tiles_n = (int32_t)(N / BN);
  const int64_t tiles = ((M + projk::kBM - 1) / projk::kBM) * pp.tiles_n;
  if (tiles >= ((int64_t)1 << 31)) {
    set_error("projection too large");
    return LF_ERR_UNSUPPORTED;
  }
  pp.tiles = (int32_t)tiles;
  return BN == 256 ? launch_proj<256>(pp, stream) : launch_proj<128>(pp, stream);
}

}  // namespace lf

extern "C" {

lf_status lf_proj_heads(const void* x, const void* w, const float* bias, void* y, int32_t B, int32_t n,
                        int32_t K, int32_t n_out, int32_t H, int32_t d, cudaStream_t stream) {
  return lf::proj_heads(x, w, bias, y, B, n, K, n_out, H, d, stream);
}

}  // extern "C"
