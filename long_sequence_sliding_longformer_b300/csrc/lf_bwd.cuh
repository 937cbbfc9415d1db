// lf_bwd.cuh -- host side of the backward (lf_attn_bwd, lf_attn_bwd_f32):
// validation, scratch for the per-row statistics, and the launches of the
// row and key passes of band_bwd.cuh, in blocks of at most kMaxBatch batch
// rows and kMaxHeadsSimt heads.  Included at the end of lf_attn.cu (same
// translation unit: it uses that file's validation and error helpers).
#pragma once

#include "band_bwd.cuh"

namespace lf {

struct BwdOut {
  float *dq, *dk, *dv, *dqg, *dkg, *dvg;
  float* drb = nullptr;  // gradient of the relative position bias [H, w + 1], or nullptr
};

static lf_status validate_bwd(const Problem& P, const void* dout, const BwdOut& g, bool bf16) {
  lf_status st = validate_pattern(P);
  if (st != LF_OK) return st;
  if (bf16 && P.d != 64 && P.d != 128) {
    set_error("bf16 backward supports d = 64 or 128 (got %d)", P.d);
    return LF_ERR_UNSUPPORTED;
  }
  if (!bf16 && P.d > 128) {
    set_error("fp32 backward supports d <= 128 (got %d)", P.d);
    return LF_ERR_UNSUPPORTED;
  }
  if (P.n >= (1 << 28)) {
    set_error("n must be < 2^28 (got %d)", P.n);
    return LF_ERR_UNSUPPORTED;
  }
  const int64_t elems = (int64_t)P.B * P.H * P.n * P.d;
  if (elems == 0) return LF_OK;
  const bool G = P.G > 0;
  const void* in[7] = {P.q, P.k, P.v, dout, P.qg, P.kg, P.vg};
  const char* in_names[7] = {"q", "k", "v", "dout", "qg", "kg", "vg"};
  const void* out[6] = {g.dq, g.dk, g.dv, g.dqg, g.dkg, g.dvg};
  const char* out_names[6] = {"dq", "dk", "dv", "dqg", "dkg", "dvg"};
  const int nin = G ? 7 : 4, nout = G ? 6 : 3;
  for (int t = 0; t < nin; ++t) {
    if (!in[t]) {
      set_error("%s must not be NULL", in_names[t]);
      return LF_ERR_INVALID_ARG;
    }
    if (((uintptr_t)in[t]) & 15) {
      set_error("%s must be 16-byte aligned", in_names[t]);
      return LF_ERR_INVALID_ARG;
    }
  }
  for (int t = 0; t < nout; ++t) {
    if (!out[t]) {
      set_error("%s must not be NULL", out_names[t]);
      return LF_ERR_INVALID_ARG;
    }
    if (((uintptr_t)out[t]) & 15) {
      set_error("%s must be 16-byte aligned", out_names[t]);
      return LF_ERR_INVALID_ARG;
    }
  }
  // no gradient may overlap an input or another gradient
  const size_t ib = (size_t)elems * P.elem, igb = (size_t)P.B * P.H * P.G * P.d * P.elem;
  const size_t ob = (size_t)elems * sizeof(float), ogb = (size_t)P.B * P.H * P.G * P.d * sizeof(float);
  if (P.rb || g.drb) {
    const size_t tb = (size_t)P.H * (P.w + 1) * sizeof(float);
    if (!P.rb) {
      set_error("d_rel_bias needs rel_bias");
      return LF_ERR_INVALID_ARG;
    }
    if ((((uintptr_t)P.rb) & 3) || (((uintptr_t)g.drb) & 3)) {
      set_error("rel_bias and d_rel_bias must be 4-byte aligned");
      return LF_ERR_INVALID_ARG;
    }
    if (g.drb && P.w > bwdk::kMaxBiasW) {
      set_error("the bias gradient supports w <= %d (got %d)", bwdk::kMaxBiasW, P.w);
      return LF_ERR_UNSUPPORTED;
    }
    for (int a = 0; a < nout; ++a)
      if (overlaps(out[a], a == 3 ? ogb : ob, P.rb, tb) || overlaps(out[a], a == 3 ? ogb : ob, g.drb, tb)) {
        set_error("%s overlaps rel_bias or d_rel_bias", out_names[a]);
        return LF_ERR_INVALID_ARG;
      }
    for (int t = 0; t < nin; ++t)
      if (overlaps(g.drb, tb, in[t], t == 4 ? igb : ib)) {
        set_error("d_rel_bias overlaps %s", in_names[t]);
        return LF_ERR_INVALID_ARG;
      }
    if (overlaps(g.drb, tb, P.rb, tb)) {
      set_error("d_rel_bias overlaps rel_bias");
      return LF_ERR_INVALID_ARG;
    }
  }
  for (int a = 0; a < nout; ++a) {
    const size_t na = a == 3 ? ogb : ob;
    for (int t = 0; t < nin; ++t)
      if (overlaps(out[a], na, in[t], t == 4 ? igb : ib)) {
        set_error("%s overlaps %s", out_names[a], in_names[t]);
        return LF_ERR_INVALID_ARG;
      }
    for (int c = a + 1; c < nout; ++c)
      if (overlaps(out[a], na, out[c], c == 3 ? ogb : ob)) {
        set_error("%s overlaps %s", out_names[a], out_names[c]);
        return LF_ERR_INVALID_ARG;
      }
  }
  return LF_OK;
}

template <typename T, int D>
static lf_status launch_bwd(const bwdk::BwdParams& bp, const void* q, const void* k, const void* v,
                            const void* qg, const void* kg, const void* vg, const void* dout,
                            const BwdOut& g, float2* stats, cudaStream_t s) {
  if (injected_fault("launch")) {
    set_error("backward launch: injected failure (LF_FAULT=launch)");
    return LF_ERR_CUDA;
  }
  static std::atomic<uint64_t> rows_attr{0}, keys_attr{0};
  constexpr int rows_smem = bwdk::rows_smem_bytes<D>(), keys_smem = bwdk::keys_smem_bytes<D>();
  // the keys pass holds the bias gradient's per-step sums after its own arrays
  constexpr int keys_smem_max = keys_smem + (bwdk::kMaxBiasW + 1) * 4;
  const int keys_dyn = keys_smem + (bp.drb_part ? bp.rb_stride * 4 : 0);
  lf_status st = smem_attr_once((const void*)bwdk::bwd_rows_tiled<T, D>, rows_smem, rows_attr, "backward rows");
  if (st == LF_OK)
    st = smem_attr_once((const void*)bwdk::bwd_keys_tiled<T, D>, keys_smem_max, keys_attr, "backward keys");
  if (st != LF_OK) return st;
  const T *tq = (const T*)q, *tk = (const T*)k, *tv = (const T*)v;
  const T *tqg = (const T*)qg, *tkg = (const T*)kg, *tvg = (const T*)vg, *tdo = (const T*)dout;
  const unsigned tiles = (unsigned)((int64_t)bp.B * bp.tiles_b);
  const unsigned gblocks = (unsigned)((int64_t)bp.B * bp.H * bp.G);
  const unsigned kwarps = (unsigned)(((int64_t)bp.B * bp.H * bp.n + bwdk::kWarps - 1) / bwdk::kWarps);
  // statistics and dq, dqg; then dk, dv (band rows, then global columns' rows); then dkg, dvg
  int launched = 0;
  bwdk::bwd_rows_tiled<T, D><<<tiles, bwdk::kThreads, rows_smem, s>>>(bp, tq, tk, tv, tdo, g.dq, stats);
  ++launched;
  if (bp.G > 0) {
    bwdk::bwd_grows<T, D><<<gblocks, bwdk::kWarps * 32, 0, s>>>(bp, tqg, tkg, tvg, tdo, g.dqg, stats);
    ++launched;
  }
  bwdk::bwd_keys_tiled<T, D><<<tiles, bwdk::kThreads, keys_dyn, s>>>(bp, tq, tk, tv, tdo, g.dk, g.dv, stats);
  ++launched;
  if (bp.drb_part) {
    const dim3 rgrid((unsigned)((bp.rb_stride + 255) / 256), (unsigned)bp.H);
    bwdk::bwd_bias_reduce<<<rgrid, 256, 0, s>>>(bp, g.drb);
    ++launched;
  }
  if (bp.G > 0) {
    bwdk::bwd_gkeys<T, D><<<gblocks, bwdk::kWarps * 32, 0, s>>>(bp, tq, tk, tv, tdo, g.dk, g.dv, stats);
    bwdk::bwd_kgvg<T, D><<<kwarps, bwdk::kWarps * 32, 0, s>>>(bp, tqg, tkg, tvg, tdo, g.dkg, g.dvg, stats);
    launched += 2;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("backward launch: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  count_launch(launched);
  return LF_OK;
}

// The parameter block of the backward launches (~18 KB: kept off the stack;
// each launch copies it), one per host thread.
static bwdk::BwdParams* bwd_params() {
  static thread_local bwdk::BwdParams* bp = nullptr;
  if (!bp) bp = new (std::nothrow) bwdk::BwdParams;
  if (!bp) set_error("host allocation of the backward parameter block failed");
  return bp;
}

template <typename T>
static lf_status backward_t(const Problem& P, const void* dout, const BwdOut& g) {
  const int nbmax = std::min(P.B, kMaxBatch), nhmax = std::min(P.H, kMaxHeadsSimt);
  const size_t sbytes = (size_t)nbmax * nhmax * P.n * sizeof(float2);
  float2* stats = nullptr;
  cudaError_t e = injected_fault("alloc") ? cudaErrorMemoryAllocation
                                          : cudaMallocAsync((void**)&stats, sbytes, P.stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("scratch allocation of %zu bytes failed: %s", sbytes, cudaGetErrorString(e));
    return LF_ERR_NO_MEMORY;
  }
  bwdk::BwdParams* holder = bwd_params();
  lf_status st = holder ? LF_OK : LF_ERR_NO_MEMORY;
  if (st == LF_OK && g.drb) {
    // the bias gradient is summed into, launch block by launch block
    e = cudaMemsetAsync(g.drb, 0, (size_t)P.H * (P.w + 1) * sizeof(float), P.stream);
    if (e != cudaSuccess) {
      set_error("clearing d_rel_bias: %s", cudaGetErrorString(e));
      st = LF_ERR_CUDA;
    }
  }
  for (int b0 = 0; st == LF_OK && b0 < P.B; b0 += kMaxBatch) {
    for (int h0 = 0; st == LF_OK && h0 < P.H; h0 += kMaxHeadsSimt) {
      bwdk::BwdParams& bp = *holder;
      memset(&bp, 0, sizeof bp);
      bp.B = std::min(kMaxBatch, P.B - b0);
      bp.H = std::min(kMaxHeadsSimt, P.H - h0);
      bp.n = P.n;
      bp.d = P.d;
      bp.Htot = P.H;
      bp.b0 = b0;
      bp.h0 = h0;
      bp.causal = P.causal;
      bp.G = P.G;
      bp.rel_bias = P.rb;
      bp.rb_stride = P.w + 1;
      bp.rb_half = P.w / 2;
      bp.scale = (float)(1.0 / std::sqrt((double)P.d));
      bp.sl2 = (float)(1.4426950408889634 / std::sqrt((double)P.d));
      for (int b = 0; b < bp.B; ++b) bp.pad[b] = P.pad ? P.pad[b0 + b] : 0;
      for (int r = 0; r < P.G; ++r) bp.gidx[r] = P.gidx[r];
      // tiles of 64 class positions: per head, the classes r < n % delta hold
      // n / delta + 1 positions, the others n / delta
      int64_t off = 0;
      for (int h = 0; h < bp.H; ++h) {
        const int delta = P.dil[h0 + h];
        bp.dil[h] = delta;
        bp.half_h[h] = (int32_t)std::min<int64_t>(win_of(P, h0 + h) / 2, P.n);
        bp.head_tile_off[h] = (int32_t)off;
        const int64_t qn = P.n / delta, rem = P.n % delta;
        off += rem * ((qn + 1 + bwdk::kTR - 1) / bwdk::kTR) + (delta - rem) * ((qn + bwdk::kTR - 1) / bwdk::kTR);
      }
      bp.head_tile_off[bp.H] = (int32_t)off;
      if (off * bp.B > 0x7fffffff) {
        st = LF_ERR_UNSUPPORTED;
        set_error("too many backward tiles (%lld)", (long long)(off * bp.B));
        break;
      }
      bp.tiles_b = (int32_t)off;
      float* part = nullptr;  // the keys pass's per-tile sums of the bias gradient
      if (g.drb) {
        const size_t pb = (size_t)bp.B * bp.tiles_b * bp.rb_stride * sizeof(float);
        e = injected_fault("alloc") ? cudaErrorMemoryAllocation : cudaMallocAsync((void**)&part, pb, P.stream);
        if (e != cudaSuccess) {
          cudaGetLastError();
          set_error("scratch allocation of %zu bytes failed: %s", pb, cudaGetErrorString(e));
          st = LF_ERR_NO_MEMORY;
          break;
        }
        bp.drb_part = part;
      }
      if (P.elem == 2) {
        st = P.d == 64 ? launch_bwd<__nv_bfloat16, 64>(bp, P.q, P.k, P.v, P.qg, P.kg, P.vg, dout, g, stats, P.stream)
                       : launch_bwd<__nv_bfloat16, 128>(bp, P.q, P.k, P.v, P.qg, P.kg, P.vg, dout, g, stats, P.stream);
      } else if (P.d <= 32) {
        st = launch_bwd<float, 32>(bp, P.q, P.k, P.v, P.qg, P.kg, P.vg, dout, g, stats, P.stream);
      } else if (P.d <= 64) {
        st = launch_bwd<float, 64>(bp, P.q, P.k, P.v, P.qg, P.kg, P.vg, dout, g, stats, P.stream);
      } else {
        st = launch_bwd<float, 128>(bp, P.q, P.k, P.v, P.qg, P.kg, P.vg, dout, g, stats, P.stream);
      }
      if (part) {
        cudaError_t pe = cudaFreeAsync(part, P.stream);
        if (st == LF_OK && pe != cudaSuccess) {
          set_error("scratch free: %s", cudaGetErrorString(pe));
          st = LF_ERR_CUDA;
        }
      }
    }
  }
  cudaError_t fe = cudaFreeAsync(stats, P.stream);
  if (st == LF_OK && fe != cudaSuccess) {
    set_error("scratch free: %s", cudaGetErrorString(fe));
    st = LF_ERR_CUDA;
  }
  return st;
}

static lf_status backward(const Problem& P, const void* dout, const BwdOut& g, bool bf16) {
  t_msg[0] = 0;
  lf_status st = validate_bwd(P, dout, g, bf16);
  if (st != LF_OK) return st;
  if ((int64_t)P.B * P.H * P.n == 0) return LF_OK;
  cudaGetLastError();  // a stale error from someone else must not be reported as ours
  return bf16 ? backward_t<__nv_bfloat16>(P, dout, g) : backward_t<float>(P, dout, g);
}

}  // namespace lf

extern "C" {

lf_status lf_attn_bwd(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                      const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                      float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg, int32_t B,
                      int32_t H, int32_t n, int32_t d, int32_t w, const int32_t* dilation, int32_t causal,
                      const int32_t* pad_len, cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, w, dilation, causal,
                pad_len, stream, 2};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg}, true);
}

lf_status lf_attn_bwd_f32(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                          const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                          float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg, int32_t B,
                          int32_t H, int32_t n, int32_t d, int32_t w, const int32_t* dilation,
                          int32_t causal, const int32_t* pad_len, cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, w, dilation, causal,
                pad_len, stream, 4};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg}, false);
}

lf_status lf_attn_bwd_bias(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                           const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                           float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg, int32_t B,
                           int32_t H, int32_t n, int32_t d, int32_t w, const int32_t* dilation, int32_t causal,
                           const int32_t* pad_len, const float* rel_bias, float* d_rel_bias,
                           cudaStream_t stream) {
  lf_status st = lf::check_bias_table(rel_bias, B, H, n);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, w, dilation, causal,
                pad_len, stream, 2, nullptr, rel_bias};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg, d_rel_bias}, true);
}

lf_status lf_attn_bwd_bias_f32(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                               const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                               float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                               int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                               const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                               const float* rel_bias, float* d_rel_bias, cudaStream_t stream) {
  lf_status st = lf::check_bias_table(rel_bias, B, H, n);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, w, dilation, causal,
                pad_len, stream, 4, nullptr, rel_bias};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg, d_rel_bias}, false);
}

lf_status lf_attn_bwd_hw(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                         const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                         float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg, int32_t B,
                         int32_t H, int32_t n, int32_t d, const int32_t* w_heads, const int32_t* dilation,
                         int32_t causal, const int32_t* pad_len, cudaStream_t stream) {
  lf_status st = lf::check_heads_window(w_heads, H);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, 0, dilation, causal,
                pad_len, stream, 2, w_heads};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg}, true);
}

lf_status lf_attn_bwd_hw_f32(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                             const void* vg, const int32_t* global_idx, int32_t n_global, const void* dout,
                             float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                             int32_t B, int32_t H, int32_t n, int32_t d, const int32_t* w_heads,
                             const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                             cudaStream_t stream) {
  lf_status st = lf::check_heads_window(w_heads, H);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, nullptr, B, H, n, d, 0, dilation, causal,
                pad_len, stream, 4, w_heads};
  return lf::backward(P, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg}, false);
}

}  // extern "C"
