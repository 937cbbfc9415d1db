// lf_varglobal.cuh -- global tokens that differ between batch rows (the
// question tokens of a QA example differ per example: "Global Attention" in
// section 3-1).  lf_attn_fwd_varglobal / lf_attn_bwd_varglobal run the
// forward or backward of each batch row with that row's own global list,
// in order on the caller's stream.  Included at the end of lf_attn.cu (it
// uses that file's Problem, validation and entry points).
#pragma once

namespace lf {

// Validates the per-row lists: offsets[0] = 0, non-decreasing, each row's
// list a valid global list (checked by the row's own validation below).
static lf_status check_offsets(const int32_t* offsets, int32_t B) {
  if (B > 0 && !offsets) {
    set_error("global_offsets must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  if (B > 0 && offsets[0] != 0) {
    set_error("global_offsets[0] must be 0 (got %d)", offsets[0]);
    return LF_ERR_INVALID_ARG;
  }
  for (int b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) {
      set_error("global_offsets must be non-decreasing (row %d)", b);
      return LF_ERR_INVALID_ARG;
    }
  return LF_OK;
}

// The Problem of batch row b (pointers offset into the tensors; qg packed).
static Problem row_problem(const Problem& P, const int32_t* offsets, int b) {
  Problem R = P;
  const size_t e = (size_t)P.elem;
  const size_t plane = (size_t)P.H * P.n * P.d * e;
  auto off = [&](const void* p, size_t bytes) -> const void* {
    return p ? static_cast<const uint8_t*>(p) + bytes : nullptr;
  };
  const int G = offsets[b + 1] - offsets[b];
  R.q = off(P.q, b * plane);
  R.k = off(P.k, b * plane);
  R.v = off(P.v, b * plane);
  R.kg = G ? off(P.kg, b * plane) : nullptr;
  R.vg = G ? off(P.vg, b * plane) : nullptr;
  R.qg = G ? off(P.qg, (size_t)offsets[b] * P.H * P.d * e) : nullptr;
  R.gidx = (G && P.gidx) ? P.gidx + offsets[b] : nullptr;
  R.G = G;
  R.out = P.out ? static_cast<uint8_t*>(P.out) + b * plane : nullptr;
  R.B = 1;
  R.pad = P.pad ? P.pad + b : nullptr;
  return R;
}

static lf_status forward_varglobal(const Problem& P, const int32_t* offsets, bool bf16) {
  t_msg[0] = 0;
  lf_status st = check_offsets(offsets, P.B);
  if (st != LF_OK) return st;
  // every row is checked before anything is enqueued
  for (int b = 0; b < P.B && st == LF_OK; ++b) st = validate(row_problem(P, offsets, b), bf16);
  if (st != LF_OK) return st;
  for (int b = 0; b < P.B && st == LF_OK; ++b) st = forward(row_problem(P, offsets, b), bf16);
  return st;
}

static lf_status backward_varglobal(const Problem& P, const int32_t* offsets, const void* dout, const BwdOut& g,
                                    bool bf16) {
  t_msg[0] = 0;
  lf_status st = check_offsets(offsets, P.B);
  if (st != LF_OK) return st;
  const size_t e = (size_t)P.elem, plane = (size_t)P.H * P.n * P.d;
  auto row_out = [&](int b) {
    const int G = offsets[b + 1] - offsets[b];
    BwdOut r;
    r.dq = g.dq + b * plane;
    r.dk = g.dk + b * plane;
    r.dv = g.dv + b * plane;
    r.dqg = G ? g.dqg + (size_t)offsets[b] * P.H * P.d : nullptr;
    r.dkg = G ? g.dkg + b * plane : nullptr;
    r.dvg = G ? g.dvg + b * plane : nullptr;
    return r;
  };
  auto row_dout = [&](int b) { return static_cast<const void*>(static_cast<const uint8_t*>(dout) + b * plane * e); };
  if (P.B > 0 && (!g.dq || !g.dk || !g.dv || !dout)) {
    set_error("dout, dq, dk and dv must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  for (int b = 0; b < P.B && st == LF_OK; ++b) st = validate_bwd(row_problem(P, offsets, b), row_dout(b), row_out(b), bf16);
  if (st != LF_OK) return st;
  for (int b = 0; b < P.B && st == LF_OK; ++b) {
    st = backward(row_problem(P, offsets, b), row_dout(b), row_out(b), bf16);
    // a row without global tokens has no global rows: its dkg, dvg are zeros
    if (st == LF_OK && offsets[b + 1] == offsets[b] && g.dkg && g.dvg) {
      cudaError_t e1 = cudaMemsetAsync(g.dkg + b * plane, 0, plane * sizeof(float), P.stream);
      cudaError_t e2 = cudaMemsetAsync(g.dvg + b * plane, 0, plane * sizeof(float), P.stream);
      if (e1 != cudaSuccess || e2 != cudaSuccess) {
        set_error("clearing dkg/dvg: %s", cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
        st = LF_ERR_CUDA;
      }
    }
  }
  return st;
}

}  // namespace lf

extern "C" {

lf_status lf_attn_fwd_varglobal(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                                const void* vg, const int32_t* global_offsets, const int32_t* global_idx,
                                void* out, int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                                const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                                cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, 0, out, B, H, n, d, w, dilation, causal, pad_len, stream, 2};
  return lf::forward_varglobal(P, global_offsets, true);
}

lf_status lf_attn_bwd_varglobal(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                                const void* vg, const int32_t* global_offsets, const int32_t* global_idx,
                                const void* dout, float* dq, float* dk, float* dv, float* dqg, float* dkg,
                                float* dvg, int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                                const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                                cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, 0, nullptr, B, H, n, d, w, dilation, causal, pad_len, stream, 2};
  return lf::backward_varglobal(P, global_offsets, dout, lf::BwdOut{dq, dk, dv, dqg, dkg, dvg}, true);
}

}  // extern "C"
