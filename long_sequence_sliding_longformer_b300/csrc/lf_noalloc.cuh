// lf_noalloc.cuh -- lf_attn_fwd_noalloc: the bf16 forward without any device
// allocation.
//
// lf_attn_fwd takes the scratch space of the global-row kernels (one partial
// softmax state per key chunk) from cudaMallocAsync on every call.  Some
// callers cannot allocate device memory while they run: an engine that
// reserves its whole memory budget up front and forbids allocations after
// start-up, code that must not risk an out-of-memory failure or allocator
// latency in the middle of a step, or a host application that owns the CUDA
// allocator and does not let plug-ins call it.  For them this entry point
// places that scratch in one fixed array in device global memory that is
// part of the library itself.
//
// The array is kStaticScratchBytes (16 MiB).  Every GPU on which the library
// is loaded holds it until the process exits.  Its device address is looked
// up once per device, on the first call made with that device current.
// All calls share the array and it keeps whatever the last call left there;
// the partial kernel writes every partial state the merge later reads, and
// the merge counters are cleared by each call.  Two calls whose kernels overlap on the GPU (for
// example on two streams at once) race on the array.
//
// Included at the end of lf_attn.cu (the library's single translation unit).
#pragma once


namespace lf {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;

static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

// Device address of g_static_scratch on the current device, looked up on
// every call rather than cached, so that it stays right after the device's
// context is torn down and rebuilt (cudaDeviceReset) between calls.
static lf_status static_scratch_for_current_device(float** addr) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    set_error("cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  *addr = static_cast<float*>(p);
  return LF_OK;
}

// Key-chunk length for the global rows of batch rows [b0, b0 + nbat): the same
// occupancy rule as the allocating path, then longer chunks until the partial
// states fit in the static array.  Returns 0 if even one chunk per row does not.
static int64_t static_scratch_chunk(const Problem& P, int nbat) {
  const int64_t bh = (int64_t)nbat * P.H;
  const int64_t qblocks = (P.G + kGQ - 1) / kGQ;
  int64_t chunk = 128;
  while (chunk * 2 <= P.n && bh * qblocks * ((P.n + chunk * 2 - 1) / (chunk * 2)) >= 4 * sm_count())
    chunk *= 2;
  auto bytes = [&](int64_t c) {
    return (size_t)(bh * ((P.n + c - 1) / c) * P.G * (P.d + 2)) * sizeof(float) +
           global_counters(bh, P.G) * sizeof(unsigned);
  };
  while (bytes(chunk) > kStaticScratchBytes && chunk < P.n) chunk *= 2;
  if (chunk > P.n) chunk = P.n;
  return bytes(chunk) <= kStaticScratchBytes ? chunk : 0;
}

static lf_status forward_noalloc(const Problem& P) {
  t_msg[0] = 0;
  lf_status st = validate(P, true);
  if (st != LF_OK) return st;
  if ((int64_t)P.B * P.H * P.n == 0) return LF_OK;
  // rows of many global tokens run on the band kernel and need no scratch
  const bool g_band = P.G > 0 && global_rows_on_band_kernel(P, true);
  // size check before anything touches the device
  if (P.G > 0 && !g_band) {
    for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
      const int nb = std::min(kMaxBatch, P.B - b0);
      if (static_scratch_chunk(P, nb) == 0) {
        const size_t need = (size_t)nb * P.H * P.G * ((P.d + 2) * sizeof(float) + sizeof(unsigned));
        set_error("global rows need at least %zu bytes of scratch (B*H*n_global*(d+2) floats and "
                  "B*H*n_global counters); "
                  "the static scratch holds %zu bytes",
                  need, kStaticScratchBytes);
        return LF_ERR_UNSUPPORTED;
      }
    }
  }
  if (!encode_fn()) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return LF_ERR_CUDA;
  }
  float* ws = nullptr;
  if (P.G > 0 && !g_band && (st = static_scratch_for_current_device(&ws)) != LF_OK) return st;
  cudaGetLastError();
  if (t_band_start && (st = record_timing(t_band_start, P.stream)) != LF_OK) return st;
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    BandParams bp;  // on the stack: no heap use on this path
    if ((st = run_band_bf16(P, b0, nb, bp)) != LF_OK) return st;
  }
  if (t_band_stop && (st = record_timing(t_band_stop, P.stream)) != LF_OK) return st;
  if (P.G == 0) return LF_OK;
  if (g_band) {
    for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
      BandParams bp;  // on the stack: no heap use on this path
      if ((st = run_global_band_bf16(P, b0, std::min(kMaxBatch, P.B - b0), bp, P.stream)) != LF_OK) return st;
    }
    return LF_OK;
  }
  // batch chunks run one after another on the stream, so they can share the array
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    PatternParams pp;  // on the stack: no heap use on this path
    fill_pattern(pp, P, b0, nb);
    const int64_t chunk = static_scratch_chunk(P, nb);
    const int nchunks = (int)((P.n + chunk - 1) / chunk);
    const size_t off = (size_t)b0 * P.H * P.n * P.d;
    const size_t goff = (size_t)b0 * P.H * P.G * P.d;
    // partial states, then the merge counters
    unsigned* counters = reinterpret_cast<unsigned*>(ws + (size_t)nb * P.H * nchunks * P.G * (P.d + 2));
    st = launch_global_rows<__nv_bfloat16>(
        pp, reinterpret_cast<const __nv_bfloat16*>(P.qg) + goff,
        reinterpret_cast<const __nv_bfloat16*>(P.kg) + off,
        reinterpret_cast<const __nv_bfloat16*>(P.vg) + off,
        reinterpret_cast<__nv_bfloat16*>(P.out) + off, ws, counters, nchunks, (int)chunk, P.stream);
    if (st != LF_OK) return st;
  }
  return LF_OK;
}

}  // namespace lf

extern "C" lf_status lf_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                         const void* qg, const void* kg, const void* vg,
                                         const int32_t* global_idx, int32_t n_global, void* out,
                                         int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                                         const int32_t* dilation, int32_t causal,
                                         const int32_t* pad_len, cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, w, dilation, causal,
                pad_len, stream, 2};
  return lf::forward_noalloc(P);
}
