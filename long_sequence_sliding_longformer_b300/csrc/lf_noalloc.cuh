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
// the partial kernel writes every entry the merge kernel later reads, so
// nothing needs clearing.  Two calls whose kernels overlap on the GPU (for
// example on two streams at once) race on the array.
//
// Included at the end of lf_attn.cu (the library's single translation unit).
#pragma once

#include <mutex>

namespace lf {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

static std::mutex g_static_scratch_mu;
static float* g_static_scratch_addr[kMaxDevicesNoAlloc] = {};

// Device address of g_static_scratch on the current device (looked up once).
static lf_status static_scratch_for_current_device(float** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) {
    set_error("device %d is beyond the %d devices the no-alloc entry point tracks", dev,
              kMaxDevicesNoAlloc);
    return LF_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      set_error("cudaGetSymbolAddress(static scratch) on device %d: %s", dev, cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
    g_static_scratch_addr[dev] = static_cast<float*>(p);
  }
  *addr = g_static_scratch_addr[dev];
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
    return (size_t)(bh * ((P.n + c - 1) / c) * P.G * (P.d + 2)) * sizeof(float);
  };
  while (bytes(chunk) > kStaticScratchBytes && chunk < P.n) chunk *= 2;
  if (chunk > P.n) chunk = P.n;
  return bytes(chunk) <= kStaticScratchBytes ? chunk : 0;
}

// The band launches of run_band_bf16, planned without heap memory: the
// (head, residue) segments are generated in order straight into a parameter
// block on the stack, one launch per kMaxSeg segments or kMaxSets map sets.
static lf_status run_band_bf16_fixed(const Problem& P, int b0, int nbat) {
  const int grid_cap = sm_count();
  const size_t off = (size_t)b0 * P.H * P.n * P.d;
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(P.q) + off;
  const __nv_bfloat16* k = reinterpret_cast<const __nv_bfloat16*>(P.k) + off;
  const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(P.v) + off;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(P.out) + off;
  const int64_t planes = (int64_t)nbat * P.H;
  const int64_t half = std::min<int64_t>(P.w / 2, P.n);
  BandParams p;
  int h = 0, r = 0;  // next segment to place
  while (h < P.H) {
    memset(&p, 0, sizeof p);
    int nsets = 0, nseg = 0, items_per_b = 0;
    int set_delta[kMaxSets], set_r[kMaxSets];
    while (h < P.H && nseg < kMaxSeg) {
      const int delta = P.dil[h];
      if (r >= delta || r >= P.n) {
        ++h;
        r = 0;
        continue;
      }
      int set = -1;
      for (int t = 0; t < nsets; ++t)
        if (set_delta[t] == delta && set_r[t] == r) set = t;
      if (set < 0) {
        if (nsets == kMaxSets) break;
        set = nsets++;
        set_delta[set] = delta;
        set_r[set] = r;
      }
      const int n_r = (P.n - r + delta - 1) / delta;
      BandSeg& bs = p.seg[nseg++];
      bs.h = h;
      bs.r = r;
      bs.delta = delta;
      bs.n_r = n_r;
      bs.tiles = (n_r + 127) / 128;
      bs.set = set;
      bs.begin = items_per_b;
      items_per_b += bs.tiles;
      ++r;
    }
    if (nseg == 0) break;
    for (int t = 0; t < nsets; ++t) {
      const int delta = set_delta[t], rr = set_r[t];
      const int64_t n_r = (P.n - rr + delta - 1) / delta;
      const int64_t rs = (int64_t)delta * P.d, ps = (int64_t)P.n * P.d;
      const size_t ro = (size_t)rr * P.d;
      lf_status st;
      if ((st = make_map(&p.tq[t], q + ro, P.d, n_r, planes, rs, ps)) != LF_OK) return st;
      if ((st = make_map(&p.tk[t], k + ro, P.d, n_r, planes, rs, ps)) != LF_OK) return st;
      if ((st = make_map(&p.tv[t], v + ro, P.d, n_r, planes, rs, ps)) != LF_OK) return st;
    }
    p.k = k;
    p.v = v;
    p.out = out;
    p.B = nbat;
    p.H = P.H;
    p.n = P.n;
    p.half = (int32_t)half;
    p.right = P.causal ? 0 : (int32_t)half;
    p.causal = P.causal;
    p.G = P.G;
    p.nseg = nseg;
    p.items_per_b = items_per_b;
    const int64_t total = (int64_t)items_per_b * nbat;
    if (total > 0x7fffffff) {
      set_error("too many band tiles (%lld)", (long long)total);
      return LF_ERR_UNSUPPORTED;
    }
    p.total_items = (int32_t)total;
    p.sl2 = (float)(1.4426950408889634 / std::sqrt((double)P.d));
    for (int b = 0; b < nbat; ++b) p.pad[b] = P.pad ? P.pad[b0 + b] : 0;
    for (int g = 0; g < P.G; ++g) p.gidx[g] = P.gidx[g];
    const int grid = (int)std::min<int64_t>(total, grid_cap);
    if (grid > 0) {
      lf_status st = launch_band_tc(p, P.d, grid, P.stream);
      if (st != LF_OK) return st;
    }
  }
  return LF_OK;
}

static lf_status forward_noalloc(const Problem& P) {
  t_msg[0] = 0;
  lf_status st = validate(P, true);
  if (st != LF_OK) return st;
  if ((int64_t)P.B * P.H * P.n == 0) return LF_OK;
  // size check before anything touches the device
  if (P.G > 0) {
    for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
      const int nb = std::min(kMaxBatch, P.B - b0);
      if (static_scratch_chunk(P, nb) == 0) {
        const size_t need = (size_t)nb * P.H * P.G * (P.d + 2) * sizeof(float);
        set_error("global rows need at least %zu bytes of scratch (B*H*n_global*(d+2) floats); "
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
  if (P.G > 0 && (st = static_scratch_for_current_device(&ws)) != LF_OK) return st;
  cudaGetLastError();
  if (t_band_start) {
    cudaError_t e = cudaEventRecord(t_band_start, P.stream);
    if (e != cudaSuccess) {
      set_error("cudaEventRecord: %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
  }
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    if ((st = run_band_bf16_fixed(P, b0, nb)) != LF_OK) return st;
  }
  if (t_band_stop) {
    cudaError_t e = cudaEventRecord(t_band_stop, P.stream);
    if (e != cudaSuccess) {
      set_error("cudaEventRecord: %s", cudaGetErrorString(e));
      return LF_ERR_CUDA;
    }
  }
  if (P.G == 0) return LF_OK;
  // batch chunks run one after another on the stream, so they can share the array
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    PatternParams pp;  // on the stack: no heap use on this path
    fill_pattern(pp, P, b0, nb);
    const int64_t chunk = static_scratch_chunk(P, nb);
    const int nchunks = (int)((P.n + chunk - 1) / chunk);
    const size_t off = (size_t)b0 * P.H * P.n * P.d;
    const size_t goff = (size_t)b0 * P.H * P.G * P.d;
    st = launch_global_rows<__nv_bfloat16>(
        pp, reinterpret_cast<const __nv_bfloat16*>(P.qg) + goff,
        reinterpret_cast<const __nv_bfloat16*>(P.kg) + off,
        reinterpret_cast<const __nv_bfloat16*>(P.vg) + off,
        reinterpret_cast<__nv_bfloat16*>(P.out) + off, ws, nchunks, (int)chunk, P.stream);
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
