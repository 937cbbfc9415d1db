// lf_attn.cu -- the C ABI of include/lf_attn.h: argument validation, planning
// of the band-kernel work (residue classes, tiles, TMA tensor maps), the
// global-row scratch space, and the launches.  Single translation unit: the
// kernels are included below.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "lf_internal.cuh"
#include "band_ring.cuh"
#include "band_duo.cuh"
#include "band_pair.cuh"
#include "band_simt.cuh"
#include "global_rows.cuh"

namespace lf {

// ------------------------------------------------------------------ band kernel choice
// D = 64 has two tensor-core band kernels: the ring kernel (one 128-row tile
// per CTA, two CTAs per SM, 64-key entries; also the global-row mode) and the
// duo kernel (two 128-row tiles per item sharing 96-key loads, one CTA per
// SM).  D = 128 runs the pair kernel (two tiles per CTA sharing 128-key
// entries, one CTA per SM).
enum class BandKernel { ring, duo, pair };


static thread_local const char* t_band_kernel = "";

// Host-side fault injection for tests: with the environment variable
// LF_FAULT set to "alloc" (or "launch") a call reports that its scratch
// allocation (or its first kernel launch) failed, at that point, before
// anything of the call has run on the device.
static bool injected_fault(const char* what) {
  const char* f = std::getenv("LF_FAULT");
  return f && std::strcmp(f, what) == 0;
}

lf_status launch_band_tc(const BandParams& p, int d, int grid, cudaStream_t s) {
  if (injected_fault("launch")) {
    set_error("band kernel launch: injected failure (LF_FAULT=launch)");
    return LF_ERR_CUDA;
  }
  if (d == 64 && (p.gmode || !p.pair_kernel)) {
    if (!p.gmode) t_band_kernel = "band_ring";
    return ringk::launch(p, grid, s);
  }
  if (d == 64) {
    t_band_kernel = "band_duo";
    return duok::launch(p, grid, s);
  }
  if (d == 128) {
    t_band_kernel = "band_pair";
    return pairk::launch(p, grid, s);
  }
  set_error("band kernel: unsupported head dimension %d", d);
  return LF_ERR_UNSUPPORTED;
}

static thread_local char t_msg[512] = "";
static thread_local cudaEvent_t t_band_start = nullptr, t_band_stop = nullptr;
static std::atomic<uint64_t> g_launches{0};

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
}

void count_launch(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

// ------------------------------------------------------------------ driver entry point for TMA maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [d, rows, planes] bf16 view with row stride `row_stride` elements, plane
// stride `plane_stride` elements; boxes of [64, box_rows, 1] with 128-byte swizzle.
static lf_status make_map(CUtensorMap* m, const void* base, int d, int64_t rows, int64_t planes,
                          int64_t row_stride, int64_t plane_stride, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return LF_ERR_CUDA;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)plane_stride * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for rows=%lld planes=%lld stride=%lld", (int)r,
              (long long)rows, (long long)planes, (long long)row_stride);
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// ------------------------------------------------------------------ problem + validation
struct Problem {
  const void *q, *k, *v, *qg, *kg, *vg;
  const int32_t* gidx;
  int32_t G;
  void* out;
  int32_t B, H, n, d, w;
  const int32_t* dil;
  int32_t causal;
  const int32_t* pad;
  cudaStream_t stream;
  int elem;  // bytes per element
  const int32_t* wh = nullptr;  // window per head (host), or nullptr: w for every head
  const float* rb = nullptr;    // relative position bias [H, w + 1] (device), or nullptr
};

// the window of head h
static inline int32_t win_of(const Problem& P, int h) { return P.wh ? P.wh[h] : P.w; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

// Checks that need no pointers: sizes, window, dilation, padding, global list.
static lf_status validate_pattern(const Problem& P) {
  if (P.B < 0 || P.H < 0 || P.n < 0) {
    set_error("B, H and n must be >= 0 (got %d, %d, %d)", P.B, P.H, P.n);
    return LF_ERR_INVALID_ARG;
  }
  if (P.d < 1) {
    set_error("d must be >= 1 (got %d)", P.d);
    return LF_ERR_INVALID_ARG;
  }
  if (!P.wh && (P.w < 0 || (P.w & 1))) {
    set_error("w must be even and >= 0 (got %d)", P.w);
    return LF_ERR_INVALID_ARG;
  }
  if (P.wh)
    for (int h = 0; h < P.H; ++h)
      if (P.wh[h] < 0 || (P.wh[h] & 1)) {
        set_error("w_heads[%d] = %d must be even and >= 0", h, P.wh[h]);
        return LF_ERR_INVALID_ARG;
      }
  if (P.causal != 0 && P.causal != 1) {
    set_error("causal must be 0 or 1 (got %d)", P.causal);
    return LF_ERR_INVALID_ARG;
  }
  if (P.G < 0) {
    set_error("n_global must be >= 0 (got %d)", P.G);
    return LF_ERR_INVALID_ARG;
  }
  if (P.G > LF_MAX_GLOBAL) {
    set_error("n_global must be <= %d (got %d)", LF_MAX_GLOBAL, P.G);
    return LF_ERR_UNSUPPORTED;
  }
  if (P.H > 0 && !P.dil) {
    set_error("dilation must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  for (int h = 0; h < P.H; ++h)
    if (P.dil[h] < 1) {
      set_error("dilation[%d] = %d must be >= 1", h, P.dil[h]);
      return LF_ERR_INVALID_ARG;
    }
  if (P.pad)
    for (int b = 0; b < P.B; ++b)
      if (P.pad[b] < 0 || P.pad[b] > P.n) {
        set_error("pad_len[%d] = %d must be in [0, n=%d]", b, P.pad[b], P.n);
        return LF_ERR_INVALID_ARG;
      }
  if (P.G > 0) {
    if (!P.gidx) {
      set_error("global_idx must not be NULL when n_global > 0");
      return LF_ERR_INVALID_ARG;
    }
    for (int r = 0; r < P.G; ++r) {
      if (P.gidx[r] < 0 || P.gidx[r] >= P.n) {
        set_error("global_idx[%d] = %d is outside [0, n=%d)", r, P.gidx[r], P.n);
        return LF_ERR_INVALID_ARG;
      }
      if (r > 0 && P.gidx[r] <= P.gidx[r - 1]) {
        set_error("global_idx must be strictly increasing (entry %d)", r);
        return LF_ERR_INVALID_ARG;
      }
    }
  }
  return LF_OK;
}

static lf_status validate(const Problem& P, bool bf16) {
  lf_status st = validate_pattern(P);
  if (st != LF_OK) return st;
  if (bf16 && P.d != 64 && P.d != 128) {
    set_error("bf16 path supports d = 64 or 128 (got %d)", P.d);
    return LF_ERR_UNSUPPORTED;
  }
  if (!bf16 && P.d > 128) {
    set_error("fp32 path supports d <= 128 (got %d)", P.d);
    return LF_ERR_UNSUPPORTED;
  }
  if (!bf16 && P.H > kMaxHeadsSimt) {
    set_error("fp32 path supports H <= %d (got %d)", kMaxHeadsSimt, P.H);
    return LF_ERR_UNSUPPORTED;
  }
  if (P.n >= (1 << 28)) {
    set_error("n must be < 2^28 (got %d)", P.n);
    return LF_ERR_UNSUPPORTED;
  }
  const int64_t elems = (int64_t)P.B * P.H * P.n * P.d;
  if (elems == 0) return LF_OK;
  const void* ptrs[7] = {P.q, P.k, P.v, P.out, P.qg, P.kg, P.vg};
  const char* names[7] = {"q", "k", "v", "out", "qg", "kg", "vg"};
  const int need = P.G > 0 ? 7 : 4;
  for (int t = 0; t < need; ++t) {
    if (!ptrs[t]) {
      set_error("%s must not be NULL", names[t]);
      return LF_ERR_INVALID_ARG;
    }
    if (((uintptr_t)ptrs[t]) & 15) {
      set_error("%s must be 16-byte aligned", names[t]);
      return LF_ERR_INVALID_ARG;
    }
  }
  const size_t bytes = (size_t)elems * P.elem;
  const size_t gbytes = (size_t)P.B * P.H * P.G * P.d * P.elem;
  for (int t = 0; t < need; ++t) {
    if (t == 3) continue;
    if (overlaps(P.out, bytes, ptrs[t], t == 4 ? gbytes : bytes)) {
      set_error("out overlaps %s", names[t]);
      return LF_ERR_INVALID_ARG;
    }
  }
  if (P.rb) {
    if (((uintptr_t)P.rb) & 3) {
      set_error("rel_bias must be 4-byte aligned");
      return LF_ERR_INVALID_ARG;
    }
    if (P.out && overlaps(P.out, bytes, P.rb, (size_t)P.H * (P.w + 1) * sizeof(float))) {
      set_error("out overlaps rel_bias");
      return LF_ERR_INVALID_ARG;
    }
  }
  return LF_OK;
}

static void fill_pattern(PatternParams& pp, const Problem& P, int b0, int nb) {
  memset(&pp, 0, sizeof pp);
  pp.B = nb;
  pp.H = P.H;
  pp.n = P.n;
  pp.d = P.d;
  pp.causal = P.causal;
  pp.G = P.G;
  pp.scale = (float)(1.0 / std::sqrt((double)P.d));
  for (int b = 0; b < nb; ++b) pp.pad[b] = P.pad ? P.pad[b0 + b] : 0;
  for (int r = 0; r < P.G; ++r) pp.gidx[r] = P.gidx[r];
}

// ------------------------------------------------------------------ global rows
// Key-chunk length of the global-row pass for batch rows [b0, b0 + nbat):
// enough CTAs to fill the GPU about four times over, then longer chunks
// until the partial states stay within 64 MiB.
static int64_t global_chunk(const Problem& P, int nbat, size_t* ws_floats) {
  const int64_t bh = (int64_t)nbat * P.H;
  const int64_t qblocks = (P.G + kGQ - 1) / kGQ;
  int64_t chunk = 128;
  while (chunk * 2 <= P.n && bh * qblocks * ((P.n + chunk * 2 - 1) / (chunk * 2)) >= 4 * sm_count())
    chunk *= 2;
  auto floats = [&](int64_t c) { return (size_t)(bh * ((P.n + c - 1) / c) * P.G * (P.d + 2)); };
  while (floats(chunk) * sizeof(float) > ((size_t)64 << 20) && chunk < P.n) chunk *= 2;
  *ws_floats = floats(chunk);
  return chunk;
}

// A second stream (and fork/join events) per host thread and device, so the
// global-row partial pass can run beside the band kernel.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxAuxDevices = 16;
static thread_local AuxStream t_aux[kMaxAuxDevices];

static AuxStream* aux_stream() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxAuxDevices) return nullptr;
  AuxStream& a = t_aux[dev];
  if (a.s && a.fork && a.join) return &a;
  // Build all three or none: a half-built entry is destroyed, so that the
  // next call starts over instead of using it.
  bool ok = cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();  // clear the sticky-free error of the failed create
    if (a.join) cudaEventDestroy(a.join);
    if (a.fork) cudaEventDestroy(a.fork);
    if (a.s) cudaStreamDestroy(a.s);
    a = AuxStream{};
    return nullptr;
  }
  return &a;
}

// Enqueues the global-row pass (partials and the merge by their last CTAs)
// on stream `ps`.  Scratch: the partial states of every batch chunk, then
// their merge counters.
template <typename T>
static lf_status global_pass(const Problem& P, float* ws, cudaStream_t ps) {
  size_t off_ws = 0, total = 0;
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    size_t nf = 0;
    global_chunk(P, std::min(kMaxBatch, P.B - b0), &nf);
    total += nf;
  }
  unsigned* counters = reinterpret_cast<unsigned*>(ws + total);
  for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    size_t nf = 0;
    const int64_t chunk = global_chunk(P, nb, &nf);
    const int nchunks = (int)((P.n + chunk - 1) / chunk);
    PatternParams pp;
    fill_pattern(pp, P, b0, nb);
    const size_t off = (size_t)b0 * P.H * P.n * P.d;
    const size_t goff = (size_t)b0 * P.H * P.G * P.d;
    lf_status st = launch_global_rows<T>(pp, reinterpret_cast<const T*>(P.qg) + goff,
                                         reinterpret_cast<const T*>(P.kg) + off,
                                         reinterpret_cast<const T*>(P.vg) + off,
                                         reinterpret_cast<T*>(P.out) + off, ws + off_ws, counters,
                                         nchunks, (int)chunk, ps);
    if (st != LF_OK) return st;
    off_ws += nf;
    counters += global_counters((int64_t)nb * P.H, P.G);
  }
  return LF_OK;
}

// ------------------------------------------------------------------ global rows on the tensor cores
// With many global tokens (d = 64, G >= kGlobalBandMin) their rows run through
// the band kernel in its global-row mode: per (batch row, head) the query
// rows are the G global tokens (128 per work item, from qg), the keys and
// values are kg and vg over the row's valid length.  No scratch is needed.
constexpr int kGlobalBandMin = 16;

static bool global_rows_on_band_kernel(const Problem& P, bool bf16) {
  return bf16 && P.d == 64 && P.G >= kGlobalBandMin;
}

static lf_status run_global_band_bf16(const Problem& P, int b0, int nbat, BandParams& p,
                                      cudaStream_t s) {
  const int grid_cap = sm_count() * ringk::BandCfg<64>::kCtaPerSm;
  const size_t off = (size_t)b0 * P.H * P.n * P.d;
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(P.qg) + (size_t)b0 * P.H * P.G * P.d;
  const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(P.kg) + off;
  const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(P.vg) + off;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(P.out) + off;
  const int64_t planes = (int64_t)nbat * P.H;
  const int qtiles = (P.G + 127) / 128;
  for (int h0 = 0; h0 < P.H; h0 += kMaxSeg) {
    memset(&p, 0, sizeof p);
    const int nh = std::min(kMaxSeg, P.H - h0);
    for (int j = 0; j < nh; ++j) {
      BandSeg& bs = p.seg[j];
      bs.h = h0 + j;
      bs.r = 0;
      bs.delta = 1;
      bs.n_r = P.n;
      bs.items = qtiles;
      bs.set = 0;
      bs.begin = j * qtiles;
      bs.half = P.n;  // every key is in reach
    }
    lf_status st;
    const int ek = ringk::BandCfg<64>::kE;
    if ((st = make_map(&p.tq[0], qg, P.d, P.G, planes, P.d, (int64_t)P.G * P.d, 128)) != LF_OK) return st;
    if ((st = make_map(&p.tk[0], kg, P.d, P.n, planes, P.d, (int64_t)P.n * P.d, ek)) != LF_OK) return st;
    if ((st = make_map(&p.tv[0], vg, P.d, P.n, planes, P.d, (int64_t)P.n * P.d, ek)) != LF_OK) return st;
    p.k = kg;
    p.v = vg;
    p.out = out;
    p.B = nbat;
    p.H = P.H;
    p.n = P.n;
    p.half = P.n;  // every key is in reach
    p.right = P.n;
    p.causal = P.causal;
    p.G = 0;
    p.gmode = 1;
    p.nrow_g = P.G;
    p.nseg = nh;
    p.items_per_b = nh * qtiles;  // this launch's heads only
    const int64_t total = (int64_t)p.items_per_b * nbat;
    if (total > 0x7fffffff) {
      set_error("too many global-row work items (%lld)", (long long)total);
      return LF_ERR_UNSUPPORTED;
    }
    p.total_items = (int32_t)total;
    p.sl2 = (float)(1.4426950408889634 / std::sqrt((double)P.d));
    for (int b = 0; b < nbat; ++b) p.pad[b] = P.pad ? P.pad[b0 + b] : 0;
    for (int g = 0; g < P.G; ++g) p.gidx[g] = P.gidx[g];
    const int grid = (int)std::min<int64_t>(total, grid_cap);
    if (grid > 0 && (st = launch_band_tc(p, P.d, grid, s)) != LF_OK) return st;
  }
  return LF_OK;
}

// ------------------------------------------------------------------ bf16 band planning
// Every (head, residue) class with at least one row is a segment; its work
// items are its 128-row tiles (D = 64) or pairs of them (D = 128).  Segments are generated in order straight
// into the parameter block `p` (no heap use), one launch per kMaxSeg segments
// or kMaxSets (dilation, residue) tensor-map sets.
// For D = 64 the choice is measured (whole calls, one B300, L2 flushed,
// both kernels reading V as loaded): with 16 or more global tokens and a
// two-sided window the duo kernel is 8-13% faster (it gathers the global key
// columns once per 256 rows instead of once per 128); with fewer global
// tokens the two are within 4% of each other and the ring kernel is taken;
// with a one-sided (causal) window the ring kernel is 21-28% faster.
static BandKernel band_kernel_for(const Problem& P) {
  if (P.d == 128) return BandKernel::pair;
  // the relative position bias is built into the ring kernel only (d = 64),
  // and so are windows that differ between heads
  bool one_window = true;
  for (int h = 1; P.wh && h < P.H; ++h) one_window = one_window && P.wh[h] == P.wh[0];
  return (P.G >= 16 && !P.causal && !P.rb && one_window) ? BandKernel::duo : BandKernel::ring;
}

// Every head's segments, each carrying its head's window reach (heads may
// differ), a launch per kMaxSeg segments or kMaxSets (dilation, residue)
// tensor-map sets.
static lf_status run_band_bf16(const Problem& P, int b0, int nbat, BandParams& p) {
  const BandKernel kind = band_kernel_for(P);
  // persistent CTAs: two per SM for the ring kernel, one for the others
  const int grid_cap = sm_count() * (kind == BandKernel::ring ? ringk::BandCfg<64>::kCtaPerSm : 1);
  // The duo kernel pairs tiles when every head's window reach is a multiple
  // of 16 keys (the tiles' key ranges then meet on 16-key steps); the pair
  // kernel always pairs, the ring kernel never.
  bool reach16 = true, varwin = false;
  for (int h = 0; h < P.H; ++h) {
    varwin = varwin || win_of(P, h) != win_of(P, 0);
    const int64_t half_h = std::min<int64_t>(win_of(P, h) / 2, P.n), right_h = P.causal ? 0 : half_h;
    reach16 = reach16 && half_h % 16 == 0 && right_h % 16 == 0;
  }
  const int pair = kind == BandKernel::pair || (kind == BandKernel::duo && reach16);
  const int rows_per_item = pair ? 256 : 128;
  // keys per K/V load
  const int ek = kind == BandKernel::ring ? ringk::BandCfg<64>::kE : kind == BandKernel::duo ? duok::kLK : 128;
  const size_t off = (size_t)b0 * P.H * P.n * P.d;
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(P.q) + off;
  const __nv_bfloat16* k = reinterpret_cast<const __nv_bfloat16*>(P.k) + off;
  const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(P.v) + off;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(P.out) + off;
  const int64_t planes = (int64_t)nbat * P.H;
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
      bs.items = (n_r + rows_per_item - 1) / rows_per_item;
      bs.set = set;
      bs.begin = items_per_b;
      bs.half = (int32_t)std::min<int64_t>(win_of(P, h) / 2, P.n);
      items_per_b += bs.items;
      ++r;
    }
    if (nseg == 0) break;
    for (int t = 0; t < nsets; ++t) {
      const int delta = set_delta[t], rr = set_r[t];
      const int64_t n_r = (P.n - rr + delta - 1) / delta;
      const int64_t rs = (int64_t)delta * P.d, ps = (int64_t)P.n * P.d;
      const size_t ro = (size_t)rr * P.d;
      lf_status st;
      if ((st = make_map(&p.tq[t], q + ro, P.d, n_r, planes, rs, ps, 128)) != LF_OK) return st;
      if ((st = make_map(&p.tk[t], k + ro, P.d, n_r, planes, rs, ps, ek)) != LF_OK) return st;
      if ((st = make_map(&p.tv[t], v + ro, P.d, n_r, planes, rs, ps, ek)) != LF_OK) return st;
    }
    p.k = k;
    p.v = v;
    p.out = out;
    p.B = nbat;
    p.H = P.H;
    p.n = P.n;
    p.causal = P.causal;
    p.G = P.G;
    p.half = P.H > 0 ? (int32_t)std::min<int64_t>(win_of(P, 0) / 2, P.n) : 0;
    p.right = P.causal ? 0 : p.half;
    p.varwin = varwin;
    p.pair = pair;
    p.pair_kernel = kind != BandKernel::ring;
    p.rel_bias = P.rb;
    p.rb_stride = P.w + 1;
    p.rb_half = P.w / 2;
    p.nseg = nseg;
    p.items_per_b = items_per_b;
    const int64_t total = (int64_t)items_per_b * nbat;
    if (total > 0x7fffffff) {
      set_error("too many band work items (%lld)", (long long)total);
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

static lf_status run_band_f32(const Problem& P, int b0, int nbat) {
  static thread_local SimtParams* sp = nullptr;  // ~18 KB: keep it off the stack
  if (!sp) sp = new (std::nothrow) SimtParams;
  if (!sp) {
    set_error("host allocation of the fp32 parameter block failed");
    return LF_ERR_NO_MEMORY;
  }
  const size_t off = (size_t)b0 * P.H * P.n * P.d;
  fill_pattern(sp->pat, P, b0, nbat);
  for (int h = 0; h < P.H; ++h) {
    sp->dil[h] = P.dil[h];
    sp->half_h[h] = (int32_t)std::min<int64_t>(win_of(P, h) / 2, P.n);
  }
  sp->rel_bias = P.rb;
  sp->rb_stride = P.w + 1;
  sp->rb_half = P.w / 2;
  if (injected_fault("launch")) {
    set_error("band kernel launch: injected failure (LF_FAULT=launch)");
    return LF_ERR_CUDA;
  }
  t_band_kernel = "band_simt_f32";
  return launch_band_simt_f32(*sp, reinterpret_cast<const float*>(P.q) + off,
                              reinterpret_cast<const float*>(P.k) + off,
                              reinterpret_cast<const float*>(P.v) + off,
                              reinterpret_cast<float*>(P.out) + off, P.stream);
}

static lf_status record(cudaEvent_t e, cudaStream_t s) {
  cudaError_t r = cudaEventRecord(e, s);
  if (r != cudaSuccess) {
    set_error("cudaEventRecord: %s", cudaGetErrorString(r));
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

// A timing event: inside a stream capture it becomes an event-record node of
// the graph (recorded again on every replay) instead of a capture dependency.
static lf_status record_timing(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t r = cudaStreamIsCapturing(s, &cs);
  if (r == cudaSuccess)
    r = (cs == cudaStreamCaptureStatusActive) ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                              : cudaEventRecord(e, s);
  if (r != cudaSuccess) {
    set_error("recording a timing event: %s", cudaGetErrorString(r));
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

static lf_status wait_event(cudaStream_t s, cudaEvent_t e) {
  cudaError_t r = cudaStreamWaitEvent(s, e, 0);
  if (r != cudaSuccess) {
    set_error("cudaStreamWaitEvent: %s", cudaGetErrorString(r));
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

// The parameter block of the bf16 band launches (~25 KB: kept off the stack;
// each launch copies it, so one per host thread serves every launch).
static BandParams* band_params() {
  static thread_local BandParams* bp = nullptr;
  if (!bp) bp = new (std::nothrow) BandParams;
  if (!bp) set_error("host allocation of the band parameter block failed");
  return bp;
}

template <typename T>
static lf_status forward_t(const Problem& P, bool bf16) {
  lf_status st;
  const bool g_band = P.G > 0 && global_rows_on_band_kernel(P, bf16);
  // ---- global rows: scratch (streaming pass only) and a fork point for the side stream
  float* ws = nullptr;
  AuxStream* aux = nullptr;
  if (P.G > 0 && !g_band) {
    size_t total = 0;
    for (int b0 = 0; b0 < P.B; b0 += kMaxBatch) {
      const int nb = std::min(kMaxBatch, P.B - b0);
      size_t nf = 0;
      global_chunk(P, nb, &nf);
      total += nf * sizeof(float) + global_counters((int64_t)nb * P.H, P.G) * sizeof(unsigned);
    }
    cudaError_t e = injected_fault("alloc") ? cudaErrorMemoryAllocation
                                            : cudaMallocAsync((void**)&ws, total, P.stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("scratch allocation of %zu bytes failed: %s", total, cudaGetErrorString(e));
      return LF_ERR_NO_MEMORY;
    }
  }
  // bf16: the band kernels leave the global tokens' rows to the global-row
  // pass, which can then run beside them; fp32: it runs after the band kernel
  if (P.G > 0 && bf16) {
    aux = aux_stream();
    if (aux && !(record(aux->fork, P.stream) == LF_OK && wait_event(aux->s, aux->fork) == LF_OK)) {
      cudaGetLastError();  // a failed fork only serialises the passes: clear it
      aux = nullptr;
    }
  }
  // ---- band kernel on the caller's stream, launched first so that it takes
  // the whole GPU; the global-row pass (side stream) then fills the SMs its
  // last CTAs leave idle
  st = LF_OK;
  if (t_band_start) st = record_timing(t_band_start, P.stream);
  for (int b0 = 0; st == LF_OK && b0 < P.B; b0 += kMaxBatch) {
    const int nb = std::min(kMaxBatch, P.B - b0);
    if (bf16) {
      BandParams* bp = band_params();
      st = bp ? run_band_bf16(P, b0, nb, *bp) : LF_ERR_NO_MEMORY;
    } else {
      st = run_band_f32(P, b0, nb);
    }
  }
  if (st == LF_OK && t_band_stop) st = record_timing(t_band_stop, P.stream);
  if (P.G > 0) {
    // the global rows beside the band kernel, or after it on the caller's stream
    cudaStream_t gs = aux ? aux->s : P.stream;
    lf_status gp = LF_OK;
    if (st == LF_OK && g_band) {
      for (int b0 = 0; gp == LF_OK && b0 < P.B; b0 += kMaxBatch) {
        BandParams* bp = band_params();
        gp = bp ? run_global_band_bf16(P, b0, std::min(kMaxBatch, P.B - b0), *bp, gs) : LF_ERR_NO_MEMORY;
      }
    } else if (st == LF_OK) {
      gp = global_pass<T>(P, ws, gs);
    }
    if (aux) {
      // join even on failure so nothing on the side stream outlives the scratch
      lf_status j = record(aux->join, aux->s);
      if (j == LF_OK) j = wait_event(P.stream, aux->join);
      if (gp == LF_OK) gp = j;
    }
    if (st == LF_OK) st = gp;
    if (ws) {
      cudaError_t fe = cudaFreeAsync(ws, P.stream);
      if (st == LF_OK && fe != cudaSuccess) {
        set_error("scratch free failed: %s", cudaGetErrorString(fe));
        st = LF_ERR_CUDA;
      }
    }
  }
  return st;
}

// The bias entries need the table whenever there is work.
static lf_status check_bias_table(const float* rel_bias, int32_t B, int32_t H, int32_t n) {
  if ((int64_t)B * H * n > 0 && !rel_bias) {
    t_msg[0] = 0;
    set_error("rel_bias must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  return LF_OK;
}

// The per-head window entries need the window list whenever there are heads.
static lf_status check_heads_window(const int32_t* w_heads, int32_t H) {
  if (H > 0 && !w_heads) {
    t_msg[0] = 0;
    set_error("w_heads must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  return LF_OK;
}

static lf_status forward(const Problem& P, bool bf16) {
  t_msg[0] = 0;
  lf_status st = validate(P, bf16);
  if (st != LF_OK) return st;
  if ((int64_t)P.B * P.H * P.n == 0) return LF_OK;
  if (bf16 && !encode_fn()) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return LF_ERR_CUDA;
  }
  cudaGetLastError();  // a stale error from someone else must not be reported as ours
  return bf16 ? forward_t<__nv_bfloat16>(P, true) : forward_t<float>(P, false);
}

}  // namespace lf

// ====================================================================== C ABI
extern "C" {

lf_status lf_attn_fwd(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                      const void* vg, const int32_t* global_idx, int32_t n_global, void* out,
                      int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                      const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                      cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, w, dilation, causal,
                pad_len, stream, 2};
  return lf::forward(P, true);
}

lf_status lf_attn_fwd_f32(const void* q, const void* k, const void* v, const void* qg,
                          const void* kg, const void* vg, const int32_t* global_idx,
                          int32_t n_global, void* out, int32_t B, int32_t H, int32_t n, int32_t d,
                          int32_t w, const int32_t* dilation, int32_t causal,
                          const int32_t* pad_len, cudaStream_t stream) {
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, w, dilation, causal,
                pad_len, stream, 4};
  return lf::forward(P, false);
}

lf_status lf_attn_fwd_bias(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                           const void* vg, const int32_t* global_idx, int32_t n_global, void* out,
                           int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                           const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                           const float* rel_bias, cudaStream_t stream) {
  lf_status st = lf::check_bias_table(rel_bias, B, H, n);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, w, dilation, causal,
                pad_len, stream, 2, nullptr, rel_bias};
  return lf::forward(P, true);
}

lf_status lf_attn_fwd_bias_f32(const void* q, const void* k, const void* v, const void* qg,
                               const void* kg, const void* vg, const int32_t* global_idx,
                               int32_t n_global, void* out, int32_t B, int32_t H, int32_t n, int32_t d,
                               int32_t w, const int32_t* dilation, int32_t causal,
                               const int32_t* pad_len, const float* rel_bias, cudaStream_t stream) {
  lf_status st = lf::check_bias_table(rel_bias, B, H, n);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, w, dilation, causal,
                pad_len, stream, 4, nullptr, rel_bias};
  return lf::forward(P, false);
}

lf_status lf_attn_fwd_hw(const void* q, const void* k, const void* v, const void* qg, const void* kg,
                         const void* vg, const int32_t* global_idx, int32_t n_global, void* out,
                         int32_t B, int32_t H, int32_t n, int32_t d, const int32_t* w_heads,
                         const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                         cudaStream_t stream) {
  lf_status st = lf::check_heads_window(w_heads, H);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, 0, dilation, causal,
                pad_len, stream, 2, w_heads};
  return lf::forward(P, true);
}

lf_status lf_attn_fwd_hw_f32(const void* q, const void* k, const void* v, const void* qg,
                             const void* kg, const void* vg, const int32_t* global_idx,
                             int32_t n_global, void* out, int32_t B, int32_t H, int32_t n, int32_t d,
                             const int32_t* w_heads, const int32_t* dilation, int32_t causal,
                             const int32_t* pad_len, cudaStream_t stream) {
  lf_status st = lf::check_heads_window(w_heads, H);
  if (st != LF_OK) return st;
  lf::Problem P{q, k, v, qg, kg, vg, global_idx, n_global, out, B, H, n, d, 0, dilation, causal,
                pad_len, stream, 4, w_heads};
  return lf::forward(P, false);
}

lf_status lf_attn_count_pairs(int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                              const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                              const int32_t* global_idx, int32_t n_global, int64_t* pairs,
                              double* flops) {
  lf::t_msg[0] = 0;
  lf::Problem P{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, global_idx, n_global, nullptr,
                B, H, n, d, w, dilation, causal, pad_len, nullptr, 1};
  lf_status st = lf::validate_pattern(P);
  if (st != LF_OK) return st;
  if (!pairs && !flops) return LF_OK;
  const int64_t half = std::min<int64_t>(w / 2, n);
  const int64_t right = causal ? 0 : half;
  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t L = n - (pad_len ? pad_len[b] : 0);
    for (int h = 0; h < H; ++h) {
      const int64_t delta = dilation[h];
      for (int64_t i = 0; i < L; ++i) {
        // global row?
        int lo = 0, hi = n_global - 1, is_g = 0;
        while (lo <= hi) {
          const int mid = (lo + hi) / 2;
          if (global_idx[mid] == i) { is_g = 1; break; }
          if (global_idx[mid] < i) lo = mid + 1; else hi = mid - 1;
        }
        if (is_g) {
          total += causal ? (i + 1) : L;
          continue;
        }
        // window steps t in [-half, right] with 0 <= i + delta*t < L
        const int64_t tlo = std::max<int64_t>(-half, -(i / delta));
        const int64_t thi = std::min<int64_t>(right, (L - 1 - i) / delta);
        int64_t cnt = thi >= tlo ? thi - tlo + 1 : 0;
        for (int r = 0; r < n_global; ++r) {
          const int64_t g = global_idx[r];
          if (g >= L || (causal && g > i)) continue;
          const int64_t o = g - i;
          if (o % delta == 0 && o / delta >= -half && o / delta <= right) continue;
          ++cnt;
        }
        total += cnt;
      }
    }
  }
  if (pairs) *pairs = total;
  if (flops) *flops = 4.0 * (double)d * (double)total;
  return LF_OK;
}

const char* lf_status_string(lf_status s) {
  switch (s) {
    case LF_OK: return "LF_OK";
    case LF_ERR_INVALID_ARG: return "LF_ERR_INVALID_ARG";
    case LF_ERR_UNSUPPORTED: return "LF_ERR_UNSUPPORTED";
    case LF_ERR_CUDA: return "LF_ERR_CUDA";
    case LF_ERR_NO_MEMORY: return "LF_ERR_NO_MEMORY";
    case LF_ERR_TIMEOUT: return "LF_ERR_TIMEOUT";
  }
  return "LF_ERR_UNKNOWN";
}

const char* lf_last_error_message(void) { return lf::t_msg; }

lf_status lf_attn_set_band_events(cudaEvent_t start, cudaEvent_t stop) {
  if ((start == nullptr) != (stop == nullptr)) {
    lf::set_error("set both band events or neither");
    return LF_ERR_INVALID_ARG;
  }
  lf::t_band_start = start;
  lf::t_band_stop = stop;
  return LF_OK;
}

uint64_t lf_attn_launch_count(void) { return lf::g_launches.load(std::memory_order_relaxed); }

const char* lf_attn_last_band_kernel(void) { return lf::t_band_kernel; }

lf_status lf_device_error(uint32_t* code, int32_t clear) {
  if (!code) {
    lf::set_error("code must not be NULL");
    return LF_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, lf::g_device_error, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(lf::g_device_error, &zero, sizeof zero);
  }
  if (e != cudaSuccess) {
    lf::set_error("reading the device error word: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

lf_status lf_set_wait_limit_ns(uint64_t ns) {
  const uint64_t v = ns ? ns : lf::kWaitLimitDefaultNs;
  cudaError_t e = cudaDeviceSynchronize();  // no running kernel reads it halfway
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(lf::g_wait_limit_ns, &v, sizeof v);
  if (e != cudaSuccess) {
    lf::set_error("setting the wait limit: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  return LF_OK;
}

#ifdef LF_TRACE
// Diagnostic builds only: copies the band kernel's timeline (first CTA) to
// host arrays dst[8][4096] and counts[8].
int lf_trace_dump(unsigned long long* dst, int* counts) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(dst, lf::g_trace, sizeof(lf::g_trace)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(counts, lf::g_trace_n, sizeof(lf::g_trace_n)) != cudaSuccess) return -1;
  return 0;
}
#endif

#ifdef LF_PROF
// Diagnostic builds only: copies and clears the phase counters, dst[8][12].
int lf_prof_dump(unsigned long long* dst) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(dst, lf::g_prof, sizeof(lf::g_prof)) != cudaSuccess) return -1;
  static const unsigned long long zeros[lf::kProfSlots][lf::kProfPhases] = {};
  if (cudaMemcpyToSymbol(lf::g_prof, zeros, sizeof(zeros)) != cudaSuccess) return -1;
  return 0;
}
#endif

}  // extern "C"

// The allocation-free variant of lf_attn_fwd (same translation unit).
#include "lf_noalloc.cuh"
// The backward (same translation unit).
#include "lf_bwd.cuh"
// The per-head projections (same translation unit).
#include "lf_proj.cuh"
// The memory combine (same translation unit).
#include "mem_combine.cuh"
// Global tokens that differ between batch rows (same translation unit).
#include "lf_varglobal.cuh"
