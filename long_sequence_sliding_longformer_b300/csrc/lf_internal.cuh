// lf_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
//
// Parameter blocks passed by value to the kernels, limits, the device error
// word, and thin inline-PTX wrappers for the sm_100-family features the band
// kernel uses: mbarriers, TMA tensor loads, and tcgen05 (TMEM allocation,
// MMA, commit, TMEM loads/stores).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/lf_attn.h"

namespace lf {

// ----------------------------------------------------------------- limits
constexpr int kMaxSets = 8;      // (dilation, residue) tensor-map sets per band launch
constexpr int kMaxSeg = 32;      // (head, residue) segments per band launch (copied to shared memory)
constexpr int kMaxBatch = 256;   // batch rows per launch (larger B is split on the host)
constexpr int kMaxGlobal = LF_MAX_GLOBAL;

// ----------------------------------------------------------------- error word
// Bits 0-7: lf_status of the failure; bits 8-15: role that gave up.
enum Role : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleDrain = 4, kRoleTranspose = 5 };
// Defined once here: the library is built as a single translation unit.
__device__ uint32_t g_device_error = 0;
// Limit of the pipeline waits, in ns (settable for tests of the timeout
// path); the drain waits at a kernel's end keep kDrainLimitNs.
constexpr uint64_t kWaitLimitDefaultNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
__device__ uint64_t g_wait_limit_ns = kWaitLimitDefaultNs;

// ----------------------------------------------------------------- timeline trace
// Built only with -DLF_TRACE (a diagnostic build, never the product): the
// first CTA of the band kernel records (SM clock << 8 | event code) per
// role into g_trace[track], read back with lf_trace_dump().
#ifdef LF_TRACE
constexpr int kTraceTracks = 8, kTraceLen = 4096;
__device__ unsigned long long g_trace[kTraceTracks][kTraceLen];
__device__ int g_trace_n[kTraceTracks];
#endif

// ----------------------------------------------------------------- phase counters
// Built only with -DLF_PROF (a diagnostic build, never the product): each
// role adds the SM cycles it spent in each phase of its loop into
// g_prof[slot][phase], summed over all CTAs; read back with lf_prof_dump().
#ifdef LF_PROF
constexpr int kProfSlots = 8, kProfPhases = 12;
__device__ unsigned long long g_prof[kProfSlots][kProfPhases];
#endif

// ----------------------------------------------------------------- band kernel params
// A segment is one (head, residue class) of the dilated window: rows
// i = r + delta*m for m in [0, n_r).  Its work items are its 128-row tiles
// (D = 64) or pairs of consecutive tiles (D = 128).  half: its head's window
// reach in steps (look-back half, look-ahead causal ? 0 : half).
struct BandSeg {
  int32_t h, r, delta, n_r, items, set, begin, half;
};

struct BandParams {
  CUtensorMap tq[kMaxSets];  // per (delta, r): dims {d, n_r, B*H}, row stride delta*d
  CUtensorMap tk[kMaxSets];
  CUtensorMap tv[kMaxSets];
  const __nv_bfloat16* k;  // row gathers of the global tokens' keys/values
  const __nv_bfloat16* v;
  __nv_bfloat16* out;
  int32_t B, H, n;
  // window reach in steps shared by every head of the launch (look-back
  // half, look-ahead right); the duo kernel is only chosen when all heads
  // share one window
  int32_t half, right;
  // Heads' windows differ (varwin = 1): the ring and pair kernels then read
  // each segment's reach (an instantiation of their own); otherwise every
  // kernel reads half and right above.
  int32_t varwin;
  int32_t causal, G, nseg, items_per_b, total_items;
  float sl2;               // log2(e) / sqrt(d)
  // Global-row mode (d = 64 kernel only): the query rows are the global
  // tokens (tq over qg, nrow_g of them per plane, at positions gidx), the
  // keys and values are kg and vg, every key below the row's valid length
  // (and at or before the token when causal) is attended, and the rows are
  // written at the tokens' positions.  G is then 0 (no global entries).
  int32_t gmode, nrow_g;
  // Work items are pairs of consecutive 128-row tiles (1) or single tiles (0).
  int32_t pair;
  // The launch runs a kernel that takes items of two tiles (duo, pair: 1) or
  // the ring kernel (0).
  int32_t pair_kernel;
  // Relative position bias of the band keys (ring and pair kernels):
  // rel_bias[h * rb_stride + rb_half + t] is added to the scaled score of the
  // key at window step t; nullptr: none.
  const float* rel_bias;
  int32_t rb_stride, rb_half;
  int32_t pad[kMaxBatch];
  BandSeg seg[kMaxSeg];
  int32_t gidx[kMaxGlobal];
};

// ----------------------------------------------------------------- simt / global-row params
struct PatternParams {
  int32_t B, H, n, d, causal, G;
  float scale;
  int32_t dil_max;               // unused by kernels; kept for host checks
  int32_t pad[kMaxBatch];
  int32_t gidx[kMaxGlobal];
};

// dilation and window per head for the SIMT kernel (at most kMaxHeadsSimt heads)
constexpr int kMaxHeadsSimt = 256;
struct SimtParams {
  PatternParams pat;
  int32_t dil[kMaxHeadsSimt];
  int32_t half_h[kMaxHeadsSimt];  // reach in steps: back half_h, ahead causal ? 0 : half_h
  // relative position bias of the band keys: rel_bias[h * rb_stride + rb_half + t]
  // is added to the scaled score at window step t (nullptr: none)
  const float* rel_bias;
  int32_t rb_stride, rb_half;
};

// ----------------------------------------------------------------- host-side launchers
struct LaunchCtx {
  cudaStream_t stream;
  cudaEvent_t band_start, band_stop;  // optional
};

// All return LF_OK or an error status and set the thread's message.
lf_status launch_band_tc(const BandParams& p, int d, int grid, cudaStream_t s);
lf_status launch_band_simt_f32(const SimtParams& p, const float* q, const float* k, const float* v,
                               float* out, cudaStream_t s);
template <typename T>
lf_status launch_global_rows(const PatternParams& p, const T* qg, const T* kg, const T* vg, T* out,
                             float* ws, unsigned* counters, int nchunks, int chunk, cudaStream_t s);

void set_error(const char* fmt, ...);
void count_launch(int k = 1);

// Raises `func`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute applies to the device that is
// current when it is set); `done` holds one bit per device already set.
inline lf_status smem_attr_once(const void* func, int bytes, std::atomic<uint64_t>& done, const char* name) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return LF_OK;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute(%s): %s", name, cudaGetErrorString(e));
    return LF_ERR_CUDA;
  }
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return LF_OK;
}

// ----------------------------------------------------------------- device helpers
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef LF_TRACE
struct Tracer {
  int track = -1, n = 0;
  __device__ void ev(int code) {
    if (track >= 0 && n < kTraceLen) g_trace[track][n++] = ((unsigned long long)clock64() << 8) | (unsigned)code;
  }
  __device__ void done() {
    if (track >= 0) g_trace_n[track] = n;
  }
};
#else
struct Tracer {
  int track = -1;
  __device__ __forceinline__ void ev(int) {}
  __device__ __forceinline__ void done() {}
};
#endif

#ifdef LF_PROF
struct Prof {
  uint32_t t, acc[kProfPhases];
  __device__ __forceinline__ Prof() : t((uint32_t)clock()) {
#pragma unroll
    for (int i = 0; i < kProfPhases; ++i) acc[i] = 0;
  }
  // cycles since the previous lap go to phase k (k a compile-time constant)
  __device__ __forceinline__ void lap(int k) {
    const uint32_t now = (uint32_t)clock();
    acc[k] += now - t;
    t = now;
  }
  __device__ __forceinline__ void flush(int slot, bool writer) {
    if (!writer) return;
#pragma unroll
    for (int i = 0; i < kProfPhases; ++i) atomicAdd(&g_prof[slot][i], (unsigned long long)acc[i]);
  }
};
#else
struct Prof {
  __device__ __forceinline__ void lap(int) {}
  __device__ __forceinline__ void flush(int, bool) {}
};
#endif

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Tests the phase; if it is not complete the thread may sleep until it
// completes or about `hint_ns` pass (so waiting warps do not spin on the
// issue slots of working ones).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 20000) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The pipeline waits' limit as set on the device.
__device__ __forceinline__ uint64_t wait_limit_ns() {
  return *reinterpret_cast<volatile uint64_t*>(&g_wait_limit_ns);
}

// Every kernel keeps its abort flag (an int at an address 4 mod 8) in shared
// memory, followed by the CTA's copy of the pipeline-wait limit, which thread
// 0 reads from wait_limit_ns() once at the kernel's start.
__device__ __forceinline__ volatile uint64_t* cta_wait_limit(volatile int* abort) {
  return reinterpret_cast<volatile uint64_t*>(abort + 1);
}

// Bounded wait: gives up after `limit_ns` (0: the CTA's pipeline limit; then
// `abort` must be the CTA's abort flag) or when *abort becomes non-zero.  On
// giving up it records the role in the device error word, raises *abort and
// returns false.  Polls suspend for up to 20 us each; below a 20 us limit
// they do not suspend at all and the limit is checked after every poll.
// Time is counted in SM cycles at two per ns (the global timer can tick as
// coarsely as 1 us): at least the limit at clocks up to 2 GHz.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t role, uint64_t limit_ns = 0) {
  if (mbar_test_wait(bar, parity)) return true;
  if (limit_ns == 0) limit_ns = *cta_wait_limit(abort);
  const bool short_limit = limit_ns < 20000ull;
  const uint64_t limit_cyc = 2 * limit_ns;
  const uint64_t c0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (short_limit ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (short_limit || (it & 7u) == 0) {
      if (*abort) return false;
      if ((uint64_t)clock64() - c0 > limit_cyc) {
        atomicCAS(&g_device_error, 0u, (uint32_t)LF_ERR_TIMEOUT | (role << 8));
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait by a whole warp; the lanes agree on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t role) {
  const bool ok = mbar_wait(bar, parity, abort, role);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same MMA issued by one lane that the (converged) warp elects; every
// lane calls it.  Issuing from a warp that stays converged is much faster
// than a run of MMAs inside a branch taken by a single lane.
__device__ __forceinline__ void mma_bf16_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, version 1 (sm_100 family).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
// b_mn_major: B operand stored with N contiguous (as V is).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp receives lane
// (32*(warp%4) + t) of TMEM, columns [col, col+32).  Waits for completion.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&f)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&f)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(f[0])), "r"(__float_as_uint(f[1])), "r"(__float_as_uint(f[2])),
      "r"(__float_as_uint(f[3])), "r"(__float_as_uint(f[4])), "r"(__float_as_uint(f[5])),
      "r"(__float_as_uint(f[6])), "r"(__float_as_uint(f[7])), "r"(__float_as_uint(f[8])),
      "r"(__float_as_uint(f[9])), "r"(__float_as_uint(f[10])), "r"(__float_as_uint(f[11])),
      "r"(__float_as_uint(f[12])), "r"(__float_as_uint(f[13])), "r"(__float_as_uint(f[14])),
      "r"(__float_as_uint(f[15])), "r"(__float_as_uint(f[16])), "r"(__float_as_uint(f[17])),
      "r"(__float_as_uint(f[18])), "r"(__float_as_uint(f[19])), "r"(__float_as_uint(f[20])),
      "r"(__float_as_uint(f[21])), "r"(__float_as_uint(f[22])), "r"(__float_as_uint(f[23])),
      "r"(__float_as_uint(f[24])), "r"(__float_as_uint(f[25])), "r"(__float_as_uint(f[26])),
      "r"(__float_as_uint(f[27])), "r"(__float_as_uint(f[28])), "r"(__float_as_uint(f[29])),
      "r"(__float_as_uint(f[30])), "r"(__float_as_uint(f[31]))
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T: A (M x K, K-major) read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// mma_bf16_ts issued by an elected lane of the converged warp (see mma_bf16_ss_w).
__device__ __forceinline__ void mma_bf16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// mma_commit by an elected lane of the converged warp.  The arrive tracks the
// MMAs that lane issued: pair it with the _w issues above, whose elected lane
// is the same (elect.sync picks the lowest active lane).
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 columns into r[0..32) without waiting; complete with tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 columns into r[0..16) without waiting; complete with tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// reg_fence32 for 16 registers.
__device__ __forceinline__ void reg_fence16(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Ties 32 registers to a point after tmem_wait_ld(), so that no use of values
// loaded by tmem_ld32_nw can be scheduled before the wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 32 lanes x 16 columns from r[0..16) without waiting; complete with tmem_wait_st().
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 32 lanes x 8 columns from r[0..8) without waiting; complete with tmem_wait_st().
__device__ __forceinline__ void tmem_st8_nw(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
      "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One lane of the (fully active) warp is elected; the others get false.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Four 8x8 b16 matrices, transposed on the way into registers (row addresses
// from lanes 8i..8i+7 for matrix i).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& x0, uint32_t& x1,
                                                  uint32_t& x2, uint32_t& x3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t x0, uint32_t x1, uint32_t x2,
                                            uint32_t x3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(x0), "r"(x1), "r"(x2), "r"(x3)
               : "memory");
}

// Per 16-bit half, the unsigned maximum.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

#endif  // __CUDACC__

}  // namespace lf
