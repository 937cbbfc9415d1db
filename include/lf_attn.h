/*
 * lf_attn.h -- C ABI of the B300 (sm_103a) Longformer-style attention library.
 *
 * The operation (velog.io/@lainshower/Longformer, section 3-1 "Attention
 * Pattern" and section 4.1 for the autoregressive pattern):
 *
 *   Each token i of a sequence of n tokens attends to the keys of its window:
 *   offsets delta*t for integer t in [-w/2, +w/2] (the token itself included,
 *   so an interior row attends w + 1 keys), where delta = dilation[h] is the
 *   per-head dilation ("Dilated Sliding Window").  With causal != 0 the window
 *   keeps only t in [-w/2, 0] (look-back only, w/2 + 1 keys).
 *   A few global tokens ("Global Attention") attend to every token and every
 *   token attends to them.  Global attention has its own projections
 *   ("Linear Projections for Global Attention"): the row of a global token g
 *   is softmax(qg[g] . kg[j] / sqrt(d)) averaged over vg[j] for all valid j
 *   (j <= g when causal); every other row scores q against k over its window
 *   plus the global tokens' columns (each key counted once) and averages v.
 *   Scores are scaled by 1/sqrt(d); there is no dropout or bias.
 *   Padding: pad_len[b] trailing tokens of batch row b are never attended and
 *   their output rows are written as zeros.
 *
 * Layouts: every [B, H, n, d] tensor is row-major and contiguous (d fastest);
 * qg is [B, H, G, d] with row r belonging to position global_idx[r].
 * All device pointers must be 16-byte aligned and `out` must not overlap any
 * input.  Index arrays (global_idx, dilation, pad_len) are HOST memory, read
 * during the call and not retained.  The caller owns every buffer; the
 * library keeps no pointer after returning.
 *
 * Calls are asynchronous on `stream` (0 = legacy default stream): they
 * enqueue kernels and return without synchronising.  Arguments are validated
 * on the host before anything is enqueued; on any error the call returns a
 * non-zero status, enqueues nothing and leaves `out` untouched.  A call that
 * fails after validation (a CUDA launch error) returns LF_ERR_CUDA.
 * lf_last_error_message() then describes the failure (per host thread).
 */
#ifndef LF_ATTN_H
#define LF_ATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LF_OK = 0,
  LF_ERR_INVALID_ARG = 1, /* a null/misaligned pointer, bad size, unsorted global list, ... */
  LF_ERR_UNSUPPORTED = 2, /* valid but outside this build's limits (e.g. bf16 d not 64/128) */
  LF_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  LF_ERR_NO_MEMORY = 4,   /* scratch space for the global rows could not be allocated */
  LF_ERR_TIMEOUT = 5      /* a kernel gave up waiting (reported by lf_device_error) */
} lf_status;

/* Largest number of global tokens per call. */
#define LF_MAX_GLOBAL 4096

/*
 * bf16 forward.  q, k, v, kg, vg, out: [B, H, n, d] bf16 device memory;
 * qg: [B, H, G, d] bf16 device memory.  G = n_global (0 <= G <= LF_MAX_GLOBAL);
 * global_idx: host array of G strictly increasing positions in [0, n), NULL
 * iff G == 0 (qg, kg, vg may then be NULL).  w: total window, even, >= 0.
 * dilation: host array of H values >= 1.  causal: 0 or 1.  pad_len: host
 * array of B trailing-pad counts in [0, n], or NULL for none.
 * Supported d: 64 and 128.  Computes in fp32 on the tensor cores (bf16
 * operands, fp32 accumulation, fp32 online softmax) and rounds the output
 * to bf16 (round to nearest even).
 *
 * Stream-ordered on `stream`.  With n_global > 0 the global tokens' rows run
 * on a second stream of the library's (one per host thread and device),
 * forked from and joined back into `stream` with events, beside the band
 * kernel; the call is still complete when work enqueued on `stream` after it
 * starts.  Scratch for those rows is allocated stream-ordered on `stream`,
 * except for d = 64 with n_global >= 16, whose rows run on the tensor cores
 * without scratch.
 */
lf_status lf_attn_fwd(const void* q, const void* k, const void* v,
                      const void* qg, const void* kg, const void* vg,
                      const int32_t* global_idx, int32_t n_global,
                      void* out,
                      int32_t B, int32_t H, int32_t n, int32_t d,
                      int32_t w, const int32_t* dilation, int32_t causal,
                      const int32_t* pad_len, cudaStream_t stream);

/*
 * fp32 forward: same arguments and semantics as lf_attn_fwd with every
 * tensor in fp32; any d in [1, 128].  CUDA-core arithmetic in fp32.
 */
lf_status lf_attn_fwd_f32(const void* q, const void* k, const void* v,
                          const void* qg, const void* kg, const void* vg,
                          const int32_t* global_idx, int32_t n_global,
                          void* out,
                          int32_t B, int32_t H, int32_t n, int32_t d,
                          int32_t w, const int32_t* dilation, int32_t causal,
                          const int32_t* pad_len, cudaStream_t stream);

/*
 * lf_attn_fwd without any device memory allocation.  The pages have no
 * counterpart to this: it is an interface choice, not part of the method.
 *
 * lf_attn_fwd allocates the scratch of its global-row pass (stream-ordered,
 * on every call with n_global > 0 that does not take the scratch-free path
 * for d = 64 with n_global >= 16).  This variant is for callers that cannot
 * allocate device memory while they run: an engine that reserves its whole
 * memory budget at start-up, code that must not meet an out-of-memory error
 * or allocator latency in the middle of a step, or a host application that
 * owns the CUDA allocator and does not let plug-ins call it.
 *
 * Same arguments, semantics and results as lf_attn_fwd (bf16; results agree
 * within rounding, since the global rows may be split into longer key
 * chunks).  The scratch is a 16 MiB array inside the library that every GPU
 * loading the library holds until the process exits.  Every call looks up
 * that array's device address (so it stays right after a device reset); the
 * first lookup on a device may load the library's module there, so make the
 * first call on a device before any stream capture.  Returns LF_ERR_UNSUPPORTED when
 * B*H*n_global*(d+2) fp32 values plus B*H*n_global 32-bit counters (per
 * block of 256 batch rows) exceed the array (never for d = 64 with
 * n_global >= 16, which needs no scratch).  Everything runs on `stream`.  All
 * calls share the array and it keeps the last call's contents (every value a
 * call reads is written earlier in that call): calls whose kernels overlap
 * on the GPU, e.g. on two streams at once, race on it.
 */
lf_status lf_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                              const void* qg, const void* kg, const void* vg,
                              const int32_t* global_idx, int32_t n_global,
                              void* out,
                              int32_t B, int32_t H, int32_t n, int32_t d,
                              int32_t w, const int32_t* dilation, int32_t causal,
                              const int32_t* pad_len, cudaStream_t stream);

/*
 * Backward of lf_attn_fwd: the gradients of L = sum(dout * out) with respect
 * to q, k, v and, when n_global > 0, qg, kg, vg, where out is the forward's
 * output for the same arguments.  The chain rule through each row's softmax
 * over the same attended sets as the forward (section 3-1 "Attention
 * Pattern"): with p the row's weights, dp_t = <dout_row, v_t> and
 * D = sum_t p_t dp_t, ds_t = p_t (dp_t - D); dq_row = sum_t ds_t k_t / sqrt(d),
 * dk_t += ds_t q_row / sqrt(d), dv_t += p_t dout_row.  A global token's row
 * uses qg, kg, vg and adds into dqg, dkg, dvg.
 *
 * Inputs as for lf_attn_fwd (bf16, d = 64 or 128), plus dout: [B, H, n, d]
 * bf16 device memory.  Outputs: dq, dk, dv, dkg, dvg [B, H, n, d] and dqg
 * [B, H, G, d], fp32 device memory, 16-byte aligned, each written in full
 * (padding rows and never-attended keys get zeros); none may overlap an
 * input or another output.  dqg, dkg, dvg may be NULL iff n_global == 0.
 * The row statistics are recomputed (no forward state is needed).  CUDA-core
 * arithmetic in fp32 with a fixed summation order: repeated calls give the
 * same bits.  Scratch of 8 * min(B, 256) * min(H, 256) * n bytes is
 * allocated stream-ordered on `stream` (LF_ERR_NO_MEMORY if that fails).
 * Two kernels per block of 256 batch rows and 256 heads, on `stream`.
 */
lf_status lf_attn_bwd(const void* q, const void* k, const void* v,
                      const void* qg, const void* kg, const void* vg,
                      const int32_t* global_idx, int32_t n_global,
                      const void* dout,
                      float* dq, float* dk, float* dv,
                      float* dqg, float* dkg, float* dvg,
                      int32_t B, int32_t H, int32_t n, int32_t d,
                      int32_t w, const int32_t* dilation, int32_t causal,
                      const int32_t* pad_len, cudaStream_t stream);

/*
 * fp32 backward: lf_attn_bwd with fp32 inputs (and dout); any d in [1, 128].
 */
lf_status lf_attn_bwd_f32(const void* q, const void* k, const void* v,
                          const void* qg, const void* kg, const void* vg,
                          const int32_t* global_idx, int32_t n_global,
                          const void* dout,
                          float* dq, float* dk, float* dv,
                          float* dqg, float* dkg, float* dvg,
                          int32_t B, int32_t H, int32_t n, int32_t d,
                          int32_t w, const int32_t* dilation, int32_t causal,
                          const int32_t* pad_len, cudaStream_t stream);

/*
 * Relative position bias (Memorizing Transformer notes, "Position bias": a
 * T5-style bias added to the attention scores, one learned scalar per head
 * and relative position): as lf_attn_fwd / lf_attn_fwd_f32, with
 *   score(i, j) = <q_i, k_j> / sqrt(d) + rel_bias[h * (w + 1) + t + w/2]
 * for every key j in row i's band, t = (j - i) / dilation[h] in [-w/2, w/2]
 * its window step (causal rows read t <= 0 only).  Global columns outside
 * the band and the global tokens' own rows carry no bias.  A bucketed bias
 * (T5's log-spaced buckets of the token distance |j - i|) is passed expanded
 * into this table.  rel_bias: fp32 DEVICE memory [H, w + 1], 4-byte
 * aligned, not overlapping `out`; NULL only for an empty problem.
 * bf16 d = 64 runs the ring kernel whatever the number of global tokens;
 * d = 128 the pair kernel; fp32 the CUDA-core kernel.  Errors as in the
 * calls they extend.
 */
lf_status lf_attn_fwd_bias(const void* q, const void* k, const void* v,
                           const void* qg, const void* kg, const void* vg,
                           const int32_t* global_idx, int32_t n_global, void* out,
                           int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                           const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                           const float* rel_bias, cudaStream_t stream);
lf_status lf_attn_fwd_bias_f32(const void* q, const void* k, const void* v,
                               const void* qg, const void* kg, const void* vg,
                               const int32_t* global_idx, int32_t n_global, void* out,
                               int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                               const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                               const float* rel_bias, cudaStream_t stream);

/*
 * Backward with the relative position bias: as lf_attn_bwd / lf_attn_bwd_f32
 * for the scores of lf_attn_fwd_bias, plus the bias's own gradient
 *   d_rel_bias[h * (w + 1) + t + w/2] = sum over the batch rows and the band
 *   entries (i, j) of head h at window step t of dL/dscore(i, j)
 * (entries no band entry reaches are 0).  d_rel_bias: fp32 DEVICE memory
 * [H, w + 1], 4-byte aligned, overlapping nothing else, or NULL to skip it;
 * it is written in full (summed in a fixed order: bitwise reproducible).
 * With d_rel_bias, w <= 4096 (LF_ERR_UNSUPPORTED otherwise); its partial
 * sums take B*H*ceil(n/64)*(w + 1)*4 bytes of stream-ordered scratch per
 * block of 256 batch rows and 256 heads.
 */
lf_status lf_attn_bwd_bias(const void* q, const void* k, const void* v,
                           const void* qg, const void* kg, const void* vg,
                           const int32_t* global_idx, int32_t n_global, const void* dout,
                           float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                           int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                           const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                           const float* rel_bias, float* d_rel_bias, cudaStream_t stream);
lf_status lf_attn_bwd_bias_f32(const void* q, const void* k, const void* v,
                               const void* qg, const void* kg, const void* vg,
                               const int32_t* global_idx, int32_t n_global, const void* dout,
                               float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                               int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                               const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                               const float* rel_bias, float* d_rel_bias, cudaStream_t stream);

/*
 * Per-head windows (velog.io/@lainshower/Longformer, section 4.1: the window
 * size is chosen per layer, and within a layer heads differ, some dilated and
 * some not): as lf_attn_fwd / lf_attn_fwd_f32 / lf_attn_bwd / lf_attn_bwd_f32,
 * with head h using the window w_heads[h] (even, >= 0) in place of the one w.
 * w_heads: host array of H values, read during the call, NULL only if H == 0.
 * bf16: one band launch holds every head's tiles, each carrying its head's
 * reach (d = 64 with windows that differ runs the ring kernel).  Errors as in
 * the calls they extend; a bad w_heads entry is LF_ERR_INVALID_ARG.
 */
lf_status lf_attn_fwd_hw(const void* q, const void* k, const void* v,
                         const void* qg, const void* kg, const void* vg,
                         const int32_t* global_idx, int32_t n_global, void* out,
                         int32_t B, int32_t H, int32_t n, int32_t d,
                         const int32_t* w_heads, const int32_t* dilation, int32_t causal,
                         const int32_t* pad_len, cudaStream_t stream);
lf_status lf_attn_fwd_hw_f32(const void* q, const void* k, const void* v,
                             const void* qg, const void* kg, const void* vg,
                             const int32_t* global_idx, int32_t n_global, void* out,
                             int32_t B, int32_t H, int32_t n, int32_t d,
                             const int32_t* w_heads, const int32_t* dilation, int32_t causal,
                             const int32_t* pad_len, cudaStream_t stream);
lf_status lf_attn_bwd_hw(const void* q, const void* k, const void* v,
                         const void* qg, const void* kg, const void* vg,
                         const int32_t* global_idx, int32_t n_global, const void* dout,
                         float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                         int32_t B, int32_t H, int32_t n, int32_t d,
                         const int32_t* w_heads, const int32_t* dilation, int32_t causal,
                         const int32_t* pad_len, cudaStream_t stream);
lf_status lf_attn_bwd_hw_f32(const void* q, const void* k, const void* v,
                             const void* qg, const void* kg, const void* vg,
                             const int32_t* global_idx, int32_t n_global, const void* dout,
                             float* dq, float* dk, float* dv, float* dqg, float* dkg, float* dvg,
                             int32_t B, int32_t H, int32_t n, int32_t d,
                             const int32_t* w_heads, const int32_t* dilation, int32_t causal,
                             const int32_t* pad_len, cudaStream_t stream);

/*
 * Per-head linear projections of hidden states (section 3-1, "Linear
 * Projections for Global Attention": the band and the global attention each
 * use their own W_q, W_k, W_v), producing the inputs of lf_attn_fwd:
 *   y[t, b, h, i, c] = sum_k x[b, i, k] * w[t*H*d + h*d + c, k] (+ bias[...])
 * x: [B, n, K] bf16 hidden states; w: [n_out*H*d, K] bf16, the weights of
 * n_out projections stacked row-wise (a row holds one output column's
 * weights, as in a linear layer's [out, in] weight); bias: [n_out*H*d] fp32
 * or NULL; y: [n_out, B, H, n, d] bf16, n_out consecutive head-major tensors
 * (e.g. q, k, v, kg, vg with n_out = 5; qg from the global tokens' hidden
 * states with its own weights in a second call).  All device memory, x, w, y
 * 16-byte aligned, y not overlapping x or w.  Requires K a multiple of 64,
 * d a multiple of 32 and n_out*H*d a multiple of 128 (LF_ERR_UNSUPPORTED
 * otherwise).  Tensor cores (bf16 operands, fp32 accumulation, output rounded
 * to bf16, nearest even); one launch on `stream`.
 */
lf_status lf_proj_heads(const void* x, const void* w, const float* bias, void* y,
                        int32_t B, int32_t n, int32_t K, int32_t n_out, int32_t H, int32_t d,
                        cudaStream_t stream);

/*
 * Memorizing-Transformer combine (Memorizing Transformer notes, section
 * "Memorizing Transformer"): each query also attends the km (key, value)
 * pairs a kNN lookup retrieved from a memory of earlier segments, and the
 * two results are mixed per head:
 *   o_mem = sum_j softmax_j(<q, mem_k[idx_j]> / sqrt(d)) mem_v[idx_j]
 *           over the non-empty slots (zero if every slot is empty)
 *   out   = gate[h] * o_mem + (1 - gate[h]) * local
 * q, local, out: [B, H, n, d] bf16 (local: the band attention's output; out
 * may be local itself, not any other input); mem_k, mem_v: [B, H, M, d] bf16
 * (the memory of each (b, h); may be NULL iff M == 0); idx: [B, H, n, km]
 * int32 positions in that memory, -1 for an empty slot; gate: [H] fp32
 * weights (the per-head scalar, already mapped to [0, 1] by the caller).
 * All device memory; bf16 tensors 16-byte aligned, idx and gate 4-byte.
 * d = 64 or 128; 1 <= km <= 32.  The lookup itself is not part of this call.
 * An index outside [-1, M) is treated as an empty slot and recorded in the
 * device error word (LF_ERR_INVALID_ARG, role 7; see lf_device_error).
 * CUDA cores, fp32 arithmetic; one launch on `stream`.
 */
lf_status lf_mem_combine(const void* q, const void* local, const void* mem_k, const void* mem_v,
                         const int32_t* idx, const float* gate, void* out,
                         int32_t B, int32_t H, int32_t n, int32_t d, int32_t M, int32_t km,
                         cudaStream_t stream);

/*
 * Global tokens that differ between batch rows (section 3-1 "Global
 * Attention": the question tokens of a QA example are its global tokens, and
 * questions differ per example).  Batch row b's global positions are
 * global_idx[global_offsets[b] .. global_offsets[b+1]) (host arrays;
 * global_offsets has B + 1 entries, starts at 0, non-decreasing; each row's
 * list strictly increasing in [0, n)).  qg is packed: batch row b's
 * [H, G_b, d] block starts at row global_offsets[b] * H (elements
 * global_offsets[b] * H * d).  kg, vg: [B, H, n, d] as for lf_attn_fwd (may
 * be NULL iff every row has no global token).  Everything else as for
 * lf_attn_fwd (bf16).  Runs each batch row's forward in turn on `stream`;
 * every row is validated before anything is enqueued.
 */
lf_status lf_attn_fwd_varglobal(const void* q, const void* k, const void* v,
                                const void* qg, const void* kg, const void* vg,
                                const int32_t* global_offsets, const int32_t* global_idx,
                                void* out,
                                int32_t B, int32_t H, int32_t n, int32_t d,
                                int32_t w, const int32_t* dilation, int32_t causal,
                                const int32_t* pad_len, cudaStream_t stream);

/*
 * Backward of lf_attn_fwd_varglobal: as lf_attn_bwd, with the global lists
 * and the packed qg of lf_attn_fwd_varglobal; dqg is packed like qg; the dkg,
 * dvg rows of a batch row without global tokens are written as zeros.
 */
lf_status lf_attn_bwd_varglobal(const void* q, const void* k, const void* v,
                                const void* qg, const void* kg, const void* vg,
                                const int32_t* global_offsets, const int32_t* global_idx,
                                const void* dout,
                                float* dq, float* dk, float* dv,
                                float* dqg, float* dkg, float* dvg,
                                int32_t B, int32_t H, int32_t n, int32_t d,
                                int32_t w, const int32_t* dilation, int32_t causal,
                                const int32_t* pad_len, cudaStream_t stream);

/*
 * Host-only: the useful work of a problem, counted exactly from the pattern.
 * *pairs = number of attended (query, key) pairs over all valid rows and
 * heads; *flops = 4 * d * pairs (one multiply-add each for QK^T and PV).
 * Takes the same pattern arguments as lf_attn_fwd; touches no GPU.
 */
lf_status lf_attn_count_pairs(int32_t B, int32_t H, int32_t n, int32_t d, int32_t w,
                              const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                              const int32_t* global_idx, int32_t n_global,
                              int64_t* pairs, double* flops);

/* Name of a status code (static storage). */
const char* lf_status_string(lf_status s);

/* Detail of the last failure on the calling host thread ("" if none). */
const char* lf_last_error_message(void);

/*
 * Profiling hook.  While set (non-NULL), every forward call records `start`
 * just before and `stop` just after its band kernel, on the call's stream.
 * Pass NULL, NULL to clear.  Per host thread.
 */
lf_status lf_attn_set_band_events(cudaEvent_t start, cudaEvent_t stop);

/* Number of kernels this library has launched in this process. */
uint64_t lf_attn_launch_count(void);

/*
 * Name of the band kernel that the last forward call on this host thread
 * launched ("band_ring", "band_duo", "band_pair" or "band_simt_f32"; "" before
 * the first).  A static string: the caller does not free it.
 */
const char* lf_attn_last_band_kernel(void);

/*
 * Synchronises the current device and reads the library's device error word
 * (0 = none; otherwise LF_ERR_TIMEOUT in the low byte and the kernel role
 * that gave up in the next byte, or LF_ERR_INVALID_ARG with role 7 when
 * lf_mem_combine met an index out of range).  clear != 0 resets it to 0.
 */
lf_status lf_device_error(uint32_t* code, int32_t clear);

/*
 * Testing hook for the timeout path.  Sets, for the current device, how long
 * a kernel's pipeline wait (a role waiting for another role's barrier) may
 * last before the kernel gives up: it then records LF_ERR_TIMEOUT in the
 * device error word, every role leaves its loop, the in-flight copies and
 * MMAs are waited for (those drain waits keep their own 200 ms limit) and
 * the kernel returns; the call's output is then undefined.  ns = 0 restores
 * the default of 2 s.  Synchronises the device first.  Returns LF_ERR_CUDA
 * if the device cannot be reached.
 */
lf_status lf_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* LF_ATTN_H */
