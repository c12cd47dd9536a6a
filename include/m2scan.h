/*
 * m2scan — C ABI of the gated temporal scan layer (forward and backward) for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer, per sample b (t = 0 is the oldest history step and is scanned
 * first; SH2 = trunk width, D = STATE_D, K = history length):
 *
 *   A[t,:]  = h_history[b,t,:] . W_A     B[t,:] = h_history[b,t,:] . W_B
 *   C       = h_s2[b,:] . W_C
 *       ("Custom Kernel Optimization -- cuBLAS Projections + Batch-Parallel
 *        Scans", Design 1, Step 1: the three projections)
 *   x_{-1} = 0,  x_t = sigmoid(A[t]) * x_{t-1} + B[t]        (elementwise)
 *       (same section, Step 2; "Custom Kernel Optimization Implementation
 *        Plan", Task 1 Step 3)
 *   ctx = C * x_{K-1}                                         (elementwise)
 *   h_enriched[b,:] = h_s2[b,:] + tw * (ctx . W_O)
 *       (the pages leave this output step open, design spec Design 1 Step 3;
 *        the layer fixes it as a residual plus a [D,SH2] output projection
 *        scaled by the scalar tw)
 *
 * and the backward is the reverse scan of the implementation plan's Task 2
 * (d_gate = dx * x_{t-1} * sigmoid', dx <- dx * gate), extended to every
 * input: dW_A, dW_B, dW_C, dW_O, d_h_history and d_h_s2.
 *
 * Conventions for every call:
 *   - All tensors are fp32, row-major and contiguous:
 *       h_history, d_h_history  [B, K, SH2]
 *       h_s2, h_enriched, d_h_enriched, d_h_s2  [B, SH2]
 *       W_A, W_B, W_C, dW_A, dW_B, dW_C  [SH2, D]
 *       W_O, dW_O  [D, SH2]
 *   - Every pointer is a DEVICE pointer (cudaMalloc or equivalent) on the
 *     current device, 16-byte aligned. The caller owns every buffer; the
 *     library allocates nothing on the device and keeps no pointer after the
 *     call returns.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise. Outputs are OVERWRITTEN, never accumulated into.
 *   - Outputs must not overlap any input or each other (checked on the host).
 *   - All argument checks run on the host before anything is launched; a
 *     failing check launches nothing and returns the status.
 *   - Results are bit-identical from run to run for the same inputs and
 *     shapes on the same GPU model: the weight gradients are summed over a
 *     fixed sample-to-slot assignment and the slots are added in slot order
 *     (the deterministic two-phase reduction of "Phase 3 Kernel Optimization
 *     Implementation Plan", Task 2), with no floating-point atomics.
 *   - The library looks up, once per device, the device addresses of its
 *     static device variables and sets its kernels' shared-memory limits,
 *     and keeps both for the life of the process. cudaDeviceReset (or
 *     anything else that destroys the device's primary context) while the
 *     library is in use is not supported: later calls would use addresses
 *     from the destroyed context.
 *   - Supported shapes: B >= 0, K >= 1, SH2 >= 4 with SH2 % 4 == 0, D >= 1,
 *     and per-sample scratch of 4*K*2*D bytes within shared memory (the
 *     generic fallback kernels): K * D <= 16384. Kernel families by shape
 *     (m2scan_path_for / m2scan_fwd_path_for answer for a shape):
 *       fused tensor-core kernels: D = 4, 8 or 16, SH2 % 32 == 0,
 *         32 <= SH2 <= 256, K <= 128;
 *       wide-state tensor-core kernels: D = 64, SH2 % 128 == 0, K <= 128,
 *         B * K < 2^31;
 *       the generic kernels: every other supported shape.
 */
#ifndef M2SCAN_H
#define M2SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* m2scan_stream_t;

typedef enum {
  M2SCAN_OK = 0,
  M2SCAN_ERR_NULL = 1,        /* a required pointer is NULL */
  M2SCAN_ERR_SHAPE = 2,       /* B < 0, K < 1, SH2 < 4, SH2 % 4 != 0 or D < 1 */
  M2SCAN_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  M2SCAN_ERR_ALIAS = 4,       /* an output range overlaps an input or another output */
  M2SCAN_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than the query says */
  M2SCAN_ERR_UNSUPPORTED = 6, /* shape outside every kernel instance (K*D too large) */
  M2SCAN_ERR_CUDA = 7,        /* a CUDA runtime call failed; see m2scan_last_cuda_error */
  M2SCAN_ERR_DEVICE = 8       /* no usable sm_100-family device is current */
} m2scan_status;

/*
 * Forward pass: writes h_enriched [B,SH2].
 *   h_history [B,K,SH2], h_s2 [B,SH2]: inputs.
 *   W_A, W_B, W_C [SH2,D], W_O [D,SH2]: weights; tw: scalar blend weight.
 * One fused kernel launch (none when B == 0).
 */
m2scan_status m2scan_fwd(const float* h_history, const float* h_s2, const float* W_A,
                         const float* W_B, const float* W_C, const float* W_O, float tw,
                         int64_t B, int32_t K, int32_t SH2, int32_t D, float* h_enriched,
                         m2scan_stream_t stream);

/*
 * Bytes of device workspace m2scan_bwd needs for these shapes: the per-slot
 * partial sums of the four weight gradients (min(B,152) slots of 4*SH2*D
 * floats); for the wide-state shapes (D = 64, SH2 % 128 == 0, K <= 128,
 * B*K < 2^31) those slots plus dA|dB (B*K*2D floats) and [dC | ctx] (B*2D
 * floats). Depends on the shapes only. Returns 0 for invalid shapes.
 */
size_t m2scan_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2, int32_t D);

/*
 * Backward pass. Inputs as for m2scan_fwd plus d_h_enriched [B,SH2] (the
 * upstream gradient dL/dh_enriched). Writes d_h_history [B,K,SH2],
 * d_h_s2 [B,SH2], dW_A, dW_B, dW_C [SH2,D] and dW_O [D,SH2].
 * `workspace` is caller-owned device scratch of at least
 * m2scan_bwd_workspace_bytes(B,K,SH2,D) bytes (16-byte aligned); its contents
 * on entry do not matter and are garbage on exit. It must not overlap any
 * input or output. The projections and the scan are recomputed from the
 * inputs (nothing is saved by the forward). Two kernel launches: the fused
 * backward and the fixed-order reduction of the weight-gradient slots; the
 * wide-state shapes (D = 64, SH2 % 128 == 0) take five: the weights' split
 * into tf32 parts and remainders, the tile kernel, d_h_s2, the
 * weight-gradient products and the slot reduction (m2scan_last_launch_count
 * reports the number). When B == 0 the weight
 * gradients are zero-filled with cudaMemsetAsync.
 */
m2scan_status m2scan_bwd(const float* h_history, const float* h_s2, const float* W_A,
                         const float* W_B, const float* W_C, const float* W_O, float tw,
                         const float* d_h_enriched, int64_t B, int32_t K, int32_t SH2,
                         int32_t D, float* d_h_history, float* d_h_s2, float* dW_A,
                         float* dW_B, float* dW_C, float* dW_O, void* workspace,
                         size_t workspace_bytes, m2scan_stream_t stream);

/*
 * The layer with the pages' optional gate multiplier ("Custom Kernel
 * Optimization Implementation Plan", Task 1: gate *= isv_signals[11] when
 * that signal is present; Task 2 carries the same factor into the reverse
 * scan): every gate becomes g * sigmoid(A_t), so
 *     x_t = g * sigmoid(A_t) * x_{t-1} + B_t,
 *     dA_t = dx * x_{t-1} * g * sigmoid'(A_t),  dx <- dx * g * sigmoid(A_t).
 * `gate_scale` is a DEVICE pointer to the one float g (4-byte aligned; read by
 * the kernels, so it may change between calls without a host
 * synchronisation), or NULL for g = 1, which is exactly m2scan_fwd /
 * m2scan_bwd. g gets no gradient. It must not overlap any output. Every other
 * argument, check and result is as for m2scan_fwd / m2scan_bwd.
 */
m2scan_status m2scan_fwd_ex(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                            int32_t D, float* h_enriched, m2scan_stream_t stream);
m2scan_status m2scan_bwd_ex(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* gate_scale, const float* d_h_enriched, int64_t B,
                            int32_t K, int32_t SH2, int32_t D, float* d_h_history,
                            float* d_h_s2, float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                            void* workspace, size_t workspace_bytes, m2scan_stream_t stream);

/*
 * Forward pass with bf16 activations ("bf16 inputs/outputs with fp32
 * accumulation", which halves the bytes of this memory-bound pass):
 * h_history [B,K,SH2] and h_s2 [B,SH2] are bfloat16 (raw 16-bit words, device,
 * 16-byte aligned), the weights fp32 as for m2scan_fwd, h_enriched [B,SH2]
 * bfloat16 (the fp32 result rounded to nearest even). Every product and sum
 * is fp32; the projections use W split into two bf16 parts (16 significant
 * bits, against the output's 8). gate_scale as for m2scan_fwd_ex. Shapes:
 * D = 16, SH2 % 64 == 0, SH2 <= 256, K <= 128; others return
 * M2SCAN_ERR_UNSUPPORTED. One kernel launch (none when B == 0).
 */
m2scan_status m2scan_fwd_bf16(const void* h_history, const void* h_s2, const float* W_A,
                              const float* W_B, const float* W_C, const float* W_O, float tw,
                              const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                              int32_t D, void* h_enriched, m2scan_stream_t stream);

/*
 * Backward pass with bf16 activations, the counterpart of m2scan_fwd_bf16:
 * h_history [B,K,SH2], h_s2 [B,SH2] and d_h_enriched [B,SH2] are bfloat16
 * inputs, d_h_history [B,K,SH2] and d_h_s2 [B,SH2] bfloat16 outputs (the fp32
 * results rounded to nearest even); weights and the weight gradients dW_A,
 * dW_B, dW_C, dW_O are fp32 as for m2scan_bwd, and every product and sum is
 * fp32 (the bf16 inputs are exact in fp32). gate_scale, workspace (at least
 * m2scan_bwd_workspace_bytes(B, K, SH2, D)), the ownership, alignment and
 * aliasing rules and the status codes are those of m2scan_bwd_ex, with the
 * activation spans counted in 2-byte elements. Any shape m2scan_bwd accepts
 * whose per-sample tile (4 * (2 * K * D + 2 * SH2 + 4 * D) bytes) fits the
 * device's shared memory; larger ones return M2SCAN_ERR_UNSUPPORTED.
 * For D = 16, SH2 % 64 == 0, SH2 <= 256, K <= 128 (and B * K < 2^31) it
 * runs a tensor-core kernel (bf16 products of the exact bf16 activations with
 * the fp32 factors split into three bf16 parts, fp32 accumulation); other
 * shapes run the per-sample generic kernel. Then the fixed-order slot sum:
 * two launches (none when B == 0, where the weight gradients are zeroed).
 * Weight gradients are bit-identical run to run.
 */
m2scan_status m2scan_bwd_bf16(const void* h_history, const void* h_s2, const float* W_A,
                              const float* W_B, const float* W_C, const float* W_O, float tw,
                              const float* gate_scale, const void* d_h_enriched, int64_t B,
                              int32_t K, int32_t SH2, int32_t D, void* d_h_history, void* d_h_s2,
                              float* dW_A, float* dW_B, float* dW_C, float* dW_O, void* workspace,
                              size_t workspace_bytes, m2scan_stream_t stream);

/*
 * The layer with the pages' own output step ("Custom Kernel Optimization
 * Implementation Plan", Task 1 Step 3) in place of tw * (ctx . W_O): one
 * scalar context per sample blended into every feature with a per-feature
 * temporal weight w and a 1/D scale,
 *     h_enriched[b, j] = h_s2[b, j] + w[j] * (sum_s C[b, s] x_{K-1}[b, s]) / D.
 *   temporal_weight: w [SH2] (device, 16-byte aligned), or NULL for w = 1.
 *   gate_scale: as for m2scan_fwd_ex (NULL: none).
 * It runs the layer's kernels with tw = 1 and W_O[s, j] = w[j] / D, which a
 * small kernel writes into the workspace first (one more launch):
 *   m2scan_fwd_blend workspace >= m2scan_blend_fwd_workspace_bytes(SH2, D).
 * The backward returns d_h_history, d_h_s2, dW_A, dW_B, dW_C as m2scan_bwd
 * does and, when d_temporal_weight is not NULL, dw [SH2] =
 * sum_b dY[b, j] * context_b / D (the gradient of that W_O folded back onto
 * w, states added in order: one more launch);
 *   m2scan_bwd_blend workspace >= m2scan_blend_bwd_workspace_bytes(B,K,SH2,D)
 * (m2scan_bwd's workspace plus two D x SH2 scratch arrays). Other arguments,
 * checks and conventions as for m2scan_fwd / m2scan_bwd; the workspace must
 * not overlap anything else.
 */
size_t m2scan_blend_fwd_workspace_bytes(int32_t SH2, int32_t D);
size_t m2scan_blend_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2, int32_t D);
m2scan_status m2scan_fwd_blend(const float* h_history, const float* h_s2, const float* W_A,
                               const float* W_B, const float* W_C, const float* temporal_weight,
                               const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                               int32_t D, float* h_enriched, void* workspace,
                               size_t workspace_bytes, m2scan_stream_t stream);
m2scan_status m2scan_bwd_blend(const float* h_history, const float* h_s2, const float* W_A,
                               const float* W_B, const float* W_C, const float* temporal_weight,
                               const float* gate_scale, const float* d_h_enriched, int64_t B,
                               int32_t K, int32_t SH2, int32_t D, float* d_h_history,
                               float* d_h_s2, float* dW_A, float* dW_B, float* dW_C,
                               float* d_temporal_weight, void* workspace, size_t workspace_bytes,
                               m2scan_stream_t stream);

/*
 * Backward pass for callers that cannot allocate device memory themselves:
 * code running where the device allocator belongs to someone else (a host
 * framework whose memory pool must account for every byte), latency-critical
 * paths that cannot afford cudaMalloc's implicit device synchronisation, and
 * minimal C hosts that only own the tensors they pass in. The pages have no
 * counterpart of this call; it is a packaging variant of m2scan_bwd.
 *
 * Same arguments and results as m2scan_bwd, without `workspace`: the
 * weight-gradient slots live in a static array of
 * M2SCAN_NOALLOC_SCRATCH_BYTES bytes that every GPU loading this library
 * holds until the process exits. The call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine); the caller still passes every
 * input and output. Shapes whose slots need more than
 * M2SCAN_NOALLOC_SCRATCH_BYTES (m2scan_bwd_workspace_bytes > the maximum)
 * return M2SCAN_ERR_WORKSPACE without launching anything.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, a synchronous runtime call); make that first
 * call before any stream capture. Every call on a device shares the one
 * array and nothing in it needs to start at zero, but calls that overlap on
 * the GPU (different streams, or different host threads, without ordering
 * between them) race on it and produce wrong weight gradients.
 */
#define M2SCAN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
m2scan_status m2scan_bwd_noalloc(const float* h_history, const float* h_s2, const float* W_A,
                                 const float* W_B, const float* W_C, const float* W_O,
                                 float tw, const float* d_h_enriched, int64_t B, int32_t K,
                                 int32_t SH2, int32_t D, float* d_h_history, float* d_h_s2,
                                 float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                                 m2scan_stream_t stream);

/*
 * Bias gradient of a fully connected layer ("Phase 3 Kernel Optimization
 * Implementation Plan", Tasks 2 and 3): the column sums of a row-major fp32
 * matrix dy [N, C],
 *     db[c] = sum over r = 0 .. N-1 of dy[r, c]           (accumulate == 0)
 *     db[c] = db[c] + sum over r of dy[r, c]              (accumulate != 0)
 * The pages use both: their main backward adds into db, their curiosity
 * trainer overwrites grad_b.
 *   dy [N, C] (device, 16-byte aligned; rows need not be): input, N >= 0,
 *       C >= 1, N * C <= 2^40.
 *   db [C] (device, 16-byte aligned): output, read too when accumulating.
 *   workspace: caller-owned device scratch of at least
 *       m2scan_bias_grad_workspace_bytes(N, C) bytes, 16-byte aligned, for
 *       the per-block partial sums; contents on entry do not matter. May be
 *       NULL when N == 0.
 * None of dy, db and workspace may overlap. Two kernel launches: partial
 * sums of fixed row ranges (the split depends on N only), then their sum in
 * range order, so db is bit-identical from run to run. N == 0: db is
 * zero-filled with cudaMemsetAsync (or left alone when accumulating).
 * Same error conventions as the layer calls (host checks, nothing launched
 * on failure).
 */
size_t m2scan_bias_grad_workspace_bytes(int64_t N, int32_t C);
m2scan_status m2scan_bias_grad(const float* dy, int64_t N, int32_t C, float* db,
                               int32_t accumulate, void* workspace, size_t workspace_bytes,
                               m2scan_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* m2scan_status_str(m2scan_status status);

/* cudaError_t value of the last failing CUDA call made by the library on the
 * calling thread (0 if none). */
int m2scan_last_cuda_error(void);

/* Kernel path selection for tests: 0 = automatic (default), 1 = always use the
 * generic fallback kernels. Process-wide; returns the previous value. */
int m2scan_set_force_generic(int force);

/* Which kernel family m2scan_bwd would launch for these shapes (any B >= 1
 * with B * K < 2^31): 1 = fused tensor-core kernels (the fast path), 2 =
 * generic fallback, 3 = wide-state tensor-core kernels (D = 64,
 * SH2 % 128 == 0, K <= 128), 0 = unsupported shape. Host-only: needs no GPU. */
int m2scan_path_for(int32_t K, int32_t SH2, int32_t D);

/* The same for m2scan_fwd. */
int m2scan_fwd_path_for(int32_t K, int32_t SH2, int32_t D);

/*
 * Device-side error flags of the current device (bit 0: a kernel gave up
 * waiting on a shared-memory barrier after its time limit). While bit 0 is
 * set, kernels that would have to wait give up at once, so every result
 * computed after the first failure is garbage until the flags are read.
 * Reading is SYNCHRONOUS (it waits for the device) and clears the flags.
 * Returns M2SCAN_OK and stores the flags in *flags.
 */
m2scan_status m2scan_read_device_flags(uint32_t* flags);

/*
 * Self-test of the time limit on the kernels' barrier waits (no counterpart
 * on the pages; it exercises the failure path that m2scan_read_device_flags
 * reports). Launches one small kernel that waits twice, with a limit of
 * `limit_ns` nanoseconds (1 us to 100 ms), on a shared-memory barrier that
 * nothing ever arrives on. The first wait gives up after the limit and sets
 * bit 0 of the device error flags; the second then gives up at its first
 * check of that bit. Nothing faults or hangs. `out` is a DEVICE pointer to
 * three uint64 values (16-byte aligned): the nanoseconds each wait took and a
 * mask (bit 0 / bit 1: the first / second wait gave up). Asynchronous on
 * `stream`. Afterwards bit 0 of the flags is set, so kernels that would have
 * to wait give up at once: read (and so clear) the flags with
 * m2scan_read_device_flags before launching anything else.
 */
m2scan_status m2scan_selftest_wait_timeout(uint64_t limit_ns, uint64_t* out,
                                           m2scan_stream_t stream);

/* Number of CUDA kernels launched by the most recent successful call of
 * m2scan_fwd, m2scan_bwd (or their _ex forms) or m2scan_bias_grad on the
 * calling thread. */
int m2scan_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* M2SCAN_H */
