/*
 * gbln.h -- C ABI of the GB300 (sm_103a) layer-operator library libgbln.so.
 *
 * Operators: RMSNorm with fused residual add (forward, backward, weight-gradient
 * finalize), rotary position embedding on Q and K (forward, backward, cos/sin
 * table, per-document positions) and SwiGLU (forward, backward); LayerNorm,
 * other gated and plain activations, and MXFP8 outputs for the next GEMM.
 *
 * Sources that name these operators (they print no formulas; the standard
 * definitions are used and written out at each entry point):
 *   [FL]  "Fast-LLM: 高效大语言模型训练框架", §三 技术架构: table "Transformer Block
 *         结构" (Normalization LayerNorm / RMSNorm; attention + RoPE; MLP gated or
 *         not, SiLU / GeLU / ReLU) and "训练配置示例" (rms_norm with epsilon;
 *         rotary type default with theta; gated MLP with activation silu;
 *         micro_batch_size in tokens with maximum_document_length).
 *   [LF]  "LLaMA-Factory Kernels 系统": the fused RMSNorm, SwiGLU and RoPE operators.
 *   [HF]  "Kernels（自定义内核）", §Liger: RMSNorm, RoPE and SwiGLU fused into single
 *         kernels for training; fusion saves memory traffic and launches.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: every pointer is DEVICE memory on the current CUDA device, owned and
 *    allocated by the caller.  The library never allocates and never frees.  Its
 *    only state is per device: the SM count, the device error word, flags that
 *    record which kernels' shared-memory limits have been raised, and the fixed
 *    scratch array of gbln_rmsnorm_bwd_noalloc.  It tracks 64 devices: on a
 *    device with ordinal 64 or above, the calls that need that state (the
 *    backward passes, RoPE, the gated units and activations, the error word)
 *    return GBLN_ERR_CUDA.  That state is looked up once per device and kept for
 *    the life of the process, so the device's primary context must not be torn
 *    down (cudaDeviceReset, or the driver API's primary-context reset) while the
 *    library is in use: after a reset the cached addresses (error word, scratch
 *    array) and shared-memory limits no longer hold.
 *  - Layout: row-major and contiguous.  "[T, H]" means T rows of H elements.
 *  - Streams: work is enqueued on `stream` (NULL = the legacy default stream) and
 *    the call returns without synchronising.  Errors raised by the kernels
 *    themselves appear on the stream, not in the returned status.
 *  - CUDA graphs: every call can be captured.  The first call of an entry point
 *    on a device does one-time set-up (SM count, the device error word's
 *    address, kernel shared-memory limits); make that first call outside
 *    stream capture.
 *  - Types: `io` is the element type of activations and gradients, `wt` the type
 *    of the RMSNorm weight.  Supported: io = wt = F32; io = wt = BF16;
 *    io = BF16 with wt = F32.  Arithmetic is float32; bf16 results are rounded
 *    to nearest even once.
 *  - Alignment: any alignment is accepted.  Pointers aligned to 16 bytes with
 *    row widths that are a multiple of 16 bytes take the 128-bit vector path;
 *    anything else takes a slower element-wise path of the same kernels.
 *  - Errors: arguments are checked on the host before any CUDA call.  A null
 *    required pointer, a negative or out-of-range size, eps < 0 or not finite,
 *    an odd head size, theta <= 0, or a workspace that is too small returns an
 *    error and launches nothing.  T == 0 returns GBLN_OK and launches nothing
 *    once sizes, scalars and dtypes pass; its pointers are not examined (empty
 *    tensors may have null data pointers).  A failed launch returns GBLN_ERR_CUDA.
 *  - Aliasing: outputs may alias their own input exactly where an entry point
 *    says so; partial overlap is undefined.
 */
#ifndef GBLN_H
#define GBLN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so that no CUDA header is needed. */
typedef struct CUstream_st* gbln_stream_t;

typedef enum {
  GBLN_OK = 0,
  GBLN_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad scalar                */
  GBLN_ERR_UNSUPPORTED = 2, /* dtype combination outside the supported set       */
  GBLN_ERR_WORKSPACE = 3,   /* dW partial workspace smaller than required        */
  GBLN_ERR_CUDA = 4         /* a CUDA runtime call or launch failed              */
} gbln_status;

typedef enum { GBLN_F32 = 0, GBLN_BF16 = 1 } gbln_dtype;

/* Activation of the gated and plain MLP units ([FL] 支持的 MLP 变体: SiLU / GeLU / ReLU). */
typedef enum {
  GBLN_ACT_SILU = 0,      /* x / (1 + exp(-x))                                    */
  GBLN_ACT_GELU_TANH = 1, /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))       */
  GBLN_ACT_GELU_ERF = 2,  /* 0.5 x (1 + erf(x / sqrt(2)))  (exact GeLU)             */
  GBLN_ACT_RELU = 3       /* max(x, 0); derivative 1 for x > 0, else 0              */
} gbln_act;

/* Human-readable name of a status code.  Never NULL; the string is static. */
const char* gbln_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int gbln_version(void);

/*
 * Per-device error word of the current device, a set of bits:
 *   1  a kernel's bounded wait on its own asynchronous (TMA bulk) copies ran
 *      out; the kernel stopped early instead of hanging, so its outputs are
 *      incomplete;
 *   2  a RoPE call met a position outside [0, max_pos); that token's outputs
 *      are NaN (the table is not read).
 * *code receives the word; clear != 0 resets it to zero.  Synchronous
 * (device-wide copy): call it outside hot loops.  Errors: INVALID_ARG for a
 * null code, CUDA if the device is unreachable.
 */
gbln_status gbln_device_error(uint32_t* code, int clear);

/*
 * Self-test of the timeout path: launches one thread that waits, with the
 * bounded poll loop of the TMA pipelines, on a barrier nothing completes; after
 * `polls` polls (1 <= polls <= 2^22) it sets bit 1 of the device error word and
 * returns.  Touches no caller memory; the context stays usable.  For tests.
 */
gbln_status gbln_selftest_wait_timeout(uint32_t polls, gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* RMSNorm with fused residual add ([FL] Transformer Block 结构, 训练配置示例;  */
/* [LF] fused RMSNorm; [HF] §Liger)                                          */
/* ------------------------------------------------------------------------- */

/*
 * Forward, per row t of T rows of H channels:
 *   h[t]    = x[t] + residual[t]           (rounded to io; h = x when residual is NULL)
 *   rstd[t] = 1 / sqrt(mean_j h[t,j]^2 + eps)
 *   y[t,j]  = weight[j] * h[t,j] * rstd[t]  (one rounding to io)
 *
 * x, residual      [T, H] io, read.  residual may be NULL (plain RMSNorm).
 * weight           [H] wt, read.
 * y                [T, H] io, written.
 * residual_out     [T, H] io, written with h.  Required iff residual != NULL,
 *                  ignored otherwise.  May alias x or residual exactly.
 * rstd             [T] float32, written; the backward pass reads it.
 * eps              >= 0 and finite.
 * Errors: INVALID_ARG for null x/weight/y/rstd, T < 0, H <= 0, H > 2^24, bad eps,
 *         missing residual_out; UNSUPPORTED for other dtype pairs.
 */
gbln_status gbln_rmsnorm_fwd(const void* x, const void* residual, const void* weight,
                             void* y, void* residual_out, float* rstd,
                             int64_t T, int64_t H, float eps,
                             gbln_dtype io, gbln_dtype wt, gbln_stream_t stream);

/*
 * Rows of the float32 weight-gradient workspace that gbln_rmsnorm_bwd writes
 * for this shape on the current device: the workspace is [P, H] float32.
 * P depends only on (T, H, io) and the device's SM count, so a fixed shape on a
 * fixed GPU model always uses the same P and the same summation order.
 * Returns P >= 1 for T >= 1, 0 for T == 0, and -1 on invalid arguments or when
 * the device cannot be queried.
 */
int64_t gbln_rmsnorm_bwd_num_partials(int64_t T, int64_t H, gbln_dtype io);

/*
 * Backward, first of two passes.  With n = h * rstd and g = dy * weight, per row:
 *   dx[t]  = rstd[t] * (g - n * mean_j(g[j] * n[j])) + dresidual_out[t]
 *   partial[p, j] = sum over the rows of block p of dy[t,j] * n[t,j]
 * dx is the gradient of both x and residual of the forward call.
 *
 * dy               [T, H] io, gradient of y.
 * dresidual_out    [T, H] io, gradient arriving on residual_out; NULL = zero.
 * h                [T, H] io, the forward's residual_out (or x if it had no residual).
 * weight           [H] wt.   rstd [T] float32 from the forward.
 * dx               [T, H] io, written.  May alias dy or dresidual_out exactly.
 * dw_partial       [P_cap, H] float32 workspace, rows 0..P-1 written, where
 *                  P = gbln_rmsnorm_bwd_num_partials(T, H, io).
 * P_cap            rows available in dw_partial; GBLN_ERR_WORKSPACE if P_cap < P.
 * The rows of a block and their order are fixed by (T, H, io, SM count): the
 * result is bitwise reproducible run to run.
 */
gbln_status gbln_rmsnorm_bwd(const void* dy, const void* dresidual_out, const void* h,
                             const void* weight, const float* rstd,
                             void* dx, float* dw_partial, int64_t P_cap,
                             int64_t T, int64_t H,
                             gbln_dtype io, gbln_dtype wt, gbln_stream_t stream);

/*
 * Backward, second pass: dw[j] = (accumulate ? dw[j] : 0) + sum_{p<P} partial[p, j],
 * summed in a fixed order (bitwise reproducible).
 * dw_partial [P, H] float32 as written by gbln_rmsnorm_bwd, P exactly the value
 * gbln_rmsnorm_bwd_num_partials returned for that call.  dw [H] float32.
 */
gbln_status gbln_rmsnorm_dw_finalize(const float* dw_partial, int64_t P, int64_t H,
                                     float* dw, int accumulate, gbln_stream_t stream);

/*
 * Backward without a caller-provided workspace: dx as gbln_rmsnorm_bwd, and the
 * finished weight gradient dw [H] float32 (as gbln_rmsnorm_dw_finalize with
 * accumulate = 0), in two launches on `stream`.  The sources have no
 * counterpart of this entry point; it exists for callers that cannot allocate
 * device memory where they run the backward pass (a region being recorded into
 * a CUDA graph under a capture mode that forbids cudaMalloc, a runtime whose
 * device memory belongs to a pool it may not bypass, a latency-critical loop in
 * which an allocation could synchronise the device).  The caller still passes
 * every input and output.
 *
 * Scratch: the dW partial rows live in one fixed array inside the library
 * (4 Mi float32 = 16 MiB, held by every GPU that loads the library until the
 * process exits).  Every call on a device uses the same array and overwrites the
 * rows it reads, so nothing needs clearing; calls that may overlap on the GPU
 * (other streams, other threads) race on it and must be serialised by the caller.
 * The usual number of partial rows is reduced when it would not fit, so the
 * summation order (still fixed for a shape and GPU) can differ from
 * gbln_rmsnorm_bwd's by float32 rounding.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  The address is kept until the process exits: resetting
 * the device's primary context (cudaDeviceReset) while the library is loaded
 * moves the array, and later calls would write through the stale address, so
 * do not reset a device that this entry point has been called on.
 * Errors: as gbln_rmsnorm_bwd; GBLN_ERR_WORKSPACE if H > 4 Mi (a partial row
 * would not fit); GBLN_ERR_CUDA if the address lookup fails.  T == 0 sets dw to
 * zero (one launch).  dx may alias dy or dresidual_out exactly.
 */
gbln_status gbln_rmsnorm_bwd_noalloc(const void* dy, const void* dresidual_out, const void* h,
                                     const void* weight, const float* rstd,
                                     void* dx, float* dw, int64_t T, int64_t H,
                                     gbln_dtype io, gbln_dtype wt, gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* LayerNorm with fused residual add ([FL] Transformer Block 结构:             */
/* normalization LayerNorm / RMSNorm)                                         */
/* ------------------------------------------------------------------------- */

/*
 * Forward, per row t of H channels:
 *   h = x + residual (rounded to io; h = x when residual is NULL)
 *   mean[t] = mean_j h;  var = mean_j (h - mean)^2;  rstd[t] = 1 / sqrt(var + eps)
 *   y = weight * (h - mean) * rstd + bias  (bias NULL = no bias; one rounding to io)
 * Arguments as gbln_rmsnorm_fwd, plus bias [H] wt (nullable) and mean [T] float32
 * (written; the backward pass reads it with rstd).
 */
gbln_status gbln_layernorm_fwd(const void* x, const void* residual, const void* weight,
                               const void* bias, void* y, void* residual_out, float* mean,
                               float* rstd, int64_t T, int64_t H, float eps, gbln_dtype io,
                               gbln_dtype wt, gbln_stream_t stream);

/* Rows P of the [P, 2H] float32 dW|dB workspace of gbln_layernorm_bwd (as gbln_rmsnorm_bwd_num_partials). */
int64_t gbln_layernorm_bwd_num_partials(int64_t T, int64_t H, gbln_dtype io);

/*
 * Backward, first pass.  With n = (h - mean) * rstd and g = dy * weight, per row:
 *   dx = rstd * (g - mean_j g - n * mean_j(g * n)) + dresidual_out
 *   partial[p, 0:H]  = sum over the rows of block p of dy * n   (dW)
 *   partial[p, H:2H] = sum over the rows of block p of dy       (dB)
 * Arguments as gbln_rmsnorm_bwd, plus mean [T] from the forward; the workspace is
 * [P_cap, 2H] float32.  Bitwise reproducible for a fixed shape and GPU model.
 */
gbln_status gbln_layernorm_bwd(const void* dy, const void* dresidual_out, const void* h,
                               const void* weight, const float* mean, const float* rstd,
                               void* dx, float* dwdb_partial, int64_t P_cap, int64_t T, int64_t H,
                               gbln_dtype io, gbln_dtype wt, gbln_stream_t stream);

/* Second pass: dw[j] (+)= sum_p partial[p, j], db[j] (+)= sum_p partial[p, H + j], fixed order. */
gbln_status gbln_layernorm_dwdb_finalize(const float* dwdb_partial, int64_t P, int64_t H,
                                         float* dw, float* db, int accumulate,
                                         gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Rotary position embedding on Q and K ([FL] attention with RoPE, rotary     */
/* type default with theta; [LF] fused RoPE; [HF] §Liger)                     */
/* ------------------------------------------------------------------------- */

/*
 * Cos/sin table: cos_sin[p, i] = (cos(p * f_i), sin(p * f_i)) as two float32,
 * f_i = theta^(-2 i / D), for p in [0, max_pos) and i in [0, D/2).  Angles and
 * their cosines are evaluated in double precision on the device and rounded once
 * to float32.  cos_sin: [max_pos, D/2, 2] float32, written.
 * Errors: INVALID_ARG for null, max_pos < 0, D <= 0 or odd, theta <= 0 or not finite.
 */
gbln_status gbln_rope_table(float* cos_sin, int64_t max_pos, int32_t D, double theta,
                            gbln_stream_t stream);

/*
 * Forward rotation, rotate-half pairing.  For every token t, every head of q and
 * of k, and i < D/2, with (c, s) = cos_sin[positions[t], i]:
 *   out[i]       = x[i] * c - x[i + D/2] * s
 *   out[i + D/2] = x[i + D/2] * c + x[i] * s
 * q [T, Hq, D], k [T, Hk, D] io, read; q_out, k_out same shapes, written (may
 * alias q and k exactly: in place).  Hk may be 0 (k, k_out ignored).
 * positions [T] int32: the position of each token inside its document.  A position
 * outside [0, max_pos) is not read from the table: that token's outputs are NaN.
 * cos_sin as written by gbln_rope_table for the same D and some max_pos.
 */
gbln_status gbln_rope_fwd(const void* q, const void* k, void* q_out, void* k_out,
                          const int32_t* positions, const float* cos_sin, int64_t max_pos,
                          int64_t T, int32_t Hq, int32_t Hk, int32_t D,
                          gbln_dtype io, gbln_stream_t stream);

/*
 * Backward: the transpose (= inverse) rotation applied to the incoming gradients:
 *   din[i]       = dout[i] * c + dout[i + D/2] * s
 *   din[i + D/2] = dout[i + D/2] * c - dout[i] * s
 * Same arguments as gbln_rope_fwd with (dq, dk) in and (dq_in, dk_in) out.
 */
gbln_status gbln_rope_bwd(const void* dq, const void* dk, void* dq_in, void* dk_in,
                          const int32_t* positions, const float* cos_sin, int64_t max_pos,
                          int64_t T, int32_t Hq, int32_t Hk, int32_t D,
                          gbln_dtype io, gbln_stream_t stream);

/* Pairing of the rotated elements. */
typedef enum {
  GBLN_ROPE_HALF = 0,       /* (i, i + D/2): the default rotary type (gbln_rope_fwd)   */
  GBLN_ROPE_INTERLEAVED = 1 /* (2i, 2i + 1), frequency index i                        */
} gbln_rope_pairing;

/*
 * gbln_rope_fwd with strided rows and a choice of pairing: head row h of token t
 * of q starts at q + t * ld_q + h * D (elements), likewise for k, q_out, k_out
 * (ld_q, ld_q_out >= Hq * D; ld_k, ld_k_out >= Hk * D).  Q and K can thus be read
 * from, and written back into, one packed [T, (Hq + 2 Hk) * D] QKV projection
 * output (q = qkv, k = qkv + Hq * D, every ld = (Hq + 2 Hk) * D; in place with
 * q_out = q, k_out = k).  Interleaved pairing rotates elements (2i, 2i + 1) by
 * pos * theta^(-2i/D) with the same cos/sin table.  Errors as gbln_rope_fwd, plus
 * INVALID_ARG for a stride below its row width or an unknown pairing.
 */
gbln_status gbln_rope_fwd_ex(const void* q, const void* k, void* q_out, void* k_out,
                             const int32_t* positions, const float* cos_sin, int64_t max_pos,
                             int64_t T, int32_t Hq, int32_t Hk, int32_t D, int64_t ld_q,
                             int64_t ld_k, int64_t ld_q_out, int64_t ld_k_out,
                             gbln_rope_pairing pairing, gbln_dtype io, gbln_stream_t stream);

/* Backward of gbln_rope_fwd_ex (inverse rotation), same layout arguments. */
gbln_status gbln_rope_bwd_ex(const void* dq, const void* dk, void* dq_in, void* dk_in,
                             const int32_t* positions, const float* cos_sin, int64_t max_pos,
                             int64_t T, int32_t Hq, int32_t Hk, int32_t D, int64_t ld_dq,
                             int64_t ld_dk, int64_t ld_dq_in, int64_t ld_dk_in,
                             gbln_rope_pairing pairing, gbln_dtype io, gbln_stream_t stream);

/*
 * Positions of packed documents: positions[t] = t - cu_seqlens[d] for the document
 * d with cu_seqlens[d] <= t < cu_seqlens[d+1] ([FL] 训练配置示例: micro-batches
 * counted in tokens hold several documents of at most maximum_document_length).
 * cu_seqlens [ndoc + 1] int32, non-decreasing, cu_seqlens[0] = 0 and
 * cu_seqlens[ndoc] = T (caller's contract: violating it gives wrong but in-bounds
 * results).  positions [T] int32, written.
 */
gbln_status gbln_positions_from_cu_seqlens(const int32_t* cu_seqlens, int32_t ndoc,
                                           int32_t* positions, int64_t T,
                                           gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* SwiGLU ([FL] 支持的 MLP 变体, 训练配置示例 gated + silu; [LF] fused SwiGLU;   */
/* [HF] §Liger)                                                              */
/* ------------------------------------------------------------------------- */

/*
 * out = silu(gate) * up = gate / (1 + exp(-gate)) * up, elementwise.
 * gate, up, out: [T, I] io.  out may alias gate or up exactly.
 */
gbln_status gbln_swiglu_fwd(const void* gate, const void* up, void* out,
                            int64_t T, int64_t I, gbln_dtype io, gbln_stream_t stream);

/*
 * With s = sigmoid(gate):
 *   dgate = dout * up * s * (1 + gate * (1 - s))
 *   dup   = dout * gate * s
 * dout, gate, up: [T, I] io, read.  dgate, dup: [T, I] io, written; dgate may
 * alias gate and dup may alias up exactly (in place).
 */
gbln_status gbln_swiglu_bwd(const void* dout, const void* gate, const void* up,
                            void* dgate, void* dup,
                            int64_t T, int64_t I, gbln_dtype io, gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Gated units with any activation and row strides; plain activations          */
/* ([FL] 支持的 MLP 变体: dense MLP gated or not, SiLU / GeLU / ReLU)           */
/* ------------------------------------------------------------------------- */

/*
 * out[t, j] = f(gate[t, j]) * up[t, j] for t < T, j < I, f = act (see gbln_act).
 * Row t of each tensor starts ld elements after row t - 1 (ld >= I), so gate and
 * up may be the two halves of one packed [T, 2I] projection output
 * (gate = p, up = p + I, ld_gate = ld_up = 2I).  With every ld = I and
 * act = GBLN_ACT_SILU this is gbln_swiglu_fwd.  out may alias gate or up exactly.
 * Errors: INVALID_ARG for a bad act, T < 0, I <= 0, ld < I, null pointers (T > 0).
 */
gbln_status gbln_glu_fwd(const void* gate, const void* up, void* out, int64_t T, int64_t I,
                         int64_t ld_gate, int64_t ld_up, int64_t ld_out, gbln_act act,
                         gbln_dtype io, gbln_stream_t stream);

/*
 * dgate = dout * up * f'(gate), dup = dout * f(gate), each with its own row
 * stride (a packed [T, 2I] gradient: dgate = q, dup = q + I, ld = 2I).  dgate may
 * alias gate and dup may alias up exactly.  Errors as gbln_glu_fwd.
 */
gbln_status gbln_glu_bwd(const void* dout, const void* gate, const void* up, void* dgate,
                         void* dup, int64_t T, int64_t I, int64_t ld_dout, int64_t ld_gate,
                         int64_t ld_up, int64_t ld_dgate, int64_t ld_dup, gbln_act act,
                         gbln_dtype io, gbln_stream_t stream);

/* y = f(x) over n contiguous elements (non-gated MLP); y may alias x. */
gbln_status gbln_act_fwd(const void* x, void* y, int64_t n, gbln_act act, gbln_dtype io,
                         gbln_stream_t stream);

/* dx = dy * f'(x) over n contiguous elements; dx may alias dy or x. */
gbln_status gbln_act_bwd(const void* dy, const void* x, void* dx, int64_t n, gbln_act act,
                         gbln_dtype io, gbln_stream_t stream);

/* ------------------------------------------------------------------------- */
/* MXFP8 outputs for the next projection GEMM ([HF] Kernels intro: fusing a    */
/* producer with its consumer's input conversion saves an HBM pass)            */
/* ------------------------------------------------------------------------- */

/*
 * MXFP8 as defined by the OCP Microscaling Formats (MX) v1.0 specification:
 * blocks of 32 consecutive values of a row share one scale 2^e, stored as an
 * E8M0 byte (e + 127); each value is stored as an E4M3 byte (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; largest finite 448).  Here
 *   e     = floor(log2(max |v| over the block)) - 8, clamped to [-127, 127]
 *           (-127 for an all-zero block),
 *   code  = E4M3(v / 2^e), rounded to nearest even, saturating to +-448.
 * Blocks run along the last axis, the reduction axis of the GEMM that
 * consumes the tensor (y @ W^T), which is the operand layout of block-scaled
 * FP8 tensor-core GEMMs.  Scales are stored row-major, [T, N / 32]; a GEMM
 * library that wants another arrangement of the scale bytes needs a permutation.
 * The quantised value is computed in float32 from the unrounded result.
 */

/*
 * gbln_rmsnorm_fwd with y also (or only) delivered as MXFP8:
 * y_e4m3 [T, H] bytes and y_scale [T, H / 32] bytes, both written.  y [T, H] io
 * may be NULL (then only the MXFP8 copy is written).  H must be a multiple of
 * 32.  Other arguments, aliasing and errors as gbln_rmsnorm_fwd; INVALID_ARG
 * also for H % 32 != 0 or a null y_e4m3 / y_scale.  Any alignment is accepted.
 */
gbln_status gbln_rmsnorm_fwd_mxfp8(const void* x, const void* residual, const void* weight,
                                   void* y, uint8_t* y_e4m3, uint8_t* y_scale,
                                   void* residual_out, float* rstd, int64_t T, int64_t H,
                                   float eps, gbln_dtype io, gbln_dtype wt,
                                   gbln_stream_t stream);

/*
 * Gated unit forward delivered as MXFP8 only: out = f(gate) * up (as
 * gbln_glu_fwd, with row strides ld_gate, ld_up >= I for packed [T, 2I] inputs)
 * written as out_e4m3 [T, I] bytes (contiguous) and out_scale [T, I / 32] bytes.
 * I must be a multiple of 32.  Errors as gbln_glu_fwd; INVALID_ARG also for
 * I % 32 != 0.  Any alignment is accepted.
 */
gbln_status gbln_glu_fwd_mxfp8(const void* gate, const void* up, uint8_t* out_e4m3,
                               uint8_t* out_scale, int64_t T, int64_t I, int64_t ld_gate,
                               int64_t ld_up, gbln_act act, gbln_dtype io,
                               gbln_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBLN_H */
