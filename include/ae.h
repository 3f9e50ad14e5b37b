/*
 * ae.h - C ABI of the GB300 flow-matching action-expert sampler.
 *
 * The library runs the action expert of a vision-language-action model for
 * n Euler steps of flow matching: starting from noise at t = 1, every step
 * evaluates a Gemma-style expert on the H action tokens of each request
 * (adaRMS conditioned on a sinusoidal time embedding, merged QKV, RoPE,
 * MQA/GQA attention over [valid prefix KV || action KV], gated residuals,
 * merged gate/up GeGLU MLP) and moves the actions by x <- x + delta * v with
 * delta = -1/n.  Sources, by page and section:
 *   - MolmoBot PR "Inference optimization for MolmoBot VLA: torch.compile +
 *     CUDA graphs + action-expert KV cache", Part 2: the VLM context is
 *     computed once per query and reused by every flow step.
 *   - LoongForge blog "How to Speed Up VLA Training Step by Step: A 3x
 *     Acceleration Case Study on Pi0.5", sections 1-3 and 5.3: the layer's
 *     ops, the prefix-LM mask, masked camera slots, pad tokens that do not
 *     advance positions, time MLP and action in/out projections.
 *   - sglang PR #34599 summary, implementation items 1-2: merged Q/K/V and
 *     gate/up weights; mask, positions and time scaling hoisted out of the
 *     step loop.
 *   - OxyGen, "Cross-task KV Sharing": one prefill's KV is read, not copied,
 *     by the action expert.
 *
 * Conventions common to every call:
 *   - Matrices are row-major [out, in] (a Linear's weight).  "T" below is the
 *     storage type chosen by ae_config.dtype: bf16 (AE_DTYPE_BF16) or fp32
 *     (AE_DTYPE_F32).  Flow state (noise, actions) is always fp32.
 *   - "device" pointers are CUDA device (or managed) memory of the device
 *     that was current when ae_create ran; "host" pointers are ordinary
 *     host memory.
 *   - Every call is stream-ordered on the context's stream and returns after
 *     enqueueing (ae_create and ae_destroy synchronize that stream).  A call
 *     that fails a host-side check returns at once and changes no state.
 *   - Device-side checks (bounds, bounded waits) set a sticky status that the
 *     next ae_sample returns as AE_ERR_DEVICE; ae_synchronize and
 *     ae_last_error report it too.  No call throws or aborts.
 *   - A context is not thread-safe; distinct contexts are independent.
 */
#ifndef AE_H_
#define AE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define AE_API __attribute__((visibility("default")))
#else
#define AE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ae_ctx ae_ctx;

typedef enum {
  AE_OK = 0,
  AE_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad enum     */
  AE_ERR_SHAPE = -2,       /* a size outside what the context supports      */
  AE_ERR_NOT_BOUND = -3,   /* ae_sample before a successful ae_bind_prefix  */
  AE_ERR_CUDA = -4,        /* a CUDA runtime call failed (see ae_last_error) */
  AE_ERR_DEVICE = -5,      /* a device-side check failed (sticky)           */
  AE_ERR_OOM = -6,         /* device memory allocation failed               */
  AE_ERR_UNSUPPORTED = -7  /* no GPU of compute capability 10.3 is current  */
} ae_status;

typedef enum { AE_DTYPE_BF16 = 0, AE_DTYPE_F32 = 1 } ae_dtype;

/*
 * Storage of the block Linears (wq, wk, wv, wo, wg, wu, wd of every layer).
 * AE_WEIGHTS_FP8_E4M3 (MolmoBot PR, Part 3: per-tensor dynamic fp8 on the
 * blocks' fused QKV, attention output, gate/up and down Linears; LoongForge
 * blog, section 7: TorchAO's tensorwise recipe, the result restored using the
 * scales): ae_create quantizes each of these tensors on its own, amax =
 * max |w|, s = fp32(448 / amax) (1 if amax == 0), code = E4M3(fp32(w * s))
 * with round-to-nearest-even and saturation at +-448 (the OCP "e4m3fn"
 * format: bias 7, subnormals, no infinities), and every GEMM output of the
 * tensor is multiplied by r = fp32(1 / s).  The library then holds the codes
 * (one byte per weight) instead of bf16 copies, halving the bytes every flow
 * step streams.  Activations, norms, the time MLP, the modulation, the
 * input/output and context projections stay bf16 / fp32.  bf16 contexts only
 * (AE_ERR_INVALID_ARG otherwise), with n_q_heads * head_dim and mlp multiples
 * of 128 (AE_ERR_SHAPE otherwise).
 */
typedef enum { AE_WEIGHTS_AS_DTYPE = 0, AE_WEIGHTS_FP8_E4M3 = 1 } ae_weight_format;

/* Limits checked by the host side of every call. */
#define AE_MAX_BATCH 64  /* requests per ae_bind_prefix                  */
#define AE_MAX_STEPS 128 /* Euler steps per ae_sample                    */

/*
 * Expert dimensions.  Requirements: every size > 0; n_q_heads % n_kv_heads
 * == 0; head_dim even, a multiple of 32 and <= 256; width and mlp multiples
 * of 32; width even (the time embedding is width/2 sines then width/2
 * cosines).  rms_eps is adaRMS's epsilon; rope_theta the RoPE base; the
 * time-embedding periods run geometrically from time_min_period to
 * time_max_period (LoongForge sections 2 and 5.3 name the sinusoidal time
 * embedding and the time MLP without printing their constants).
 */
typedef struct {
  int layers;      /* L  */
  int width;       /* D  */
  int mlp;         /* F  */
  int n_q_heads;   /* Hq */
  int n_kv_heads;  /* Hkv */
  int head_dim;    /* dh */
  int action_dim;  /* A  */
  int horizon;     /* H, action tokens per request */
  double rms_eps;
  double rope_theta;
  double time_min_period; /* double: the smallest period's angle reaches ~1.6e3 rad */
  double time_max_period;
  int dtype;       /* ae_dtype: storage type T of weights and prefix K/V */
  int ctx_dim;     /* C, width of the per-layer VLM hidden states that
                      ae_bind_context projects into K/V; 0 = no context
                      projection (w_ck / w_cv are then ignored) */
  int weight_format; /* ae_weight_format of the block Linears */
} ae_config;

/*
 * Weights, as device pointers of type T.  The per-layer members are HOST
 * arrays of `layers` device pointers.  ae_create copies and repacks all of
 * them into library-owned memory (merged QKV and gate/up as in sglang
 * PR #34599 item 1), so the caller keeps ownership and may free them once
 * ae_create has returned.
 *   w_in [D, A], b_in [D]               action input projection
 *   w_t1 [D, D], b_t1 [D], w_t2, b_t2   time MLP: c = silu(W2 silu(W1 e + b1) + b2)
 *   wq [Hq*dh, D], wk [Hkv*dh, D], wv [Hkv*dh, D], wo [D, Hq*dh]
 *   wg [F, D], wu [F, D], wd [D, F]     GeGLU MLP: (gelu_tanh(y Wg^T) * y Wu^T) Wd^T
 *   w_mod1/w_mod2 [3D, D], b_mod1/b_mod2 [3D]   adaRMS (scale, shift, gate) of
 *                                       the attention / MLP sublayer
 *   w_mod_f [2D, D], b_mod_f [2D]       final adaRMS (scale, shift)
 *   w_out [A, D], b_out [A]             action output projection
 *   w_ck, w_cv [Hkv*dh, C]              context K / V projections (ae_bind_context);
 *                                       required when ctx_dim > 0, else may be NULL
 */
typedef struct {
  const void *w_in, *b_in;
  const void *w_t1, *b_t1, *w_t2, *b_t2;
  const void *w_mod_f, *b_mod_f;
  const void *w_out, *b_out;
  const void *const *wq, *const *wk, *const *wv, *const *wo;
  const void *const *wg, *const *wu, *const *wd;
  const void *const *w_mod1, *const *b_mod1, *const *w_mod2, *const *b_mod2;
  const void *const *w_ck, *const *w_cv;
} ae_weights;

/*
 * Create a context on the current CUDA device.
 *   max_batch       requests a bind may hold, 1..AE_MAX_BATCH
 *   max_prefix_rows physical prefix rows one request may have (valid + masked)
 *   stream          cudaStream_t the context enqueues on (NULL = legacy default)
 *   out             receives the context; set to NULL on failure
 * Allocates all device memory the context will use (weights, scratch, bind
 * tables); later calls allocate only a per-n_steps time table on first use.
 * With cfg->weight_format == AE_WEIGHTS_FP8_E4M3 the block Linears are
 * quantized here (see ae_weight_format).
 * Errors: AE_ERR_INVALID_ARG, AE_ERR_SHAPE, AE_ERR_UNSUPPORTED, AE_ERR_OOM,
 * AE_ERR_CUDA.
 */
AE_API ae_status ae_create(const ae_config* cfg, const ae_weights* w, int max_batch,
                    int max_prefix_rows, void* stream, ae_ctx** out);

/* Destroy a context (synchronizes its stream first).  NULL is ignored. */
AE_API void ae_destroy(ae_ctx* ctx);

/* Change the stream later calls enqueue on. */
AE_API ae_status ae_set_stream(ae_ctx* ctx, void* stream);

/*
 * Bind the VLM prefix KV of `batch` requests (MolmoBot Part 2: computed once,
 * reused by every flow step; OxyGen: borrowed, never copied).
 *   prefix_k, prefix_v  device T, packed varlen [layers][total_rows][Hkv*dh]
 *                       with total_rows = cu_lens[batch].  K is already
 *                       rotated at the VLM's positions and is not re-roped.
 *   cu_lens             HOST int32 [batch + 1]: request b owns physical rows
 *                       cu_lens[b] .. cu_lens[b+1]-1; cu_lens[0] == 0,
 *                       non-decreasing, at most max_prefix_rows per request.
 *   prefix_mask         device uint8 [total_rows], 1 = valid, 0 = masked or
 *                       padding; NULL = every row valid.  Masked rows are never
 *                       read (they may hold NaN) and do not advance positions
 *                       (LoongForge section 1): action token i of request b
 *                       sits at position n_b + i, n_b = its valid row count.
 * prefix_k, prefix_v and prefix_mask must stay alive and unchanged until the
 * last ae_sample that uses this binding has completed on the stream.
 * batch == 0 is legal (ae_sample then does nothing).
 * Errors: AE_ERR_INVALID_ARG, AE_ERR_SHAPE (batch > max_batch, a request
 * longer than max_prefix_rows, bad cu_lens), AE_ERR_CUDA.
 */
AE_API ae_status ae_bind_prefix(ae_ctx* ctx, int batch, const void* prefix_k,
                         const void* prefix_v, const int32_t* cu_lens,
                         const uint8_t* prefix_mask);

/*
 * Bind ONE request's VLM prefix KV for n_samples action samples of the same
 * observation (OxyGen, "Cross-task KV Sharing": the prefill's KV is a shared
 * resource that every consumer reads in place).  Every sample attends to the
 * same prefix rows; each has its own noise and actions in ae_sample
 * ([n_samples][horizon][action_dim]).  The result equals ae_bind_prefix of
 * n_samples copies of the prefix, without the copies: the K/V stay in one
 * place and are read by all samples' attention work.
 *   prefix_k, prefix_v  device T [layers][n_rows][Hkv*dh], K already rotated
 *   n_rows              physical rows per layer, 0..max_prefix_rows
 *   prefix_mask         device uint8 [n_rows] (1 = valid) or NULL
 * Lifetime rules, positions and errors as for ae_bind_prefix (n_samples plays
 * the part of batch: AE_ERR_SHAPE above max_batch).
 */
AE_API ae_status ae_bind_prefix_shared(ae_ctx* ctx, int n_samples, const void* prefix_k,
                                const void* prefix_v, int32_t n_rows,
                                const uint8_t* prefix_mask);

/*
 * Bind `batch` requests whose prefix arrives as per-layer VLM hidden states
 * (the cross-attention form of MolmoBot PR Part 2: "compute the cross-attention
 * K/V once per query and reuse them across every step").  The library
 * projects every valid row once, here, into its own K/V buffers:
 *   K = RoPE(hidden W_ck^T) at the row's position among its request's valid
 *   rows (0 .. n_b - 1),  V = hidden W_cv^T,
 * and binds them exactly as ae_bind_prefix binds a pre-projected prefix;
 * every later ae_sample reuses them.  hidden is only read during this call's
 * work on the stream: it may be freed or changed once that work is done.
 *   hidden       device T, packed varlen [layers][total_rows][ctx_dim],
 *                total_rows = cu_lens[batch]
 *   cu_lens      HOST int32 [batch + 1], as in ae_bind_prefix
 *   prefix_mask  device uint8 [total_rows] (1 = valid) or NULL; masked rows
 *                are never read (they may hold NaN) and do not advance positions
 * Errors: AE_ERR_UNSUPPORTED (context created with ctx_dim == 0), and those
 * of ae_bind_prefix.
 */
AE_API ae_status ae_bind_context(ae_ctx* ctx, int batch, const void* hidden, const int32_t* cu_lens,
                          const uint8_t* prefix_mask);

/*
 * VLM prefill producing the prefix KV (OxyGen: the prefill of a frame's
 * observation and instruction produces KV[t]; MolmoBot PR Part 2: the VLM
 * backbone runs once per query).  The context must describe the VLM: a
 * Gemma-style decoder with the action expert's layer, whose RMSNorm weights
 * w are given as the biases (w, 0, 1) of zero modulation Linears (w_mod1 /
 * w_mod2 zero, b_mod1 / b_mod2 = [w | 0 | 1]): RMSNorm x rsqrt(mean(x^2) +
 * eps) (1 + w) with plain residuals.  `horizon` of its config is the number
 * of prefix tokens of a request.  For each of `batch` requests the prefix
 * tokens attend to each other (bidirectionally) at positions 0..horizon-1,
 * and every layer's K (after RoPE) and V are written out in the layout
 * ae_bind_prefix reads.  bf16 contexts only.
 *   embeddings  device bf16 [batch * horizon][width], request-major
 *   out_k, out_v device bf16 [layers][batch * horizon][n_kv_heads * head_dim]
 * Replaces the context's binding (an empty prefix for `batch` requests).
 * Errors: AE_ERR_UNSUPPORTED (fp32 context), AE_ERR_SHAPE (batch outside
 * 1..max_batch), AE_ERR_INVALID_ARG, AE_ERR_OOM, AE_ERR_CUDA.
 */
AE_API ae_status ae_prefill(ae_ctx* ctx, int batch, const void* embeddings, void* out_k, void* out_v);

/*
 * Run n_steps Euler steps of delta = -1/n_steps from t = 1 for every bound
 * request (MolmoBot Part 2), the velocity of step k taken at t = 1 - k/n_steps.
 *   noise        device fp32 [batch][horizon][action_dim], the state at t = 1
 *   out_actions  device fp32 [batch][horizon][action_dim]; may equal noise
 * The time-conditioning table for this n_steps is built on first use and
 * cached in the context (it depends on the weights and n_steps only).
 * Errors: AE_ERR_NOT_BOUND, AE_ERR_INVALID_ARG, AE_ERR_SHAPE (n_steps outside
 * 1..AE_MAX_STEPS), AE_ERR_DEVICE (sticky status of an earlier call),
 * AE_ERR_OOM, AE_ERR_CUDA.
 */
AE_API ae_status ae_sample(ae_ctx* ctx, const float* noise, int n_steps, float* out_actions);

/*
 * ae_sample for callers that cannot allocate device memory while sampling.
 * The pages have no counterpart to this call; it exists for callers such as
 * code that samples while a CUDA stream capture is open (an allocation there
 * breaks the capture), a serving process whose HBM is pre-reserved for its own
 * caches, or a real-time control loop that forbids allocator calls after
 * start-up.  ae_sample may allocate on its first call with a new n_steps (the
 * time-conditioning table) and when it records its CUDA graph; this call runs
 * the same kernels, launched one by one on the context's stream, and calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *   - The attention kernel's split-KV partial results live in one static
 *     16 MiB __device__ array of the library (held by every GPU that loads
 *     the library until the process exits) instead of context memory.  A
 *     batch whose partials do not fit (about 30 requests at head_dim 256)
 *     returns AE_ERR_SHAPE.
 *   - The time-conditioning table of n_steps must already exist: call
 *     ae_sample once with the same n_steps first, else AE_ERR_NOT_BOUND.
 *   - The first call on a device looks up the array's device address (a
 *     module load, not an allocation by this library); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and leaves its contents behind;
 *     calls that overlap on the GPU (different streams or contexts of one
 *     device) race on it.
 * bf16 contexts only (AE_ERR_UNSUPPORTED otherwise).  Arguments and other
 * errors as for ae_sample.
 */
AE_API ae_status ae_sample_noalloc(ae_ctx* ctx, const float* noise, int n_steps,
                                   float* out_actions);

/*
 * Self-test of device-side failure detection (the pages have no counterpart;
 * it checks this library's own error path).  The tensor-core kernels bound
 * every wait on an mbarrier by a cycle budget (about one second); a wait that
 * runs out records a timeout in the context's sticky device status and the
 * kernel returns instead of hanging.  This call enqueues one small kernel that
 * runs that same bounded wait on an mbarrier nothing ever completes, with a
 * budget of `budget_cycles` SM clock cycles, and with no copy, MMA or TMEM
 * allocation in flight.  After it, ae_synchronize, ae_last_error and every
 * later ae_sample of this context report AE_ERR_DEVICE; the status is not
 * cleared (create a new context to continue).  The GPU and other contexts are
 * not affected.
 * Errors: AE_ERR_INVALID_ARG (NULL ctx, budget_cycles < 0), AE_ERR_CUDA.
 */
AE_API ae_status ae_selftest_wait_timeout(ae_ctx* ctx, int64_t budget_cycles);

/*
 * Optional per-layer hidden-state dump for parity checks.  When set, every
 * ae_sample writes the fp32 residual stream entering layer l (l = 0..L-1) and
 * leaving the last layer (l = L) of every step s to
 *   hidden[((s * (L + 1) + l) * batch + b) * horizon + i][0 .. D-1].
 * hidden: device fp32 with room for `capacity` floats; NULL switches it off.
 * ae_sample returns AE_ERR_SHAPE if the dump does not fit.
 */
AE_API ae_status ae_set_debug_dump(ae_ctx* ctx, float* hidden, size_t capacity);

/* Wait for the context's stream, then report the sticky device status. */
AE_API ae_status ae_synchronize(ae_ctx* ctx);

/*
 * Copy a NUL-terminated description of the last error of this context (or of
 * the last failed ae_create when ctx is NULL) into buf[0..n-1].  Returns the
 * sticky device status (AE_OK if none).
 */
AE_API ae_status ae_last_error(const ae_ctx* ctx, char* buf, size_t n);

/* Static name of a status code. */
AE_API const char* ae_status_string(ae_status s);

/*
 * Copy out one quantized block Linear of a context created with
 * AE_WEIGHTS_FP8_E4M3, in the caller's layout (row-major [out, in], rows in
 * the order of the weight given to ae_create, whatever the library's packing).
 *   layer   0..layers-1
 *   which   0 wq, 1 wk, 2 wv, 3 wo, 4 wg, 5 wu, 6 wd
 *   codes   HOST uint8 with room for the tensor's out * in codes, or NULL
 *   scale   HOST float: the tensor's dequantization factor r, or NULL
 * Synchronizes the context's stream.
 * Errors: AE_ERR_INVALID_ARG (NULL ctx, layer or which out of range),
 * AE_ERR_UNSUPPORTED (the weights are not fp8), AE_ERR_CUDA.
 */
AE_API ae_status ae_get_fp8_weight(ae_ctx* ctx, int layer, int which, uint8_t* codes, float* scale);

/* Counters a caller can read after ae_sample, e.g. to report kernel launches. */
typedef struct {
  int64_t launches_last_sample; /* kernels the last ae_sample enqueued      */
  int64_t launches_last_bind;   /* kernels the last ae_bind_prefix enqueued */
  int64_t device_bytes;         /* device memory the context holds          */
  int sm_count;                 /* SMs of the context's device              */
  int path;                     /* 0 = fp32 SIMT path, 1 = bf16 path         */
} ae_info;

AE_API ae_status ae_get_info(const ae_ctx* ctx, ae_info* info);

#ifdef __cplusplus
}
#endif

#endif /* AE_H_ */
