/*
 * ob.h -- C ABI of libob, the GB300 (sm_103a) implementation of the
 * error-compensated 1-bit compressed optimizer step (1-bit Adam and 1-bit
 * LAMB) and of a block-wise INT8 stochastic-rounding quantizer.
 *
 * Sources, cited by page title and section:
 *   [BLOG] lqnn.cn, "1bit Adam" write-up: 2.1 error compensation, 6 warmup.
 *   [TUT]  FreeGuideOnline, "梯度量化：将梯度从 FP32 压到 INT8 甚至 1-bit":
 *          "FP32 → INT8 量化", "1-bit 梯度量化", GradientQuantizeINT8 example.
 *   [LAMB] "1-bit LAMB (Error-Compensated LAMB-Preconditioned Large-Batch
 *          Compressed Optimization)", paragraphs 1-4.
 *
 * Model.  W data-parallel workers are simulated as W resident buffer sets
 * on one GPU.  One compressed step is
 *     ob_compress       every worker compresses its momentum   ([LAMB] 2-3)
 *     ob_server_reduce  server j averages partition j of all workers,
 *                       adds its own error and compresses again ([LAMB] 3-4)
 *     ob_adam_step      unpack + frozen-variance Adam            ([LAMB] 1)
 *  or ob_lamb_step      unpack + 1-bit LAMB update               ([LAMB] 1-2)
 * The worker-to-server "all-to-all" is the server kernel reading the
 * workers' packed words straight from HBM (bulk copies of each worker's
 * 16-byte aligned run of words for a tile).  After a compressed step the
 * momentum is exactly the server's scaled signs, so it can be held in that
 * form between steps: ob_compress_signm (1-bit Adam, server in place) and
 * ob_compress_signm_ls + ob_server_reduce_db + ob_lamb_step_signm (1-bit
 * LAMB, server output double-buffered), or ob_step / ob_step_db in one
 * call.
 *
 * Device errors.  Pipelined kernels wait on shared-memory barriers for
 * their own bulk copies; every wait is bounded (about a second), and a
 * wait that runs out records a code in the workspace and lets the kernel
 * return.  ob_device_error() reads (and clears) that code.
 *
 * Layout.  n real elements, W workers, alignment A, chunk C (both multiples
 * of 32).  P = roundup(ceil(n/W), A); n_pad = W*P; server j owns
 * [jP, (j+1)P).  Each partition is cut into chunks of min(C, P) elements
 * (the last one may be short); chunk g = j*cpp + kc, cpp = ceil(P/C).
 * Elements k >= n are padding: they are excluded from every scale, their
 * bit is 0, their error 0.
 *   grads      W buffers of n_pad elements (fp32 or bf16)
 *   err        W buffers of n_pad fp32 (worker error, deferred form)
 *   bits       [W][words] uint32, words = n_pad/32 rounded up to a multiple
 *              of 4 (16-byte rows); bit k%32 of word k/32 of a row (LSB
 *              first) is 1 iff x[k] >= 0.0f (sign(+0) = sign(-0) = +1,
 *              NaN -> -1); the rounding words are never written
 *   scales     [W][n_chunks] fp32, each worker's scale of every chunk
 *   err_s      n_pad fp32 (server error, deferred form)
 *   sbits      [words] uint32; sscales [n_chunks] fp32
 *   m, v, p    n_pad fp32 (momentum, frozen variance, parameters)
 * Padding entries of m and of the errors are written as 0; padding entries
 * of p and v are never written.
 *
 * Deferred errors.  ob_compress stores the compensated value x in err
 * instead of e' = x - scale*sign(x): the scale needs the whole chunk, and
 * storing x keeps the step single-pass.  The next ob_compress recovers e'
 * from (x, bits, scales) bit for bit before using it.  The same holds for
 * the server (err_s, sbits, sscales).  ob_materialize_errors writes e' into
 * err/err_s and zeroes the scales, a state the next call reads the same
 * way (e' - 0*sign = e').
 *
 * Arithmetic.  fp32, every operation rounded on its own (no contracted
 * multiply-add, IEEE division and square root, no flush to zero).  Every
 * sum that decides a scale or a norm follows one fixed order (4096-element
 * tiles, 256 lanes adding elements 1024*i + 4*lane + c for i, c = 0..3,
 * warp butterflies, a pairwise tree over 8 warps, tile totals added in
 * order), so results are reproducible bit for bit.
 *
 * Conventions.
 *   - Every function returns ob_status; ob_last_error(ctx) (or
 *     ob_last_error(NULL) for calls without a ctx) gives a message.
 *   - All device buffers are owned by the caller; the library allocates
 *     no device memory.  ob_workspace_bytes() gives the size of the
 *     scratch area the caller passes to ob_set_workspace().
 *   - Calls are asynchronous on `stream`; nothing synchronises.  A launch
 *     failure is reported as OB_ERR_CUDA.
 *   - Device pointers must be 16-byte aligned (scales 4-byte, INT8 codes
 *     4-byte).  Invalid arguments are rejected before any launch.
 *   - A ctx is not thread-safe; distinct ctxs are independent.  Calls that
 *     share a ctx (and so its workspace) must not overlap on the GPU.
 */
#ifndef OB_H
#define OB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ob_stream_t; /* the same handle as cudaStream_t */
typedef int ob_status;

#define OB_OK 0
#define OB_ERR_INVALID 1     /* bad argument or size */
#define OB_ERR_ALIGN 2       /* misaligned pointer */
#define OB_ERR_UNSUPPORTED 3 /* a configuration the library does not support */
#define OB_ERR_CUDA 4        /* a CUDA call or launch failed */
#define OB_ERR_STATE 5       /* call out of order (e.g. no workspace) */

#define OB_GRAD_F32 0
#define OB_GRAD_BF16 1

#define OB_MODE_ADAM 0
#define OB_MODE_LAMB 1

#define OB_MAX_WORKERS 64

/* ob_config.flags */
#define OB_FLAG_NO_RATIO_EF (1u << 0) /* LAMB: error feedback factor rho = 1
                                         instead of c_{t-2}/c_{t-1} */
#define OB_FLAG_FROZEN_C (1u << 1)    /* LAMB: r = 1, c = c_avg ("LAMB +
                                         basic 1-bit", [LAMB] 1) */

typedef struct ob_config {
  size_t n;                     /* real elements, >= 1, < 2^34 */
  int W;                        /* workers, 1..OB_MAX_WORKERS */
  size_t chunk;                 /* C: multiple of 32, >= 32 (clamped to P) */
  size_t align;                 /* A: multiple of 32, >= 32 */
  int grad_dtype;               /* OB_GRAD_F32 or OB_GRAD_BF16 */
  int n_layers;                 /* 0: one layer [0, n) */
  const size_t* layer_offsets;  /* host, n_layers+1 entries, 0 = off[0] <
                                   off[1] < ... < off[n_layers] = n; copied */
  float b1, b2, eps, lr;        /* Adam/LAMB hyperparameters */
  float r_thr, r_min, r_max;    /* LAMB ratio clip ([LAMB] 1) */
  float c_min, c_max;           /* LAMB coefficient clip ([LAMB] 3) */
  uint32_t flags;               /* OB_FLAG_* */
  float clip_value;             /* > 0: workers' compensated values are
                                   limited to [-clip_value, clip_value]
                                   before compression ([BLOG] 4.1); 0 = off */
  /* The method's schedules ([BLOG] 4.1, 3.2 table, 6 layerwise_bits); see
   * ob_plan_step.  All zero: no reset, every step exchanged, key = bits. */
  uint32_t reset_interval;      /* > 0: worker and server errors are reset
                                   to 0 before every reset_interval-th
                                   compressed step ([BLOG] 4.1: every 2000);
                                   0 = never */
  uint32_t send_period;         /* FP16 codec groups: exchanged on the
                                   compressed steps t with t % send_period
                                   == 0 ([BLOG] 3.2: every 10th); 0 or 1 =
                                   every step */
  uint64_t seed;                /* b-bit codec groups: the Philox key is
                                   seed + bits, one stream per width */
} ob_config;

typedef struct ob_layout {
  size_t n, n_pad, P, chunk;    /* chunk = min(C, P) */
  size_t chunks_per_partition;  /* cpp */
  size_t n_chunks;              /* W * cpp: length of sscales, and of each
                                   worker's row of scales */
  size_t words_per_worker;      /* row stride of bits: n_pad/32 rounded up
                                   to a multiple of 4 */
  size_t n_tiles;               /* 4096-element tiles, counted per chunk */
  int W, n_layers;              /* n_layers >= 1 */
} ob_layout;

/* Per-layer state of 1-bit LAMB: device arrays of n_layers floats. */
typedef struct ob_layer_state {
  float* s;        /* fixed momentum scale sigma_l ([LAMB] 2) */
  float* c_avg;    /* warmup average of LAMB's coefficient ([LAMB] 1) */
  float* r_prev;   /* r_{t-1} */
  float* c_prev;   /* c_{t-1} */
  float* c_prev2;  /* c_{t-2} */
  float* c_sum;    /* warmup: running sum of c */
  float* c_t;      /* output: c of the latest step */
} ob_layer_state;

typedef struct ob_ctx ob_ctx;

/* Validates cfg and builds the layout (host only; no CUDA call).
 * OB_ERR_INVALID on a bad size, OB_ERR_UNSUPPORTED on W > OB_MAX_WORKERS. */
ob_status ob_init(const ob_config* cfg, ob_ctx** out);
ob_status ob_destroy(ob_ctx* ctx);
const char* ob_last_error(const ob_ctx* ctx);
ob_status ob_get_layout(const ob_ctx* ctx, ob_layout* out);

/* Scratch: per-tile partial sums and arrival counters of the chunk scales,
 * per-layer tables and accumulators.  Owned by the caller, device memory,
 * 256-byte aligned, valid until the ctx is destroyed or another workspace
 * is set.  ob_set_workspace enqueues its initialisation on `stream`. */
ob_status ob_workspace_bytes(const ob_ctx* ctx, size_t* bytes);
ob_status ob_set_workspace(ob_ctx* ctx, void* workspace, size_t bytes,
                           ob_stream_t stream);

/* One uncompressed warmup step ([BLOG] 6, [TUT] "预热训练"; [LAMB] 1):
 *   g_bar = (sum_w g_w)/W; m = b1*m + (1-b1)*g_bar; v = b2*v + (1-b2)*g_bar^2
 *   ADAM: p -= lr*(m/(sqrt(v)+eps))
 *   LAMB: u = m/(sqrt(v)+eps); c_l = clip(||p_l||/||u_l||, c_min, c_max)
 *         (1 if a norm is 0); p -= (lr*c_l)*u; ls->c_sum += c; ls->c_t = c
 * grads: host array of W device pointers.  ls: NULL for ADAM. */
ob_status ob_warmup_step(ob_ctx* ctx, const void* const* grads, float* m,
                         float* v, float* p, int mode,
                         const ob_layer_state* ls, ob_stream_t stream);

/* End of warmup.  Zeroes err (W host-array pointers), err_s, bits, scales,
 * sbits, sscales (the deferred form of e = 0); all six may be NULL together
 * (a rank of a multi-process job clears its own slices).  v becomes the frozen
 * variance v_Tw.  LAMB (ls != NULL): v_fresh = v; per layer
 *   rms_l = ||m_l||/sqrt(n_l); s_l = mean(rms)/rms_l (1 if rms_l = 0)
 *   c_avg = c_sum/warmup_steps; r_prev = 1; c_prev = c_prev2 = c_avg
 * ([LAMB] 1-2).  m, v, v_fresh, ls may be NULL for ADAM. */
ob_status ob_begin_compression(ob_ctx* ctx, float* const* err, float* err_s,
                               uint32_t* bits, float* scales, uint32_t* sbits,
                               float* sscales, const float* m, const float* v,
                               float* v_fresh, const ob_layer_state* ls,
                               int warmup_steps, ob_stream_t stream);

/* Worker compression, all W workers ([BLOG] 2.1, [TUT] "1-bit 梯度量化",
 * [LAMB] 2-3):
 *   m_w = b1*m + (1-b1)*g_w
 *   x   = sigma_l*m_w + rho_l*e_w    (ADAM: x = m_w + e_w)
 *   x   = clamp(x, -clip_value, clip_value) if clip_value > 0 ([BLOG] 4.1)
 *   scale(chunk) = mean |x| over the chunk's real elements
 *   bit = x >= 0;  e_w' = x - scale*sign(x)   (stored deferred)
 * sigma_l = ls->s, rho_l = ls->c_prev2/ls->c_prev (1 with
 * OB_FLAG_NO_RATIO_EF); ls == NULL means 1-bit Adam.  m is not written. */
ob_status ob_compress(ob_ctx* ctx, const void* const* grads, const float* m,
                      float* const* err, uint32_t* bits, float* scales,
                      const ob_layer_state* ls, ob_stream_t stream);

/* ob_compress for 1-bit Adam with the momentum in its sign form: after a
 * compressed Adam step the momentum is exactly sscale*sign(sbit) of that
 * step's server output, so the next compression can read those words
 * (1/8 byte per element) instead of a dense fp32 m (4 bytes), and the
 * update need not write m (ob_adam_step with m == NULL); ob_decompress
 * gives m whenever it is wanted.  sbits/sscales are read before the
 * following ob_server_reduce overwrites them.  Not for the first
 * compressed step after ob_begin_compression (m comes from warmup then),
 * nor after ob_materialize_errors (which zeroes sscales): use ob_compress
 * with the dense m there. */
ob_status ob_compress_signm(ob_ctx* ctx, const void* const* grads, const uint32_t* sbits,
                            const float* sscales, float* const* err, uint32_t* bits,
                            float* scales, ob_stream_t stream);

/* ob_compress_signm for 1-bit LAMB as well (ls != NULL): after a compressed
 * LAMB step the momentum is exactly sscale*sign(sbit)/sigma_l of that
 * step's server output (the update stores M/sigma_l, [LAMB] 1-2), and
 * +-sscale/sigma_l is one correctly rounded division per layer.  ls == NULL
 * is ob_compress_signm.  The same conditions apply; with LAMB the server
 * output must be double-buffered (ob_server_reduce_db), because the
 * update reads the previous step's words too (ob_lamb_step_signm). */
ob_status ob_compress_signm_ls(ob_ctx* ctx, const void* const* grads, const uint32_t* sbits,
                               const float* sscales, float* const* err, uint32_t* bits,
                               float* scales, const ob_layer_state* ls, ob_stream_t stream);

/* Server average and re-compression, all partitions ([LAMB] 3-4):
 *   z = (sum_w scale_w(chunk)*sign_w)/W;  y = rho_l*e_s + z
 *   sscale(chunk) = mean |y|;  sbit = y >= 0;  e_s' = y - sscale*sign(y) */
ob_status ob_server_reduce(ob_ctx* ctx, const uint32_t* bits,
                           const float* scales, float* err_s, uint32_t* sbits,
                           float* sscales, const ob_layer_state* ls,
                           ob_stream_t stream);

/* ob_server_reduce with the server output double-buffered: the deferred
 * error e_s is decoded with the previous step's (sbits_old, sscales_old),
 * and the new words and scales go to (sbits, sscales), leaving the old
 * ones intact.  Each pair either is the same buffer (then this is
 * ob_server_reduce) or does not overlap (OB_ERR_INVALID otherwise). */
ob_status ob_server_reduce_db(ob_ctx* ctx, const uint32_t* bits, const float* scales,
                              float* err_s, const uint32_t* sbits_old, const float* sscales_old,
                              uint32_t* sbits, float* sscales, const ob_layer_state* ls,
                              ob_stream_t stream);

/* out = sscale*sign(sbit) (/ sigma_l if ls != NULL); padding -> 0. */
ob_status ob_decompress(ob_ctx* ctx, const uint32_t* sbits,
                        const float* sscales, const ob_layer_state* ls,
                        float* out, ob_stream_t stream);

/* 1-bit Adam update with the frozen variance ([LAMB] 1, [BLOG] 2.1):
 *   m = sscale*sign(sbit);  p -= lr*(m/(sqrt(v_frozen)+eps))
 * m may be NULL: then it is not written, and the momentum stays held
 * exactly by (sbits, sscales) -- see ob_compress_signm. */
ob_status ob_adam_step(ob_ctx* ctx, const uint32_t* sbits,
                       const float* sscales, const float* v_frozen, float* m,
                       float* p, ob_stream_t stream);

/* 1-bit LAMB update ([LAMB] 1-3), in two element passes:
 *   A: m_t = sscale*sign/sigma_l; g = (m_t - b1*m)/(1-b1);
 *      v_fresh = b2*v_fresh + (1-b2)*g^2; R_l = max(v_frozen/v_fresh)
 *      (NaN skipped)
 *      then per layer r = clip(clip(R_l, (1-r_thr)r_prev, (1+r_thr)r_prev),
 *      r_min, r_max); c = clip(c_avg*r, c_min, c_max); shift c_prev2 <-
 *      c_prev <- c; r_prev <- r; ls->c_t = c
 *   B: p -= (lr*c_l)*(m_t/(sqrt(v_frozen)+eps)) */
ob_status ob_lamb_step(ob_ctx* ctx, const uint32_t* sbits,
                       const float* sscales, const float* v_frozen,
                       float* v_fresh, float* m, float* p,
                       const ob_layer_state* ls, ob_stream_t stream);

/* ob_lamb_step with the momentum in its sign form: the previous momentum
 * is sscale_prev*sign(sbit_prev)/sigma_l from the previous step's server
 * output, m_t = sscale*sign(sbit)/sigma_l from this step's, and no dense m
 * is read or written.  The two server buffers must not overlap
 * (OB_ERR_INVALID). */
ob_status ob_lamb_step_signm(ob_ctx* ctx, const uint32_t* sbits_prev, const float* sscales_prev,
                             const uint32_t* sbits, const float* sscales, const float* v_frozen,
                             float* v_fresh, float* p, const ob_layer_state* ls,
                             ob_stream_t stream);

/* compress + server_reduce + adam_step (ls == NULL) or lamb_step, in one
 * call, in that order.  With m == NULL (1-bit Adam only) the momentum is
 * held in its sign form: ob_compress_signm + server + ob_adam_step without
 * m.  1-bit LAMB in sign form needs the double-buffered ob_step_db. */
ob_status ob_step(ob_ctx* ctx, const void* const* grads, float* m,
                  float* const* err, uint32_t* bits, float* scales,
                  float* err_s, uint32_t* sbits, float* sscales,
                  const float* v_frozen, float* v_fresh, float* p,
                  const ob_layer_state* ls, ob_stream_t stream);

/* One compressed step with the momentum in its sign form and the server
 * output double-buffered, 1-bit Adam (ls == NULL) or 1-bit LAMB:
 * ob_compress_signm_ls from (sbits_prev, sscales_prev), then
 * ob_server_reduce_db into (sbits, sscales), then ob_adam_step without m or
 * ob_lamb_step_signm.  The caller swaps the two buffers between steps.  The
 * same conditions as ob_compress_signm apply (not the first compressed
 * step after ob_begin_compression or ob_materialize_errors). */
ob_status ob_step_db(ob_ctx* ctx, const void* const* grads, float* const* err, uint32_t* bits,
                     float* scales, float* err_s, const uint32_t* sbits_prev,
                     const float* sscales_prev, uint32_t* sbits, float* sscales,
                     const float* v_frozen, float* v_fresh, float* p, const ob_layer_state* ls,
                     ob_stream_t stream);

/* Writes the true errors e' into err and err_s and zeroes scales and
 * sscales.  Call only after a complete step (the update has consumed the
 * scales). */
ob_status ob_materialize_errors(ob_ctx* ctx, float* const* err,
                                const uint32_t* bits, float* scales,
                                float* err_s, const uint32_t* sbits,
                                float* sscales, ob_stream_t stream);

/* The periodic error reset of [BLOG] 4.1 (every reset_interval steps the
 * compensation term is set to zero): after this call the next compression
 * sees worker and server errors of exactly 0.  The deferred form is kept
 * (err := scale*sign, err_s := sscale*sign, so that err - scale*sign = 0),
 * so bits and scales -- and a momentum held in sign form -- are untouched. */
ob_status ob_reset_errors(ob_ctx* ctx, float* const* err, const uint32_t* bits,
                          const float* scales, float* err_s, const uint32_t* sbits,
                          const float* sscales, ob_stream_t stream);

/* The quantisation-error monitor of [TUT] "监控与诊断" (watch the norm of
 * the quantisation error) and [BLOG] 7 (check that the error term stays
 * bounded), for the 1-bit compressor.  From the deferred buffers of the
 * last step (the same ones ob_materialize_errors reads; nothing is
 * written but `out` and the workspace's tile totals):
 *   out[w*n_chunks + g] = sum over chunk g's real elements of e_w'^2,
 *   out[W*n_chunks + g] = the same for the server error e_s',
 * e' = x - scale*sign(x) decoded as the next compression would, each sum
 * in the fixed order of the scales.  out: (W+1)*n_chunks floats, 4-byte
 * aligned; the square root of a row's total is that error's 2-norm.  Uses
 * the workspace like the other calls of the ctx. */
ob_status ob_error_norm(ob_ctx* ctx, const float* const* err, const uint32_t* bits,
                        const float* scales, const float* err_s, const uint32_t* sbits,
                        const float* sscales, float* out, ob_stream_t stream);

/* Reads and clears the device error word of the workspace (0 = none;
 * 1 = a consumer's wait for a copy ran out, 2 = the producer's wait for a
 * free stage ran out, 3 = copies still in flight at exit).  Synchronises
 * `stream`. */
ob_status ob_device_error(ob_ctx* ctx, unsigned* code, ob_stream_t stream);

/* No counterpart in the pages: an addition of this library for callers
 * that cannot allocate device memory -- code inside a runtime whose own
 * pool owns the device and gives extensions no allocator, or code that
 * cannot afford the device-wide synchronisation of cudaMalloc/cudaFree.
 * Same arguments and results as ob_compress with ls == NULL (1-bit Adam),
 * and no workspace is needed: the scratch (per-tile totals and an error
 * word) is a static device array of OB_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until exit.  Allocates nothing.
 *   - A layout is accepted exactly when
 *       W * n_chunks * ceil(chunk / 4096) * 4  <=  OB_NOALLOC_SCRATCH_BYTES - 256
 *     (n_chunks and chunk as ob_get_layout reports them; the last 256
 *     bytes hold the error word); others get OB_ERR_UNSUPPORTED before
 *     any launch (e.g. up to about 2^28 elements at W = 8).
 *   - The first call on a device (of this function or of
 *     ob_noalloc_device_error) looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and clears the error
 *     word on `stream`; make that first call before any stream capture.
 *   - All calls share the array: calls that overlap on the GPU race.
 *   - A bounded wait that gives up records its code (as for ob_device_error)
 *     in the array's error word, which no call clears: read it with
 *     ob_noalloc_device_error. */
#define OB_NOALLOC_SCRATCH_BYTES (4u << 20)
ob_status ob_compress_noalloc(ob_ctx* ctx, const void* const* grads, const float* m,
                              float* const* err, uint32_t* bits, float* scales,
                              ob_stream_t stream);

/* No counterpart in the pages.  Reads and clears the error word of the
 * current device's static scratch array used by ob_compress_noalloc (0 =
 * none, else the first code any call recorded since the last read; codes
 * as for ob_device_error).  Needs no ctx and allocates nothing.
 * Synchronises `stream`. */
ob_status ob_noalloc_device_error(unsigned* code, ob_stream_t stream);

/* Block-wise INT8 stochastic rounding ([TUT] "FP32 → INT8 量化" and the
 * GradientQuantizeINT8 example), blocks of 256 elements (the last may be
 * short):
 *   mx = max |g| (NaN never wins); scale = mx/127 (0 if mx = 0, then q = 0)
 *   x = g/scale; f = floor(x); q = f + (u < x - f); clamp to [-127, 127]
 *   (a NaN codes as 0); deq = q*scale if deq != NULL
 * u = (word >> 8) * 2^-24 from Philox4x32-10 (Salmon et al., SC'11) with
 * key = seed, counter = (k>>2, step) as two 64-bit halves, word k&3.
 * g and deq 16-byte aligned, q 4-byte aligned; n < 2^34.
 * block_scales: ceil(n/256) floats. */
ob_status ob_quant_int8(const float* g, size_t n, int8_t* q,
                        float* block_scales, uint64_t seed, uint64_t step,
                        float* deq, ob_stream_t stream);

/* INT8 with error feedback ([TUT] "1-bit 梯度量化" error feedback and
 * "精度恢复技巧": the residual is kept and added back before the next
 * quantisation): x = g + e; per block of 256 the quantizer of ob_quant_int8
 * is applied to x; e := x - q*scale (in place).  block_err2 (optional):
 * per block, the sum of the squared residuals -- the quantisation-error
 * monitor of [TUT] "监控与诊断" -- summed in a fixed order (lane j of 32
 * adds its elements 4j..4j+3 then 128+4j..128+4j+3, then a warp
 * butterfly).  e 16-byte aligned, n_pad-free: n elements. */
ob_status ob_quant_int8_ef(const float* g, float* e, size_t n, int8_t* q, float* block_scales,
                           uint64_t seed, uint64_t step, float* deq, float* block_err2,
                           ob_stream_t stream);

/* The schedule of compressed step t (t = 1, 2, ... counts the compressed
 * steps since ob_begin_compression or ob_zero_errors) for a group of width
 * `bits` (1, 2, 4, 8 or 16), from the ctx's configuration -- host only, no
 * CUDA call:
 *   reset  1 iff reset_interval > 0, t > 1 and (t - 1) % reset_interval == 0:
 *          the errors are reset before this step ([BLOG] 4.1), by
 *          ob_reset_errors (width 1) or ob_zero_errors (the codecs)
 *   send   width 16: 1 iff t % send_period == 0 ([BLOG] 3.2, "FP16, 每10步");
 *          other widths: 1
 *   key    width 2, 4, 8: seed + bits, the Philox key of ob_compress_qb and
 *          ob_server_reduce_qb; other widths: 0
 *   step   t, their Philox step counter
 * ob_codec_step applies it; a caller of the width-1 calls reads `reset`. */
typedef struct ob_plan {
  int reset, send;
  uint64_t key, step;
} ob_plan;
ob_status ob_plan_step(const ob_ctx* ctx, int bits, uint64_t t, ob_plan* out);

/* ------------------------------------------------------------------------
 * One rank of a multi-process job: one worker and one server per process
 * ([LAMB] 2 and 4: the 3-phase compressed exchange -- local compression,
 * an all-to-all of the compressed chunks, each server's average and
 * re-compression, an all-gather of the result).  The collectives are the
 * caller's (e.g. NCCL all-to-all and all-gather of the blocks below); these
 * calls do the compute of rank j, on the same kernels as the resident
 * path, with the same layout (ctx for n, W = the number of ranks, ...).
 *
 * Per step on rank j:
 *   ob_compress_worker      own gradient -> bits_row [words_per_worker],
 *                           scales_row [n_chunks]; partition i's block is
 *                           words [i*P/32, (i+1)*P/32) and scales
 *                           [i*cpp, (i+1)*cpp)
 *   all-to-all              block i to rank i: recv_bits [W][P/32] and
 *                           recv_scales [W][cpp], row w from rank w
 *   ob_server_reduce_part   partition j -> sbits_part [P/32],
 *                           sscales_part [cpp] (err_s_part [P] kept)
 *   all-gather              in rank order: sbits [n_pad/32] and sscales
 *                           [n_chunks], the whole server output
 *   ob_adam_step / ob_lamb_step on the whole (replicated) m, v, p
 * The rank's own bits_row/scales_row and sbits_part/sscales_part must be
 * kept from one step to the next (the deferred errors decode with them),
 * and are zeroed with err and err_s_part at the start of compression; for
 * 1-bit LAMB, ob_begin_compression with all six error and sign buffers
 * NULL does the rest.  The warmup steps average all W gradients
 * (ob_warmup_step on a gathered set).  P must be a multiple of 128 (A a
 * multiple of 128) for ob_server_reduce_part.  With the momentum in sign
 * form (after the first compressed step) ob_compress_worker reads it from
 * the last gathered output; for 1-bit LAMB the gathered output is then
 * double-buffered, since ob_lamb_step_signm reads the previous one too,
 * while sbits_part/sscales_part are rewritten in place.  The periodic reset
 * is ob_reset_errors_rank on every rank before the same steps. */

/* Rank compression of one worker: ob_compress for worker `rank`'s own
 * buffers only.  grad, err: n_pad elements; bits_row: words_per_worker
 * words; scales_row: n_chunks floats (both from the previous step on entry,
 * for the deferred error).  The momentum is dense (m, msbits = msscales =
 * NULL) or in its sign form (m = NULL, msbits/msscales the last step's
 * gathered server output, as ob_compress_signm_ls).  ls: 1-bit LAMB. */
ob_status ob_compress_worker(ob_ctx* ctx, const void* grad, const float* m,
                             const uint32_t* msbits, const float* msscales, float* err,
                             uint32_t* bits_row, float* scales_row, const ob_layer_state* ls,
                             ob_stream_t stream);

/* Rank server of partition j, from the W received blocks: recv_bits
 * [W][P/32] words (row w from worker w), recv_scales [W][cpp];
 * err_s_part [P] (deferred form), sbits_part [P/32] and sscales_part [cpp]
 * are read as the previous step's output and overwritten with this
 * step's.  The same arithmetic as ob_server_reduce on partition j.
 * OB_ERR_UNSUPPORTED if P % 128 != 0. */
ob_status ob_server_reduce_part(ob_ctx* ctx, int j, const uint32_t* recv_bits,
                                const float* recv_scales, float* err_s_part,
                                uint32_t* sbits_part, float* sscales_part,
                                const ob_layer_state* ls, ob_stream_t stream);

/* Rank form of ob_reset_errors ([BLOG] 4.1, the periodic reset): rank j's
 * own worker error (err [n_pad], decoded with bits_row and scales_row) and
 * its server partition's error (err_s_part [P], with sbits_part [P/32] and
 * sscales_part [cpp]) become exactly 0 for the next compression, in the
 * deferred form (err := scale*sign, err_s_part := sscale*sign), so the
 * words and scales -- and a momentum held in sign form -- are untouched.
 * Every rank calls it before the same steps (ob_plan_step's `reset`).
 * Needs no workspace. */
ob_status ob_reset_errors_rank(ob_ctx* ctx, int j, float* err, const uint32_t* bits_row,
                               const float* scales_row, float* err_s_part,
                               const uint32_t* sbits_part, const float* sscales_part,
                               ob_stream_t stream);

/* ------------------------------------------------------------------------
 * Layerwise mixed bit widths ([BLOG] 3.2 table: a bit width and an update
 * period per parameter type -- embeddings and transformer FFN 1 bit, CNN
 * weights 2 bits, LayerNorm parameters FP16 every 10 steps; [BLOG] 6
 * layerwise_bits [1, 2, 1, 16]; [TUT] "更激进的组合策略").
 *
 * The layers of one width form a fused buffer of their own with its own
 * ctx (the layout above, n = that group's elements).  Width 1 uses the
 * calls above.  Widths 2, 4 and 8 use the b-bit codec below, width 16 the
 * FP16 codec; both run 1-bit Adam's frozen-variance update (no LAMB) with
 * a dense m, and keep their errors in plain form (e' itself, not deferred).
 * Their ctx needs A = cfg.align a multiple of 256 (else
 * OB_ERR_UNSUPPORTED) and no workspace; cfg.b1, eps, lr and clip_value
 * apply, cfg.chunk and the layers are not used.
 *
 * b-bit codec, per block of 256 elements (block k/256 of each worker's
 * buffer; no block straddles two partitions since A % 256 == 0), the
 * quantizer of [TUT] "FP32 → INT8 量化" with the width as an argument (as
 * its GradientQuantizeINT8 example takes it):
 *   scale = max|x| / (2^(b-1) - 1) over the block's real elements (0 if the
 *   max is 0; a NaN never wins); q = floor(x/scale) + (u < frac) clamped to
 *   +-(2^(b-1) - 1), a NaN codes as 0; e' = x - q*scale.
 *   u as in ob_quant_int8 (Philox4x32-10, key = seed, counter = (i>>2,
 *   step), word i&3) with i = w*n_pad + k for worker w's element k and
 *   i = W*n_pad + k for the server's.
 *   codes: [W][words_per_worker] uint32, words_per_worker = n_pad*b/32; the
 *   field q mod 2^b of element k at bit (k*b)%32 of word (k*b)/32 (LSB
 *   first, two's complement).  bscales: [W][n_blocks] floats,
 *   n_blocks = n_pad/256.  Padding elements code 0 with error 0.
 * ---------------------------------------------------------------------- */

/* words_per_worker = n_pad*bits/32 and n_blocks = n_pad/256 (either may
 * be NULL).  bits: 2, 4 or 8. */
ob_status ob_qb_sizes(const ob_ctx* ctx, int bits, size_t* words_per_worker,
                      size_t* n_blocks);

/* e = 0 for every worker and e_s = 0 (start of the compressed phase, and
 * the periodic reset of [BLOG] 4.1) for the codecs whose errors are kept in
 * plain form. */
ob_status ob_zero_errors(ob_ctx* ctx, float* const* err, float* err_s, ob_stream_t stream);

/* Worker compression, all W workers:
 *   m_w = b1*m + (1-b1)*g_w;  x = m_w + e_w (clamped if clip_value > 0)
 *   per block: codes, bscales, e_w := x - q*scale.  m is not written. */
ob_status ob_compress_qb(ob_ctx* ctx, int bits, const void* const* grads, const float* m,
                         float* const* err, uint32_t* codes, float* bscales, uint64_t seed,
                         uint64_t step, ob_stream_t stream);

/* Server average and re-compression:
 *   z = (sum over w in order, from 0, of q_w*scale_w)/W;  y = e_s + z
 *   per block: scodes [words_per_worker], sbscales [n_blocks],
 *   e_s := y - q*sscale. */
ob_status ob_server_reduce_qb(ob_ctx* ctx, int bits, const uint32_t* codes,
                              const float* bscales, float* err_s, uint32_t* scodes,
                              float* sbscales, uint64_t seed, uint64_t step,
                              ob_stream_t stream);

/* m = q*sscale; p -= lr*(m/(sqrt(v_frozen)+eps)).  Padding: m = 0, p is
 * not written. */
ob_status ob_adam_step_qb(ob_ctx* ctx, int bits, const uint32_t* scodes, const float* sbscales,
                          const float* v_frozen, float* m, float* p, ob_stream_t stream);

/* FP16 codec.  send != 0 on the steps the group is exchanged (every 10th
 * in [BLOG] 3.2); h: [W][n_pad] uint16 (IEEE binary16 bit patterns).
 *   x = b1*m + (1-b1)*g_w + e_w (clamped if clip_value > 0)
 *   send:  h_w = f16(x) (nearest, ties to even); e_w := x - f32(h_w)
 *   else:  e_w := x; h untouched (may be NULL). */
ob_status ob_compress_f16(ob_ctx* ctx, int send, const void* const* grads, const float* m,
                          float* const* err, uint16_t* h, ob_stream_t stream);

/* Sending steps only: z = (sum over w, in order, from 0, of f32(h_w))/W;
 * y = e_s + z; hs = f16(y); e_s := y - f32(hs).  hs: [n_pad]. */
ob_status ob_server_reduce_f16(ob_ctx* ctx, const uint16_t* h, float* err_s, uint16_t* hs,
                               ob_stream_t stream);

/* send: m = f32(hs); p -= lr*(m/(sqrt(v_frozen)+eps)).  Otherwise m = 0 and
 * p is left as it is (hs, v_frozen, p may be NULL).  Padding: m = 0. */
ob_status ob_adam_step_f16(ob_ctx* ctx, int send, const uint16_t* hs, const float* v_frozen,
                           float* m, float* p, ob_stream_t stream);

/* One compressed step of a codec group of width `bits` (2, 4, 8 or 16) at
 * compressed step t >= 1, following ob_plan_step(ctx, bits, t): the errors
 * are zeroed first if `reset`; then, width 2/4/8: ob_compress_qb,
 * ob_server_reduce_qb, ob_adam_step_qb with the plan's key and step, msg =
 * codes [W][words_per_worker] u32, msg_scales = bscales, smsg = scodes,
 * smsg_scales = sbscales; width 16: ob_compress_f16 with the plan's send,
 * then (sending steps) ob_server_reduce_f16 and ob_adam_step_f16, msg = h
 * [W][n_pad] u16, smsg = hs [n_pad] u16, the two scale pointers unused
 * (may be NULL).  Arguments as for those calls. */
ob_status ob_codec_step(ob_ctx* ctx, int bits, uint64_t t, const void* const* grads, float* m,
                        float* const* err, void* msg, float* msg_scales, float* err_s,
                        void* smsg, float* smsg_scales, const float* v_frozen, float* p,
                        ob_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OB_H */
