/*
 * moe.h — C ABI of the routed block-scaled mixture-of-experts layer for
 * GB300 (sm_103a).
 *
 * The layer is the routed MoE of Inkling 2 Small: hidden H = 4608, E = 384
 * routed experts, top-k = 8, expert FFN width F = 2304, no shared experts,
 * soft-capped SwiGLU, expert weights in NVFP4 (W4A4) or MXFP8 (W8A8).
 * Sources (pages on the Inkling 2 Small release):
 *   [SGL]  "SGLang and Miles Add Day-0 Support for Inkling 2 Small",
 *          section Performance (MegaMoE and kernel-fusion bullets).
 *   [CB]   "Inkling-2-Small" SGLang cookbook, section 2 Configuration Tips
 *          (Checkpoints, Parallelism, MegaMoE paragraphs).
 *   [TS]   "TML Inkling 2 Small at Day 0" (TokenSpeed), table "What's new"
 *          (MoE and Checkpoint rows) and section "Serving ... on the
 *          TokenSpeed stack".
 *   [MI]   "inkling-2-small" Miles docs, section 1 Model Introduction and
 *          section 5.3 Rollout and precision.
 *
 * Conventions for every call:
 *   - Pointers named *_dev are device pointers; the caller owns every buffer,
 *     the workspace and the stream.  The library allocates no device memory
 *     and keeps no state besides per-device set-up done on first use (kernel
 *     shared-memory limits, the device address of moe_route_noalloc's
 *     scratch).  That set-up belongs to the device's current context: after
 *     cudaDeviceReset the library must not be called again in the process.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, passed as void*).
 *   - On invalid arguments a call returns a non-zero status and enqueues
 *     nothing.  Checks: shapes (see moe_config), 16-byte alignment of every
 *     pointer, workspace size, device compute capability 10.3.
 *   - A CUDA launch error is returned as MOE_ERR_CUDA.  Device-side bounded
 *     waits that ran out are recorded in the workspace status word and are
 *     reported by moe_poll_device_status.
 *   - Inputs must be finite; NaN/Inf behaviour is unspecified.
 *   - Row-major everywhere; the reduction (K) dimension is contiguous.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED_SHAPE = 2,
  MOE_ERR_MISALIGNED = 3,
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_ARCH = 5,
  MOE_ERR_CUDA = 6,
  MOE_ERR_DEVICE_TIMEOUT = 7,
  MOE_ERR_BOUNDS = 8
} moe_status;

/* Expert weight / activation encodings [CB Checkpoints; TS Checkpoint row;
 * MI 5.3: W4A4 / W8A8]:
 *   NVFP4: E2M1 codes packed two per byte (low nibble = lower k), one E4M3
 *          scale per 16 elements along K, one fp32 global decode factor g
 *          (per expert matrix for weights, per token row for activations):
 *          value = e2m1(code) * e4m3(scale) * g.
 *   MXFP8: E4M3 codes, one E8M0 scale per 32 elements along K:
 *          value = e4m3(code) * 2^(scale - 127). */
typedef enum { MOE_FMT_NVFP4 = 0, MOE_FMT_MXFP8 = 1 } moe_format;

/* Layout of block-scale bytes.
 *   ROWMAJOR: scales[r][c], c = k / block, shape [rows, K/block].
 *   TILED:    the layout the expert GEMMs consume: rows padded to a multiple
 *             of 128 and scale columns to a multiple of 4; the byte of
 *             (r, c) sits at
 *               ((r/128) * (C/4) + c/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + c%4
 *             with C the (padded) number of scale columns.  Same byte count
 *             as ROWMAJOR when rows%128 == 0 and C%4 == 0. */
typedef enum { MOE_SCALES_ROWMAJOR = 0, MOE_SCALES_TILED = 1 } moe_scale_layout;

/* Format of the expert outputs y (the rows the down GEMM writes and the
 * combine reads, before the routing weights apply; the pages do not fix it):
 *   MOE_Y_FP32:  fp32 [P, H].
 *   MOE_Y_FP16E: fp16 significands with a power-of-two exponent per 32
 *     features.  For row p and feature block b (features 32b .. 32b+31),
 *     amax = max |y| over the block and
 *       e = 0 if amax = 0, else max(floor(log2 amax) - 14, -110),
 *       code = fp16_rne(y * 2^-e),   y decoded = code * 2^e,
 *     so every block's largest value lands in [2^14, 2^15) of the fp16
 *     range: nothing overflows and each element keeps 11 significant bits
 *     (|error| <= 2^-11 |y|).  Layout: the fp16 codes [P, H], then the int8
 *     exponents [P, H/32].  Half the bytes of fp32 between the down GEMM
 *     and the combine. */
typedef enum { MOE_Y_FP32 = 0, MOE_Y_FP16E = 1 } moe_y_format;

/* Layer shape and options.
 *   T tokens (1..65536), H hidden, E experts (1..1024), k experts per token
 *   (1..min(E,32)), F expert FFN width.  H and F must be multiples of 256 for
 *   NVFP4 and of 128 for MXFP8, and at most 16384.
 *   swiglu_cap: c in cap(v) = c*tanh(v/c), applied to the gate and up
 *     pre-activations; 0 disables the cap.  Default 10.  [TS MoE row and MI 1
 *     call the activation a capped / soft-capped SwiGLU but give neither the
 *     form nor the constant, so both are this parameter.]
 *   act_global_mode: NVFP4 only.  The FP32 global scale of the activations
 *     (x and h rows): 0 = dynamic, from each row's absolute maximum over its
 *     full width (default; G = 2688 / amax, decode factor g = 1/G); 1 =
 *     static per expert: the caller passes decode factors g_x[e], g_h[e]
 *     (act_static_scales of moe_expert_ffn / moe_forward) and a row routed to
 *     expert e is encoded with G = 1/g (fp32), block maxima beyond 2688 g
 *     saturating.  [CB Parallelism paragraph: the activation scales must
 *     cover an expert's full input width; the pages fix no granularity, so
 *     both readings are offered.]  MXFP8 requires 0.
 *   mx_scale_mode: MXFP8 only.  0 = OCP rule X = 2^(floor(log2 amax) - 8)
 *     (default; block maxima in (448, 512)*X saturate); 1 = X =
 *     2^ceil(log2(amax/448)) (never saturates).
 *   bias_in_weights: 0 (default) = the router bias steers selection only and
 *     the weights normalise the unbiased sigmoid scores; 1 = weights
 *     normalise the biased keys.
 *   routed_scale: multiplies the normalised routing weights (default 1).
 *   ffn_schedule: how the expert FFN runs for decode batches (64-row token
 *     tiles, T * k < 64 * E): 0 (default) = from 64 pairs (T * k >= 64) one
 *     persistent kernel for GEMM1, the h quantisation and GEMM2, a down
 *     tile starting as soon as its h rows exist, separate kernels below;
 *     1 = separate kernels always.  The results are the same bit for bit.
 *     Prefill batches always use separate kernels.
 *   y_format: moe_y_format of the expert outputs (the buffers that
 *     moe_expert_ffn writes and moe_combine reads, and the workspace's y
 *     rows in moe_forward).  MOE_Y_FP16E is the faster choice; a zeroed
 *     config gets MOE_Y_FP32. */
typedef struct {
  int T, H, E, k, F;
  moe_format fmt;
  float swiglu_cap;
  int act_global_mode;
  int mx_scale_mode;
  int bias_in_weights;
  float routed_scale;
  int ffn_schedule;
  int y_format;
} moe_config;

/* One quantised expert matrix for all E experts (device pointers).
 *   gate, up: N = F rows, K = H;  down: N = H rows, K = F.
 *   codes:  NVFP4 u8 [E, N, K/2];  MXFP8 u8 [E, N, K].
 *   scales: TILED layout over the E*N rows (moe_quantize with
 *           MOE_SCALES_TILED, or moe_pack_scales from ROWMAJOR).
 *   global_scale: NVFP4 fp32 [E] decode factors; MXFP8: NULL. */
typedef struct {
  const void* codes;
  const void* scales;
  const float* global_scale;
} moe_qweight;

/* Bytes of workspace that moe_route / moe_dispatch / moe_expert_ffn /
 * moe_forward need for this configuration.  The workspace must be 256-byte
 * aligned; its contents need no initialisation. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Fused router [SGL Performance, kernel-fusion bullet: sigmoid, bias and
 * top-k selection share one kernel; MI 1: sigmoid routing over 384 experts,
 * 8 per token].
 *   x_dev        bf16 [T, H] tokens
 *   w_router_dev bf16 [E, H]
 *   bias_dev     fp32 [E]
 *   topk_idx_dev int32 [T, k] (out): experts by descending key = s + bias,
 *                s = sigmoid(x . w_e); ties go to the lower expert index.
 *   topk_w_dev   fp32 [T, k] (out): routed_scale * s_j / sum_i s_i.
 * Logits accumulate in fp32 in chunks of 32 products, the chunk sums
 * compensated (Kahan): |error| <= 40 * 2^-24 * sum_h |x_h w_eh|.  For T > 256
 * (and E % 16 == 0) the logits are first computed on the tensor cores, and
 * only the experts that can reach the top-k within 2^-11 ||x|| ||w_e|| of
 * tensor-core rounding are recomputed with that bound; the selection and the
 * weights use the recomputed logits.  The status word of the workspace is
 * cleared, and set on a bounded-wait timeout (moe_poll_device_status). */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                     const float* bias_dev, int32_t* topk_idx_dev, float* topk_w_dev,
                     void* ws_dev, size_t ws_bytes, void* stream);

/* The router of moe_route for callers that cannot allocate device memory
 * when they route (inside a captured CUDA graph region, in a plugin without
 * access to its host framework's allocator, or in a runtime that forbids
 * allocation after start-up).  The pages have no counterpart: it is an
 * interface convenience, with the same arguments and results as moe_route
 * but no workspace.
 *   Its scratch (a status word area and the fp32 logits) is a fixed 4 MiB
 *   array inside the library, reserved on every device that loads the
 *   library until the process exits.  Configurations whose scratch does not
 *   fit return MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued:
 *     T <= 256 (CUDA-core router): 64 + splits * T * E <= 2^20 floats, where
 *       splits is the largest s <= 24 (T <= 64) or <= 8 (T <= 256) with
 *       H % (64*s) == 0; every T <= 256 fits at E = 384, H = 4608;
 *     T > 256 with E % 16 == 0 and H % 64 == 0 (tensor-core router):
 *       64 + T * E + ceil(E/64)*64 <= 2^20; at E = 384 exactly T <= 2729.
 *   The first call on a device looks up the array's device address; make that
 *   first call before any stream capture.
 *   Every call uses the same array: calls that may overlap on the GPU (other
 *   streams, other threads) race and must be serialised by the caller.  No
 *   call allocates or frees memory.
 *   A bounded wait of the tensor-core router that ran out is recorded in the
 *   array's status word: moe_route_noalloc_poll_status reads it. */
MOE_API moe_status moe_route_noalloc(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                                     const float* bias_dev, int32_t* topk_idx_dev, float* topk_w_dev,
                                     void* stream);

/* Status of the last moe_route_noalloc call(s) on the current device:
 * synchronises `stream`, reads and clears the status word of the library's
 * fixed router scratch.  Returns MOE_ERR_DEVICE_TIMEOUT if a bounded wait ran
 * out (topk_idx / topk_w are then unspecified), MOE_OK otherwise.  Allocates
 * nothing. */
MOE_API moe_status moe_route_noalloc_poll_status(void* stream);

/* Token dispatch [CB MegaMoE: dispatch is a step of the fused unit]: groups
 * the P = T*k pairs (t, j)
 * by expert, and within an expert by token.
 *   topk_idx_dev int32 [T, k]: each row k distinct experts in [0, E), as
 *                moe_route writes them (entries outside [0, E) are ignored,
 *                and leave perm / pair_pos entries unwritten)
 *   counts_dev   int32 [E] (out)     pairs per expert
 *   offsets_dev  int32 [E+1] (out)   exclusive scan of counts
 *   perm_dev     int32 [P] (out)     perm[p] = t*k + j, sorted by (e, t)
 *   pair_pos_dev int32 [T, k] (out)  inverse: pair_pos[t*k + j] = p
 * Deterministic. */
MOE_API moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx_dev, int32_t* counts_dev,
                        int32_t* offsets_dev, int32_t* perm_dev, int32_t* pair_pos_dev,
                        void* ws_dev, size_t ws_bytes, void* stream);

/* Expert FFN of every pair [CB MegaMoE: the fused unit holds the two expert
 * GEMMs and the capped SwiGLU between them; TS: the expert GEMMs run on
 * block-scaled tensor cores; SGL kernel-fusion bullet: activation
 * quantisation lives inside the expert GEMMs; MI 5.3: W4A4 / W8A8]:
 *   a   = quantise(x_t) per token over the full H (NVFP4: per-row global,
 *         or expert e's static global in act_global_mode 1)
 *   g,u = W_gate,e a , W_up,e a          (tcgen05 block-scaled MMA, fp32)
 *   h   = bf16( silu(cap g) * cap u )
 *   y_p = W_down,e quantise(h)           (NVFP4: per-row global over F;
 *                                         MXFP8: quantised in GEMM1's epilogue)
 *   x_dev        bf16 [T, H]
 *   topk_idx_dev, offsets_dev, perm_dev, pair_pos_dev: from moe_route /
 *                moe_dispatch (the tile plan is rebuilt from offsets_dev)
 *   gate/up/down quantised weights (see moe_qweight)
 *   act_static_scales fp32 [E, 2] (g_x[e], g_h[e]) when act_global_mode = 1,
 *                else NULL (ignored)
 *   y_perm_dev   (out) the P rows y_p in perm order, in cfg->y_format
 *                (moe_y_bytes bytes, 16-byte aligned). */
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* x_dev, const int32_t* topk_idx_dev,
                          const int32_t* offsets_dev, const int32_t* perm_dev,
                          const int32_t* pair_pos_dev, const moe_qweight* gate,
                          const moe_qweight* up, const moe_qweight* down,
                          const float* act_static_scales, void* y_perm_dev,
                          void* ws_dev, size_t ws_bytes, void* stream);

/* Bytes of the y rows of this configuration in its y_format: P*H*4 (fp32)
 * or P*H*2 + P*H/32 (fp16 codes, then exponents), P = T*k. */
MOE_API moe_status moe_y_bytes(const moe_config* cfg, size_t* bytes);

/* Weighted combine [CB MegaMoE: the combine ends the fused unit]:
 *   out[t] = bf16_rne( sum_{j=0..k-1} topk_w[t,j] * y_perm[pair_pos[t,j]] ),
 * summed in fp32 in slot order (deterministic), y_perm the decoded rows.
 * For MOE_Y_FP16E each product is fma(topk_w * 2^e, code, sum) (the weight
 * times a power of two is exact), i.e. the same sum over the decoded values.
 *   y_perm_dev rows in cfg->y_format (as moe_expert_ffn writes them);
 *   topk_w_dev fp32 [T, k]; pair_pos_dev int32 [T, k]; out_dev bf16 [T, H]
 *   (out). */
MOE_API moe_status moe_combine(const moe_config* cfg, const void* y_perm_dev, const float* topk_w_dev,
                       const int32_t* pair_pos_dev, void* out_dev, void* stream);

/* The whole layer in one call: moe_route, moe_dispatch, moe_expert_ffn and
 * moe_combine chained on `stream` with every intermediate in the workspace
 * [CB MegaMoE: one fused unit per layer; SGL: programmatic dependent
 * launch between kernels].  act_static_scales as for moe_expert_ffn.
 * out_dev bf16 [T, H]. */
MOE_API moe_status moe_forward(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                       const float* bias_dev, const moe_qweight* gate, const moe_qweight* up,
                       const moe_qweight* down, const float* act_static_scales, void* out_dev,
                       void* ws_dev, size_t ws_bytes, void* stream);

/* Number of kernels one moe_forward call launches for this configuration
 * (2 or 3 router + 1 or 3 dispatch + x quantisation + either the fused
 * decode FFN, or GEMM1 + h quantisation unless GEMM1 did it + GEMM2; +
 * combine).  Host-only; no device is touched.
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE as moe_forward's checks. */
MOE_API moe_status moe_forward_kernel_count(const moe_config* cfg, int* count);

/* moe_forward, also recording events[i] (cudaEvent_t handles, created by the
 * caller) on `stream` at the start of stage i and events[MOE_NUM_STAGES] after
 * the last, so that the caller can time each stage:
 *   0 router (logits, top-k)      1 dispatch (bitmap, scan, scatter)
 *   2 x quantisation              3 GEMM1 gate/up + capped SwiGLU
 *   4 h quantisation (empty when GEMM1 did it)  5 GEMM2 down
 *   6 combine
 * Same results as moe_forward. */
#define MOE_NUM_STAGES 7
MOE_API moe_status moe_forward_profiled(const moe_config* cfg, const void* x_dev, const void* w_router_dev,
                                        const float* bias_dev, const moe_qweight* gate, const moe_qweight* up,
                                        const moe_qweight* down, const float* act_static_scales, void* out_dev,
                                        void* ws_dev, size_t ws_bytes, void* stream, void* const* events);

/* Block quantiser [MI 1 and 5.2: weight sync re-encodes experts in the layer's
 * format and recomputes NVFP4 global scales].  Encodes rows x cols values.
 *   src_is_fp32: 1 = src fp32, 0 = src bf16.
 *   group_rows:  NVFP4 global-scale granularity: 0 = one global per row
 *                (activations); G > 0 = one global per G consecutive rows
 *                (weights: G = N, one per expert matrix); rows % G == 0.
 *                Ignored for MXFP8.
 *   codes_dev:   NVFP4 u8 [rows, cols/2]; MXFP8 u8 [rows, cols].
 *   scales_dev:  ROWMAJOR [rows, cols/bs] or TILED (rows % 128 == 0 and
 *                (cols/bs) % 4 == 0 required).
 *   global_dev:  NVFP4 fp32 [rows] or [rows/G]; MXFP8: NULL.
 * NVFP4 steps (fp32, each rounded to nearest): G = 2688/amax (1 if amax = 0),
 * g = 1/G, scale = E4M3((amax_b/6)*G), code = E2M1(v * (G/scale)).
 * MXFP8: scale as mx_scale_mode, code = E4M3(v * 2^(127 - scale)).
 * Conversions round to nearest even and saturate; zero keeps its sign. */
MOE_API moe_status moe_quantize(moe_format fmt, int mx_scale_mode, int src_is_fp32, const void* src_dev,
                        int64_t rows, int64_t cols, int64_t group_rows, moe_scale_layout layout,
                        void* codes_dev, void* scales_dev, float* global_dev, void* stream);

/* Fake quantisation [MI 5.3: full-parameter training fake-quantises the
 * expert weights to their layer's format with a straight-through gradient]:
 * out = decode(encode(src)) in fp32, bit for bit the value the layer's GEMMs
 * see (encode as moe_quantize; decode e2m1*scale*g or e4m3*2^(s-127), one
 * fp32 rounding).  Its gradient is the identity (straight-through), so a
 * trainer applies it in the forward pass and passes gradients unchanged.
 *   out_dev fp32 [rows, cols]; global_dev as in moe_quantize (NVFP4 only;
 *   receives the decode factors). */
MOE_API moe_status moe_fake_quantize(moe_format fmt, int mx_scale_mode, int src_is_fp32, const void* src_dev,
                                     int64_t rows, int64_t cols, int64_t group_rows, float* out_dev,
                                     float* global_dev, void* stream);

/* MXFP8 KV-cache quantiser [SGL features table: a block-scaled MXFP8 KV cache
 * on Blackwell]: the new K (or V) rows of a batch are encoded along head_dim
 * with the layer's MXFP8 rule (32-element blocks, E8M0 scale as
 * mx_scale_mode, E4M3 codes, round to nearest even, saturating) and written to
 * their slots of a cache.
 *   kv_dev       bf16 [tokens, heads, head_dim]; token t's row starts at
 *                element t * token_stride (token_stride >= heads * head_dim,
 *                a multiple of 8, e.g. K inside a fused [tokens, 3, heads,
 *                head_dim] projection); 16-byte aligned.
 *   slot_dev     int64 [tokens] (nullable, 8-byte aligned): the cache slot of
 *                token t; slots < 0 or >= num_slots are skipped (padding
 *                tokens).  NULL: token t goes to slot t (num_slots >= tokens).
 *   codes_dev    u8 E4M3 [num_slots, heads, head_dim] (16-byte aligned)
 *   scales_dev   u8 E8M0 [num_slots, heads, head_dim / 32]
 *   value = e4m3(code) * 2^(scale - 127); an all-zero block has scale 0.
 * head_dim % 32 == 0, 32..1024; heads 1..4096; tokens 0..2^31-1 (0 enqueues
 * nothing).  Slots of other tokens are left untouched; two tokens mapped to
 * one slot race. */
MOE_API moe_status moe_kv_quantize_mxfp8(const void* kv_dev, int64_t tokens, int heads, int head_dim,
                                         int64_t token_stride, const int64_t* slot_dev, int64_t num_slots,
                                         int mx_scale_mode, void* codes_dev, void* scales_dev, void* stream);

/* ROWMAJOR -> TILED scale re-layout (rows % 128 == 0, scale columns % 4 == 0). */
MOE_API moe_status moe_pack_scales(const void* rowmajor_dev, int64_t rows, int64_t scale_cols, void* tiled_dev,
                           void* stream);

/* Synchronises `stream`, reads and clears the workspace status word.
 * Returns MOE_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out. */
MOE_API moe_status moe_poll_device_status(void* ws_dev, void* stream);

/* Block-scaled tensor-core peak, measured [TS serving section: the expert
 * GEMMs run on block-scaled tensor cores; the prefill roofline divides by
 * this rate].  Launches one CTA on every SM (*ctas receives the count); each
 * issues mmas_per_cta (a multiple of 4) back-to-back tcgen05 block-scaled
 * MMAs of M = 128, N = 256 from one thread into one TMEM accumulator, the
 * operands and scales resident in shared memory and TMEM (no global memory
 * traffic): NVFP4 kind::mxf4nvf4 scale_vec::4X (K = 64), MXFP8
 * kind::mxf8f6f4 scale_vec::1X (K = 32), the forms the expert GEMMs issue.
 * *flops_per_mma receives 2*128*256*K.  The caller times the launch with
 * events on `stream`: rate = ctas * mmas_per_cta * flops_per_mma / time.
 *   cycles_dev   u64 [*ctas] (nullable): each CTA's SM cycles from its first
 *                MMA to the completion of its last
 *   status_dev   a 4-byte word (4-byte aligned), cleared here; a bounded wait
 *                that ran out sets it (read it with moe_poll_device_status).
 * Allocates nothing. */
MOE_API moe_status moe_bench_mma_peak(moe_format fmt, int64_t mmas_per_cta, unsigned long long* cycles_dev,
                                      void* status_dev, int* ctas, double* flops_per_mma, void* stream);

/* Index checks of the bounds-checked build.  The library can be built with
 * MOE_DEBUG_BOUNDS defined (a separate libmoe_debug.so): the indices its
 * kernels derive from data (pair positions, padded activation rows, canonical
 * pair rows, row-tile indices) are then checked before the accesses they
 * address, and a failed check skips the access and sets a device flag
 * instead of reading or writing out of bounds (nothing traps).  This call
 * synchronises `stream`, then reads and clears the flags of the current
 * device: MOE_ERR_BOUNDS if a check failed since the last call, MOE_OK
 * otherwise.  *checked = 1 in the checked build; in the normal build
 * *checked = 0 and the call returns MOE_OK without touching the device.
 * site (nullable): the source line of a failed check, for diagnosis (0 if
 * none). */
MOE_API moe_status moe_debug_bounds_status(void* stream, int* checked, int* site);

/* Test hook for the device-side failure detection: launches the gate/up GEMM
 * over the tile plan already in the workspace (a moe_forward or
 * moe_expert_ffn must have run on it) with its loads withheld and every
 * bounded wait limited to limit_cycles (1000 .. 4e9) SM cycles, so that the
 * waits run out and the kernel exits with a timeout bit in the workspace
 * status word, which moe_poll_device_status then reports as
 * MOE_ERR_DEVICE_TIMEOUT.  The device stays usable. */
MOE_API moe_status moe_selftest_bounded_wait(const moe_config* cfg, const moe_qweight* gate, const moe_qweight* up,
                                             void* ws_dev, size_t ws_bytes, int64_t limit_cycles, void* stream);

/* Test hook for the fused decode FFN's dependency waits (decode batches,
 * 64-row tiles; a moe_forward or moe_expert_ffn must have run on the
 * workspace): launches the fused kernel with its gate/up tiles' completion
 * reports withheld and every bounded wait limited to limit_cycles (1000 ..
 * 4e9) SM cycles, so that the down tiles' waits for their h rows run out and
 * the kernel exits with a timeout bit in the workspace status word
 * (moe_poll_device_status: MOE_ERR_DEVICE_TIMEOUT).  The device stays
 * usable; the workspace's y rows are unspecified afterwards. */
MOE_API moe_status moe_selftest_dependency_wait(const moe_config* cfg, const moe_qweight* gate,
                                                const moe_qweight* up, const moe_qweight* down, void* ws_dev,
                                                size_t ws_bytes, int64_t limit_cycles, void* stream);

/* Byte offsets of the layer's intermediates inside the workspace, for
 * inspection by tests (all buffers in padded expert-row order: each expert's
 * rows start at a multiple of tile_rows = NT).  R = padded row capacity.
 * ffn_sync: the fused decode FFN's counters (per row tile a completion count
 * and a ready flag, a tile counter, per padded row the |h| maximum).  The
 * activation block scales (xq_scales, hq_scales) use one 512-byte atom per
 * NT-row tile and 4 scale columns: row r, column c at
 *   ((r/NT)*(C/4) + c/4)*512 + (r%NT%32)*16 + (r%NT/32)*4 + c%4.
 * h_bf16 is empty (sharing its offset with hq_codes) when GEMM1's epilogue
 * quantises h itself: MXFP8. */
typedef struct {
  int64_t R;
  int64_t tile_rows; /* token rows per expert tile: 64 (decode) or 128 */
  size_t status, logits, topk_idx, topk_w, counts, offsets, perm, pair_pos, bitmap, seg_start,
      tiles, rt_base, ffn_sync, xq_codes, xq_scales, xq_global, h_bf16, hq_codes, hq_scales, hq_global,
      y_perm, total;
} moe_ws_layout;
MOE_API moe_status moe_workspace_layout(const moe_config* cfg, moe_ws_layout* layout);

MOE_API const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
