/*
 * fmad.h - C ABI of the GB300 flow-matching action decoder (libfmad.so).
 *
 * The library runs the single-batch flow-matching action-decoder loop of a
 * vision-language-action policy (FlashRT-PAI pages): L transformer layers x S
 * Euler denoise steps over an M-row action chunk. Each layer is
 *   AdaRMSNorm (x / sqrt(mean(x^2) + eps) * (1 + scale) + shift, fixed gamma
 *     folded into the next GEMM's weights W' = diag(gamma) W)
 *   -> static-scale quantise -> QKV GEMM (split along K)
 *   -> attention of the chunk over [persistent prefix KV cache; chunk KV]
 *   -> O GEMM -> gated residual + AdaRMSNorm + quantise
 *   -> gate|up GEMM -> GeGLU + quantise -> down GEMM
 *   -> gated residual + the next layer's AdaRMSNorm + quantise.
 * Sources: blog post "Embodied inference acceleration: first ask how old the
 * observation is" (sections "CUDA Graph vs graph simplification": RMSNorm,
 * gamma fold, QKV merge, CUDA Graph replay; "Static quantisation": static
 * activation scales, fused gated residual + AdaRMSNorm + FP8 convert, next
 * layer's condition parameters; "Small-M GEMM": K-split with FP32 partials
 * reduced before the consumer's transform); news article "FlashRT-PAI"
 * (section "It optimises the relay": launch overlap with Programmatic
 * Dependent Launch, the execution contract of named persistent buffers with
 * reuse of instruction-dependent state and selective refresh of
 * image-dependent state, and execution-state capsules that snapshot and
 * restore in-process state bound to the plan and device addresses).
 *
 * Conventions for every entry point:
 *   - Returns int status (fm_status). No exceptions, aborts or device traps.
 *   - The caller owns ALL device memory, including the workspace; the library
 *     never allocates or frees device memory. Pointers documented "device"
 *     must be device pointers on the current CUDA device; "host" pointers are
 *     ordinary host memory (pinned recommended for async copies).
 *   - Work is stream-ordered on the given cudaStream_t (passed as void*; NULL
 *     means the legacy default stream) and asynchronous unless noted.
 *   - A policy is used from one stream at a time.
 *   - Matrices are row-major; "[R][C]" means R rows of C contiguous elements.
 *   - fp8 means OCP E4M3 (E4M3FN: max 448, no infinities), one byte per code;
 *     bf16 tensors are passed as uint16_t bit patterns.
 */
#ifndef FMAD_H
#define FMAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FM_ABI_VERSION 3

typedef enum fm_status {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,     /* NULL pointer, bad enum, bad ABI version */
  FM_ERR_SHAPE = 2,           /* a size violates a documented precondition */
  FM_ERR_ALIGN = 3,           /* a pointer is not 16-byte (workspace: 1024-byte) aligned */
  FM_ERR_WORKSPACE = 4,       /* workspace smaller than fm_workspace_size() */
  FM_ERR_CUDA = 5,            /* a CUDA runtime call failed; see fm_last_error() */
  FM_ERR_STATE_MISMATCH = 6,  /* capsule from another plan, policy or address */
  FM_ERR_DEVICE = 7,          /* a kernel gave up a bounded wait and set the error word */
  FM_ERR_UNSUPPORTED = 8      /* valid request this library does not implement */
} fm_status;

typedef enum fm_format {
  FM_FMT_BF16 = 0,   /* bf16 operands, no quantisation */
  FM_FMT_FP8 = 1,    /* E4M3 codes with a static per-tensor scale */
  FM_FMT_NVFP4 = 2   /* E2M1 + E4M3 scale per 16 along K + fp32 tensor scale (weights: all three
                        fixed at create; activations: static tensor scale, block scales taken
                        from the activation at run time) */
} fm_format;

enum {
  FM_FLAG_USE_GRAPH = 1u,  /* replay the whole decision as one CUDA graph */
  FM_FLAG_USE_PDL = 2u,    /* launch every kernel with Programmatic Dependent Launch */
  /* FP8/BF16: run the consumers inside the GEMMs (5 kernels per layer instead of 7): the
   * O and down GEMM epilogues apply the gated residual and emit per-tile sums of squares
   * of x, the QKV and gate|up GEMMs normalise and quantise x in a prologue. Off by
   * default: every CTA of those GEMMs re-reads the fp32 x of its K range, which at M = 50
   * costs more than the two kernel boundaries it removes. Taken only where the shapes
   * allow it (the O and down GEMMs reduce every K slice in one cluster of <= 8, the QKV
   * and gate|up GEMMs hold their K range in one stage); otherwise, and for NVFP4, the
   * flag is ignored: fm_test_kernel_count reports the placement in use. */
  FM_FLAG_FUSED_CONSUMERS = 4u,
  /* FP8 weights and activations, d <= 1024, H * Dh <= 1024, M <= 64: run the O projection
   * and its consumer (gated residual + pre-MLP AdaRMSNorm + quantise) as one kernel whose
   * thread-block cluster spans every column tile, each CTA over the whole K, so each row's
   * norm is finished inside it (6 kernels per layer). Off by default: eight CTAs carry the
   * whole projection and the cluster's row statistics, which at M = 50 takes longer than
   * the row kernel and hand-off it removes (expert_fp8_m50: 6.26 ms against 5.80 ms).
   * Ignored where the shapes do not allow it; fm_test_kernel_count reports the placement. */
  FM_FLAG_O_CONSUMER_IN_GEMM = 8u
};

enum {
  FM_COND_TIME = 0,   /* cond of step k = sinusoidal embedding of t_k = 1 - k/S */
  FM_COND_GIVEN = 1   /* cond of step k = caller-supplied vector (fm_weights.conds) */
};

/* Activation quant points per layer, the column index of the [L][4] scale table
 * ([L][7] with FP8 attention: columns 4-6 are the static scales of Q, K and V,
 * the prefix cache's keys and values included). */
enum {
  FM_SITE_ATTN_IN = 0,   /* pre-attention AdaRMSNorm output (QKV GEMM input) */
  FM_SITE_ATTN_OUT = 1,  /* attention output (O GEMM input) */
  FM_SITE_MLP_IN = 2,    /* pre-MLP AdaRMSNorm output (gate|up GEMM input) */
  FM_SITE_GEGLU = 3,     /* GeGLU output (down GEMM input) */
  FM_SITE_Q = 4,         /* FP8 attention: queries */
  FM_SITE_K = 5,         /* FP8 attention: keys (chunk and prefix) */
  FM_SITE_V = 6          /* FP8 attention: values (chunk and prefix) */
};

/* Policy shape and options. Preconditions (FM_ERR_SHAPE otherwise):
 *   d, F and H*Dh multiples of 128; Dh == 128; H a multiple of Hkv;
 *   1 <= M <= 256; 1 <= A <= 32; P >= 0; L, S >= 1; 0 <= warm_t <= 1 (warm_t > 0
 *   requires FM_COND_TIME);
 *   ksplit[i] (0 = automatic) divides the GEMM's K/128-byte block count.
 * weight_fmt FP8 requires act_fmt FP8, BF16 requires BF16, NVFP4 takes FP8 or NVFP4
 * (four-bit weights and activations: the activation scale table then holds each quant
 * point's static tensor scale, amax / (448 * 6)). With NVFP4 weights the K-split counts
 * 64-element blocks, the gate|up GEMM is not split (ksplit[2] 0 or 1), and a
 * layer runs 8 kernels (the QKV partial planes are reduced by their own kernel). */
typedef struct fm_config {
  int abi_version;     /* must be FM_ABI_VERSION */
  int L, S, M, d, H, Hkv, Dh, F, P, A;
  int weight_fmt;      /* fm_format */
  int act_fmt;         /* fm_format (FP8, BF16, or NVFP4 with NVFP4 weights) */
  int attn_fmt;        /* fm_format of the attention operands: BF16, or FP8 (E4M3 Q, K, V
                          with static scales and probabilities coded E4M3(P * 448));
                          FP8 requires FP8 weights and activations */
  int cond_mode;       /* FM_COND_TIME or FM_COND_GIVEN */
  float rms_eps;       /* AdaRMSNorm epsilon */
  int ksplit[4];       /* K-split of the QKV, O, gate|up and down GEMMs; 0 = auto */
  unsigned flags;      /* FM_FLAG_* */
  float warm_t;        /* flow time of the one-step warm start (fm_decode_warm); 0 = none */
} fm_config;

/* One layer's raw parameters (device pointers, read only during policy_create).
 * GEMM weights are fp32 in [out][in] layout (y = x W^T):
 *   w_qkv [(H+2Hkv)*Dh][d] (rows: Q heads, then K heads, then V heads),
 *   w_o [d][H*Dh], w_gu [2F][d] (rows 0..F-1 gate, F..2F-1 up), w_d [d][F].
 * gamma1 [d] folds into w_qkv's columns, gamma2 [d] into w_gu's columns.
 * w_mod bf16 [6d][d], b_mod fp32 [6d]: modulation = cond . w_mod^T + b_mod,
 * split as [scale1, shift1, gate1, scale2, shift2, gate2]. */
typedef struct fm_layer_weights {
  const float* w_qkv;
  const float* w_o;
  const float* w_gu;
  const float* w_d;
  const float* gamma1;
  const float* gamma2;
  const uint16_t* w_mod;
  const float* b_mod;
} fm_layer_weights;

/* Whole-policy parameters. `layers` is a HOST array of L entries whose fields
 * are device pointers; everything else is a device pointer.
 *   w_in bf16 [d][A], b_in fp32 [d]      : x = a . w_in^T + b_in
 *   w_out bf16 [A][d], b_out fp32 [A]    : v = h_f . w_out^T + b_out
 *   gamma_f fp32 [d]                     : h_f = AdaRMSNorm_f(x) * gamma_f
 *   w_mod_f bf16 [2d][d], b_mod_f [2d]   : [scale_f, shift_f] of the final norm
 *   conds fp32 [S][d] when cond_mode == FM_COND_GIVEN, else NULL. */
typedef struct fm_weights {
  const fm_layer_weights* layers;
  const uint16_t* w_in;
  const float* b_in;
  const uint16_t* w_out;
  const float* b_out;
  const float* gamma_f;
  const uint16_t* w_mod_f;
  const float* b_mod_f;
  const float* conds;
} fm_weights;

typedef struct fm_policy fm_policy;   /* opaque; owned by the library */

/* Human-readable name of a status code (static string). */
const char* fm_status_string(int status);

/* Detail of the last failure on this policy (or of the last policy-free call
 * on this thread when p is NULL). Valid until the next call. */
const char* fm_last_error(const fm_policy* p);

/* Bytes of device workspace a policy with this config needs (host call). */
int fm_workspace_size(const fm_config* cfg, size_t* bytes);

/* sizeof of the ABI structs as this library was compiled (fm_config, fm_weights,
 * fm_layer_weights, fm_timing), for bindings to check their mirrors. Any pointer may
 * be NULL. Never fails. */
int fm_abi_sizes(size_t* config, size_t* weights, size_t* layer_weights, size_t* timing);

/* Build a policy in a caller-owned workspace (device, 1024-byte aligned,
 * >= fm_workspace_size bytes). Folds gamma into the GEMM weights, computes each
 * weight's static scale (amax/448 for FP8; amax/(448*6) tensor scale plus E4M3
 * block scales for NVFP4), quantises and re-tiles the weights into
 * K-major 128-byte swizzled tiles, precomputes the per-step modulation table
 * (the t-schedule is fixed, so modulation is per-create state), copies the
 * in/out projections, stores the static activation scales (host [L][4] fp32,
 * [L][7] with FP8 attention, columns FM_SITE_*; ignored for BF16 activations and
 * may then be NULL) and,
 * with FM_FLAG_USE_GRAPH, captures the whole decision as one CUDA graph.
 * Synchronises `stream` before returning. The prefix cache starts zeroed.
 * On failure nothing is leaked and *out is NULL.
 * Source: blog post "Embodied inference acceleration", sections "CUDA Graph vs graph
 * simplification" (gamma fold, graph replay) and "Static quantisation" (static
 * scales); news article "FlashRT-PAI", section "It optimises the relay" (the plan
 * and its named persistent buffers). */
int policy_create(const fm_config* cfg, const fm_weights* w, const float* act_scales,
                  void* workspace, size_t ws_bytes, void* stream, fm_policy** out);

/* Release the host-side policy or session (graphs, plan). Does not touch the
 * workspace. The caller must not destroy a policy with work in flight on its
 * stream; a base policy with live sessions is not destroyed (FM_ERR_INVALID_ARG).
 * Source: news article "FlashRT-PAI", section "It optimises the relay". */
int policy_destroy(fm_policy* p);

/* Replace the static activation scales (host [L][4] fp32, [L][7] with FP8
 * attention). Stream-ordered copy into the policy's scale buffer; the captured
 * graph reads them from there. With FP8 attention the prefix cache's E4M3 copy
 * is re-derived with the new K and V scales. */
int fm_set_act_scales(fm_policy* p, const float* act_scales, void* stream);

/* Overwrite the whole prefix KV cache: k, v device bf16 [L][P][Hkv][Dh]. With
 * FP8 attention the cache's E4M3 copy (static K and V scales) is derived here.
 * Source: news article "FlashRT-PAI", section "It optimises the relay" (the prefix
 * state reused across decisions). */
int set_prefix_kv(fm_policy* p, const uint16_t* k, const uint16_t* v, void* stream);

/* Overwrite rows [tok_begin, tok_end) of every layer's prefix K and V (the
 * image-dependent part after a new observation); other rows persist.
 * k, v: device bf16 [L][tok_end - tok_begin][Hkv][Dh]. 0 <= begin < end <= P.
 * Source: news article "FlashRT-PAI", section "It optimises the relay" (selective
 * refresh of the image-dependent state). */
int refresh_prefix(fm_policy* p, int tok_begin, int tok_end, const uint16_t* k,
                   const uint16_t* v, void* stream);

/* One decision: S Euler steps from the noise (t = 1) to the action chunk (t = 0).
 * noise: device fp32 [M][A], or NULL to start from the policy's noise/action
 * buffer as it stands (e.g. after restore_state). actions: device fp32 [M][A]
 * (may equal noise). Asynchronous.
 * Source: blog post "Embodied inference acceleration", section "Static
 * quantisation" (18 layers x 10 denoise steps); news article "FlashRT-PAI", section
 * "It optimises the relay" (one graph, Programmatic Dependent Launch). */
int decode_actions(fm_policy* p, const float* noise, float* actions, void* stream);

/* Same as decode_actions with HOST buffers (pinned recommended): copies the
 * noise in, decodes, copies the actions out, then synchronises the stream. */
int decode_actions_host(fm_policy* p, const float* noise_host, float* actions_host, void* stream);

/* Decision noise on the device (no host noise input): element i of the [n]
 * fp32 output comes from Philox4x32-10 (Salmon et al., "Parallel random numbers:
 * as easy as 1, 2, 3", SC'11) block b = i / 4 with counter words
 * (b, 0, counter & 0xffffffff, counter >> 32) and key (seed & 0xffffffff,
 * seed >> 32); words (w0, w1) give elements 4b and 4b+1, (w2, w3) give 4b+2 and
 * 4b+3, by Box-Muller: u = (w + 1/2) / 2^32, z = sqrt(-2 ln u_a) * (cos, sin)
 * (2 pi u_b), evaluated in double and rounded to float. Distinct (seed, counter)
 * pairs give independent streams; the same pair gives the same noise.
 * out: device fp32 [n]; raw_words: NULL or device u32 [ceil(n/4)][4] receiving the
 * Philox words (for tests). Asynchronous. */
int fm_philox_noise(float* out, int64_t n, uint64_t seed, uint64_t counter, uint32_t* raw_words, void* stream);

/* decode_actions whose noise is fm_philox_noise(M * A, seed, counter), generated
 * on the device into the policy's noise/action buffer. actions: device fp32 [M][A].
 * Asynchronous. */
int fm_decode_actions_seeded(fm_policy* p, uint64_t seed, uint64_t counter, float* actions, void* stream);

/* One-step warm start (blog post, section "Few-step denoise brings the error back
 * into consecutive decisions"): the previous decision's chunk (the policy's
 * noise/action buffer) is moved forward by `executed` actions, its tail padded
 * with its last action, mixed with the new noise at flow time tau = cfg.warm_t,
 * a_tau = tau * noise + (1 - tau) * shifted, and one Euler step of dt = -tau with
 * the modulation at t = tau gives the actions. The previous chunk is kept from the
 * last decision of any kind; fm_episode_reset clears it, and a warm decode without
 * one runs the full S-step decision instead. noise: device fp32 [M][A];
 * 0 <= executed <= M; actions: device fp32 [M][A]. FM_ERR_UNSUPPORTED when
 * cfg.warm_t is 0. Asynchronous. */
int fm_decode_warm(fm_policy* p, const float* noise, int executed, float* actions, void* stream);

/* Start of an episode: the next fm_decode_warm runs the full decision. */
int fm_episode_reset(fm_policy* p);

/* Timestamps of the last decision (blog post, section on the observation age
 * A_k = t_apply,k - t_capture, measured with timestamps rather than summed stage
 * estimates). host_submit_ns: steady-clock time the decision was enqueued;
 * device_start_ns / device_end_ns: GPU globaltimer at the start of the decision's
 * first kernel and at the end of its last kernel, so T_infer = end - start (the two
 * clocks are not comparable with each other). Synchronises `stream`. */
typedef struct fm_timing {
  uint64_t host_submit_ns;
  uint64_t device_start_ns;
  uint64_t device_end_ns;
} fm_timing;
int fm_last_timing(fm_policy* p, fm_timing* t, void* stream);

/* Bytes of an execution-state capsule (header + prefix K/V + noise/action
 * buffer + activation scales + counters). */
int fm_state_size(const fm_policy* p, size_t* bytes);

/* Copy the policy's persistent state into dst (host if dst_on_device == 0, else
 * device), stream-ordered; host copies synchronise the stream.
 * Source: news article "FlashRT-PAI", section "It optimises the relay"
 * (execution-state capsules). */
int snapshot_state(fm_policy* p, void* dst, size_t bytes, int dst_on_device, void* stream);

/* Restore a capsule made by snapshot_state of THIS policy (same plan hash,
 * workspace address and shapes); otherwise FM_ERR_STATE_MISMATCH and nothing is
 * written. Capsules are in-process only, bound to the plan and device addresses.
 * Source: news article "FlashRT-PAI", section "It optimises the relay" (capsules
 * bound to the plan and device addresses). */
int restore_state(fm_policy* p, const void* src, size_t bytes, int src_on_device, void* stream);

/* Sessions (paper, "execution-state capsules" for snapshot, restore and fork of the
 * persistent state): several policies that share one plan and its read-only buffers
 * (packed weights, weight scales, modulation tables, in/out projections) while each
 * owns its state (prefix K/V cache and its E4M3 copy, activation scales,
 * noise/action buffer, activations, error word) in its own workspace.
 *
 * fm_session_workspace_size: bytes of a session's workspace (1024-aligned device
 * memory owned by the caller) for sessions of `base`.
 * fm_session_create: a new session of `base` (or of base's own base, if `base` is a
 * session) with an empty prefix cache, a zero action buffer and base's current
 * activation scales; it has its own CUDA graphs and runs independently of, and
 * concurrently with, the base and other sessions on other streams.
 * fm_session_fork: a session started from a capsule made by snapshot_state of
 * `base` or of any session of it: the one way a capsule moves to another workspace
 * (restore_state stays bound to the capsule's own workspace address).
 * policy_destroy of a base with live sessions fails with FM_ERR_INVALID_ARG and
 * destroys nothing: destroy the sessions first. */
int fm_session_workspace_size(const fm_policy* base, size_t* bytes);
int fm_session_create(fm_policy* base, void* workspace, size_t ws_bytes, void* stream, fm_policy** out);
int fm_session_fork(fm_policy* base, const void* capsule, size_t bytes, int capsule_on_device, void* workspace,
                    size_t ws_bytes, void* stream, fm_policy** out);

/* Synchronise `stream`, read and clear the device error word. Returns FM_OK, or
 * FM_ERR_DEVICE with *word = the bits a kernel set when it abandoned a bounded
 * wait (1 = TMA/MMA pipeline wait expired). */
int fm_device_status(fm_policy* p, void* stream, int* word);

/* Error word of the policy-free building blocks (fm_test_skinny_gemm, fm_gemm_consumer,
 * fm_gemm_consumer_noalloc): synchronise `stream`, read and clear the bits their kernels
 * set when they abandoned a bounded wait on the current device. Returns FM_OK, or
 * FM_ERR_DEVICE with *word = the bits (1 = TMA/MMA pipeline wait expired); the outputs of
 * the calls since the previous check are then not to be trusted. Those entry points are
 * asynchronous, so they cannot report this themselves. */
int fm_standalone_status(void* stream, int* word);

/* Address and size of one of the policy's named persistent buffers (the
 * execution contract's named buffers), for inspection and for zero-copy input:
 *   "prefix_k"              bf16 [L][P][Hkv][Dh]
 *   "prefix_v"              bf16 [L][Hkv][Dh][P_pad], P_pad = P rounded up to 8 (values
 *                           kept transposed: the layout attention's P.V operand reads)
 *   "actions"               fp32 [M][A] noise/action state
 *   "x"                     fp32 [M][d] residual stream
 *   "q", "q2"               codes [M][d] (pre-attention / pre-MLP GEMM operand)
 *   "attn_out"              codes [M][H*Dh]
 *   "geglu_out"             codes [M][F]
 *   "y_qkv"                 bf16 [M][(H+2Hkv)*Dh] dequantised Q | K | V (FP8 attention:
 *                           their E4M3 codes, one byte each, static scales FM_SITE_Q..V)
 *   "prefix_k8", "prefix_v8"  FP8 attention only: E4M3 copies of the prefix cache,
 *                           keys [L][P][Hkv][Dh], values transposed [L][Hkv][Dh][P16]
 *                           (P16 = P rounded up to 16)
 *   "y_o", "y_d"            fp32 [parts][M][N] GEMM partial planes
 *   "act_scales"            fp32 [L][8] (columns FM_SITE_*, column 7 unused)
 *   "weight_scales"         fp32 [L][4]
 *   "mod"                   fp32 [S][L][6][d]; "mod_final" fp32 [S][2][d]
 * Codes are one byte (FP8 activations), bf16 (BF16), or, with NVFP4 weights, the
 * E4M3 codes' f16 values (two bytes, exact: the operand format of the NVFP4 GEMM) or,
 * with NVFP4 activations, the f16 values e * bs of the four-bit codes (exact).
 * FM_ERR_INVALID_ARG for an unknown name. */
int fm_named_buffer(const fm_policy* p, const char* name, void** ptr, size_t* bytes);

/* Bytes of one decision trace (see fm_decode_trace). */
int fm_trace_size(const fm_policy* p, size_t* bytes);

/* Run one decision with the same kernels and launch configuration as
 * decode_actions, launched one by one (no graph), and record after the kernels
 * of every layer-step a copy of the buffers they wrote into `trace` (device,
 * >= fm_trace_size bytes), for stage-by-stage verification. Records are ordered
 * step-major then layer; each record holds, contiguously in this order:
 *   x_in fp32 [M][d]          residual stream entering the layer
 *   q codes [M][d]            pre-attention operand
 *   y_qkv bf16 [M][Nqkv]      dequantised Q | K | V (the QKV GEMM's output)
 *   attn_out codes [M][H*Dh]
 *   y_o fp32 [P1][M][d]       O partial planes (P1 = fm_named_buffer size / (M*d*4))
 *   x_mid fp32 [M][d]         after the attention gated residual
 *   q2 codes [M][d]
 *   geglu_out codes [M][F]    the gate|up GEMM's output (GeGLU applied in its epilogue)
 *   y_d fp32 [P3][M][d]
 *   x_out fp32 [M][d]         after the MLP gated residual; for the last layer of
 *                             a step that is not the last, the next step's x
 *                             (after the Euler update and input projection)
 *   actions fp32 [M][A]       the noise/action state after this layer-step
 * Codes are one byte (FP8), bf16 (BF16 activations), or f16 values with NVFP4 weights
 * (E4M3 code values, or e * bs with NVFP4 activations). Synchronous. */
int fm_decode_trace(fm_policy* p, const float* noise, float* actions, void* trace, size_t bytes, void* stream);

/* The warm start of fm_decode_warm (same arguments, launched one by one, no graph),
 * recording into `trace` (device, >= fm_warm_trace_size bytes) first the mixed input of
 * the single Euler step, a_tau = tau * noise + (1 - tau) * shifted as fp32 [M][A], then
 * one fm_decode_trace record per layer of that step (the last record's actions are the
 * decision's). Needs a previous chunk (FM_ERR_INVALID_ARG after fm_episode_reset or
 * before the first decision). Synchronous. */
int fm_warm_trace_size(const fm_policy* p, size_t* bytes);
int fm_decode_warm_trace(fm_policy* p, const float* noise, int executed, float* actions, void* trace,
                         size_t bytes, void* stream);

/* One decision (as decode_actions: the same kernels, launch configuration and graph)
 * whose kernels also record a timeline into `buf` (device, 16-byte aligned): u32
 * record count, u32 capacity, 56 bytes of padding, then one 128-byte record per CTA of
 * every kernel: u64 id = kind (1 skinny GEMM, 2 attention, 3 row kernel, 4 NVFP4 GEMM)
 * | gridDim.x << 8 | grid rows << 20 | blockIdx.x << 32 | block row << 44 | SM << 56,
 * then fifteen u64 %globaltimer stamps in ns (0 = not recorded): GEMM - entry, after
 * the programmatic-dependent-launch wait, MMAs complete, partial rows pushed, split-K
 * rows received, outputs written, exit; attention - entry, after the wait, operands
 * loaded, chunk values transposed, S = Q K^T complete, pass 1 done, cluster peers
 * started, statistics sent, statistics received, P written, O = P V complete, O band
 * copies issued, O band received, band stored, exit; row kernel - entry, after the
 * wait, exit. Records past the capacity (bytes - 64) / 128 are dropped. Runs the
 * decision twice (the first warms the new graph up) and synchronises; a diagnostic,
 * not the timed path. */
int fm_decode_timeline(fm_policy* p, const float* noise, float* actions, void* buf, size_t bytes, void* stream);

/* Kernel launches per decoder layer and per decision of the captured plan. */
int fm_test_kernel_count(const fm_policy* p, int* per_layer, int* per_decision);

/* The attention plan of the policy: keys per slice (one CTA's share of the P + M keys;
 * 64, 128, 192, or 256 for the wide slice) and slices (the cluster size). */
int fm_test_attn_plan(const fm_policy* p, int* keys_per_slice, int* slices);

/* Launch only kernel `index` (0 .. per_layer - 1, in the decision's order: FP8/BF16
 * QKV GEMM, attention, O GEMM, consumer, gate|up GEMM + GeGLU, down GEMM, consumer or
 * step boundary) of layer `layer` at Euler step `step`, with exactly the arguments and
 * launch configuration the decision uses (Programmatic Dependent Launch when the
 * policy's flags hold FM_FLAG_USE_PDL, as in the decision), on the policy's current
 * buffers: for timing one kernel on its own or back to back (the buffers hold the last
 * decision's data). It updates the policy's state as that kernel does. Asynchronous. */
int fm_test_launch_kernel(fm_policy* p, int layer, int step, int index, void* stream);

/* Hand-off diagnostics (no counterpart in the pages: they measure the kernel
 * boundaries the decision is made of). Both are synchronous.
 *
 * fm_test_pdl_chain: a CUDA graph of `kernels` (1..4096) dependent launches of a
 * nearly empty kernel of `ctas` x `threads` (threads a multiple of 32, <= 1024) in
 * thread-block clusters of `cluster` CTAs (1, 2, 4 or 8; dividing ctas), each
 * launched with programmatic dependent launch when pdl != 0 (it signals its
 * dependents at entry, then waits for its predecessor), else in plain stream order;
 * after the wait every thread stores `writes` (0..64) 4-byte words. The graph is run
 * once, then `reps` (1..1000) times between two events; *us_per_kernel = elapsed /
 * (reps * kernels). scratch: device, scratch_bytes >= 4 * (1 + ctas * threads *
 * writes) (a counter the kernels update, then the stored words). The graph, its
 * stream and events are created and destroyed inside the call. Errors:
 * FM_ERR_INVALID_ARG (NULL), FM_ERR_SHAPE (a count out of range), FM_ERR_WORKSPACE
 * (scratch too small), FM_ERR_CUDA.
 *
 * fm_test_grid_barrier: one cooperative launch of `ctas` x `threads` that runs
 * `rounds` (1..10^6) grid-wide barriers on an arrive counter in global memory.
 * mode 0: each CTA arrives by a release reduction and polls with acquire loads (gpu
 * scope); mode 1: a full fence, a relaxed atomic add, volatile polls, a full fence
 * after; mode 2: as 0 but CTA 0 never arrives, so every wait runs out (the failure
 * path). Each wait is bounded by budget_ns (1 us .. 10 s); one that runs out sets an
 * error word that releases every other waiter. scratch: device, 16-byte aligned,
 * >= 8 bytes (counter and error word, zeroed by the call). out: device u64
 * [ctas][2]: CTA b's time over its completed rounds (ns) and that round count.
 * Errors: FM_ERR_INVALID_ARG, FM_ERR_SHAPE (also when the CTAs cannot all be resident
 * at once), FM_ERR_ALIGN, FM_ERR_UNSUPPORTED (no cooperative launch), FM_ERR_CUDA,
 * FM_ERR_DEVICE (a barrier wait ran out: always so in mode 2). */
int fm_test_pdl_chain(int ctas, int threads, int kernels, int reps, int pdl, int cluster, int writes, void* scratch,
                      size_t scratch_bytes, float* us_per_kernel);
int fm_test_grid_barrier(int ctas, int threads, int rounds, int mode, unsigned long long budget_ns, void* scratch,
                         unsigned long long* out, void* stream);

/* ---------------------------------------------------------------------------
 * Building blocks, exported for tests and standalone use (same conventions).
 * ------------------------------------------------------------------------- */

/* Static-scale E4M3 quantisation: codes[i] = E4M3_RNE_satfinite(x[i] * (1/scale)),
 * the reciprocal rounded to fp32. x device fp32 [n], codes device uint8 [n]. */
int fm_test_quant_e4m3(const float* x, int64_t n, float scale, uint8_t* codes, void* stream);

/* Bytes of a packed weight [N][K] in format fmt (N, K multiples of 128). */
int fm_packed_weight_bytes(int N, int K, int fmt, size_t* bytes);

/* Fold gamma (device fp32 [K] or NULL), quantise and tile a weight w (device fp32
 * [N][K]) into `packed` (device, 1024-byte aligned, fm_packed_weight_bytes).
 * scale_out (device fp32 [1]) receives the tensor scale (1.0 for BF16).
 * NVFP4 (news article "FlashRT-PAI", 4-bit weights): ts = fp32(amax) / 2688;
 * per 16 consecutive K elements bs = E4M3(amax_block / fp32(6 ts)); elements
 * e = E2M1_RNE(w' / fp32(bs ts)) (0 where bs ts == 0), w' = fp32(w gamma); all
 * divisions fp32 round-to-nearest. Layout: blocks (n/128, k/64) of 4608 bytes,
 * n-tile-major then k-block, each [128 rows][32 bytes] of codes (element 2i in
 * the low nibble) followed by [128 rows][4] block-scale codes.
 * FP8 tile layout: tile (n/128, k/128) is 128 rows x 128 bytes, rows n, bytes k,
 * tiles ordered n-tile-major then k-block; each tile is [128 rows][128 bytes]
 * (BF16: [128][64] elements) with the 128-byte swizzle applied: the 16-byte
 * chunk c of row r is stored at chunk position c ^ (r mod 8), the layout the
 * tensor cores read, so one bulk copy moves consecutive tiles into place. */
int fm_pack_weight(const float* w, const float* gamma, int N, int K, int fmt,
                   void* packed, float* scale_out, void* stream);

/* Skinny GEMM with K-split on tcgen05 tensor cores (blog post, "Small-M GEMM"):
 * partials[j][m][n] = sum_{k in slice j} A[m][k] * Wcodes[n][k] for the s equal
 * contiguous K slices (fp32, unscaled). A: device [M][K], fp8 codes (fmt FP8)
 * or bf16 (fmt BF16), 16-byte aligned; w_packed from fm_pack_weight.
 * cluster_reduce = c (1, 2, 4 or 8, dividing s): the c CTAs of consecutive
 * slices sum their partials in fixed order through distributed shared memory,
 * so partials holds s/c slices [s/c][M][N]. 1 <= M <= 256; N, K multiples of
 * 128; s divides K/128 (FP8) or K/64 (BF16). fmt NVFP4: A holds the f16
 * values of E4M3 codes [M][K], w_packed NVFP4 from fm_pack_weight, the partials
 * are sum A * (e * bs) without ts, s divides K/64 and cluster_reduce is 1. */
int fm_test_skinny_gemm(const void* a, int M, int K, const void* w_packed, int N, int fmt,
                        int s, int cluster_reduce, float* partials, void* stream);

/* fm_test_skinny_gemm with the weight rows per CTA (the MMA's M) chosen: tile_rows 128,
 * or 64 (each CTA takes one half of a packed 128-row tile; FP8 and BF16 only). The
 * partials are the same sums. */
int fm_test_skinny_gemm_tile(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s,
                             int cluster_reduce, int tile_rows, float* partials, void* stream);

/* Bytes of scratch fm_gemm_consumer needs for its fp32 split-K partial planes. */
int fm_gemm_consumer_scratch_bytes(int M, int N, int K, int fmt, int s, size_t* bytes);

/* Skinny GEMM + fused consumer in one call (blog post, "Small-M GEMM": K-split
 * with FP32 partials reduced by the consumer, which applies its own transform;
 * section "Static quantisation": bias + gated residual + AdaRMSNorm + static
 * quantise): y = (A Wcodes^T) * fp32(s_a * s_w) + bias, x <- x + gate * y,
 * q = Q(AdaRMSNorm(x; scale, shift), s_q). The s K-slices' partials go through
 * `scratch` (device, 16-byte aligned, >= fm_gemm_consumer_scratch_bytes; its
 * contents on entry do not matter). A, w_packed, fmt and s as in
 * fm_test_skinny_gemm (N <= 16384); bias (may be NULL), gate, scale, shift
 * device fp32 [N]; x device fp32 [M][N] in/out; s_a, s_w, s_q device fp32 [1];
 * q device [M][N] codes (E4M3 bytes for FP8, bf16 for BF16). */
int fm_gemm_consumer(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s, const float* s_a,
                     const float* s_w, const float* bias, float* x, const float* gate, const float* scale,
                     const float* shift, float eps, const float* s_q, void* q, void* scratch, size_t scratch_bytes,
                     void* stream);

/* fm_gemm_consumer for callers that cannot allocate device memory (no
 * counterpart in the paper). Same arguments and results, minus the scratch
 * buffer: the split-K partials go to an 8 MiB array built into the library's
 * device image, so this call allocates nothing. Shapes whose partials need more
 * (s/cluster x M x N x 4 bytes > 8 MiB) return FM_ERR_WORKSPACE. The first call
 * on each device looks the array's address up (make it before any stream
 * capture); every GPU that loads the library keeps the array until exit; calls
 * that overlap on the GPU share the array and race. */
int fm_gemm_consumer_noalloc(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s,
                             const float* s_a, const float* s_w, const float* bias, float* x, const float* gate,
                             const float* scale, const float* shift, float eps, const float* s_q, void* q,
                             void* stream);

/* Fused consumer (blog post, "Static quantisation"): with y = (sum_j
 * partials[j]) * fp32(s_a * s_w) + bias,  x <- x + gate * y,
 * q = Q(AdaRMSNorm(x; scale, shift), s_q) where Q is E4M3 with the fp32
 * reciprocal of s_q (act_fmt FP8) or bf16 rounding (BF16). partials device fp32
 * [nparts][M][N]; bias/gate/scale/shift device fp32 [N] (bias may be NULL);
 * x device fp32 [M][N] in/out; s_a, s_w, s_q device fp32 [1]; q device [M][N]. */
int fm_test_consumer(const float* partials, int nparts, int M, int N, const float* s_a,
                     const float* s_w, const float* bias, float* x, const float* gate,
                     const float* scale, const float* shift, float eps, const float* s_q,
                     void* q, int act_fmt, void* stream);

/* One decoder layer of a policy on a given residual input, launched exactly as
 * decode_actions launches it: q = Q(AdaRMSNorm_l(x_in)), the layer, then the
 * next layer's ((layer+1) mod L) pre-attention norm + quantise.
 * x_in, x_out device fp32 [M][d]; q_out device [M][d] codes (fp8 or bf16). */
int fm_test_layer(fm_policy* p, const float* x_in, int layer, int step, float* x_out,
                  void* q_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FMAD_H */
