/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) qwen3moe Mixture-of-Experts FFN over
 * GGUF k-quant expert weights.
 *
 * The operation (aprender issue "qwen3moe (Qwen3-30B-A3B, Qwen3-Coder-30B-A3B,
 * Q4_K_M) has NO working CUDA path", sections "File facts" and "Gaps ... G3"):
 *
 *   logits = Wr x (+ bias)                        F32 router GEMV [E x H]
 *   S, w   = top-k(softmax(logits)), renormalised  ("softmax, top-8, renorm")
 *   for each selected expert e (addressed in place as base + e * stride):
 *     g = Wg_e x, u = Wu_e x                      Q4_K gate / up dequant-GEMV
 *     a = silu(g) * u                             fused SwiGLU
 *     y_e = Wd_e a                                Q6_K or Q4_K down dequant-GEMV
 *   out = residual + sum_j w_j y_{S_j}            weighted sum into the residual
 *
 * qmoe_forward_q8k runs the same layer with x and a quantised to 8-bit (Q8_K)
 * activations before every expert GEMV (the int8 variant of "Gaps ... G8").
 * qmoe_forward_fp8 and qmoe_forward_nvfp4 run it over FP8 block-scaled and
 * NVFP4 experts instead of k-quants (qmoe_nvfp4_quantize makes NVFP4 weights
 * from BF16 ones).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer that the caller allocated and owns
 *    (except qmoe_forward_host, whose activations are host pointers).  The
 *    library never copies, repacks or frees caller memory.
 *  - Quantised tensors are raw GGUF superblocks: Q4_K = 144 B per 256 weights
 *    (fp16 d, fp16 dmin, 12 B packed 6-bit scales/mins, 128 B nibbles); Q6_K =
 *    210 B per 256 weights (128 B ql, 64 B qh, 16 int8 scales, fp16 d).  A
 *    matrix with R outputs and C inputs is R rows of C/256 consecutive
 *    superblocks; expert e of a 3-D expert tensor starts at
 *    base + e * R * (C/256) * block_bytes.
 *  - F32 activations are row-major [n_tokens][hidden].
 *  - Work is enqueued asynchronously on the context's stream; no call below
 *    synchronises the host, allocates memory or copies weights, except
 *    qmoe_create / qmoe_destroy (allocate / free the workspace),
 *    qmoe_forward_host (copies activations and synchronises) and
 *    qmoe_get_status (synchronises).
 *  - Errors are returned as qmoe_status; no exception crosses the ABI.
 *    Argument errors are detected on the host before anything is enqueued.
 *    qmoe_last_error() gives a one-line description of the last failure.
 *  - A context is not thread-safe: one host thread at a time, and calls that
 *    share a context must be ordered on its stream (they share the workspace).
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_INVALID_ARG = 1,       /* null pointer, bad size or count */
    QMOE_ERR_MISALIGNED = 2,        /* a base pointer is not 16-byte aligned */
    QMOE_ERR_UNSUPPORTED_QTYPE = 3, /* qtype not allowed for that tensor */
    QMOE_ERR_SHAPE = 4,             /* hidden/ffn not a multiple of 256, n_tokens > max */
    QMOE_ERR_NO_MEMORY = 5,         /* workspace does not fit; message names the bytes */
    QMOE_ERR_CUDA = 6,              /* a CUDA runtime call failed; message names it */
    QMOE_ERR_TIMEOUT = 7,           /* a bounded device-side wait gave up */
    QMOE_ERR_DEVICE_CHECK = 8       /* a device-side index check failed */
} qmoe_status;

typedef enum { QMOE_Q4_K = 1, QMOE_Q6_K = 2 } qmoe_qtype;

typedef struct qmoe_ctx qmoe_ctx;

/* Geometry fixed at create time.  The MoE part (hidden, n_experts, top_k, ffn)
 * is required; the attention part is needed only by qmoe_decode_step and may
 * be all zero otherwise (Qwen3-30B-A3B: 32 q heads, 4 kv heads, head_dim 128,
 * rope base 1e7, RMSNorm eps 1e-6; head_dim is NOT hidden / n_heads -- aprender
 * issue "Qwen3 GPU inference produces garbage output", "Fix Applied"). */
typedef struct {
    int hidden;          /* H, multiple of 256 */
    int n_experts;       /* E, 1..1024 */
    int top_k;           /* k, 1..min(E, 16) */
    int ffn;             /* F, expert FFN width, multiple of 256 */
    int norm_topk_prob;  /* 1: renormalise the k selected probabilities (qwen3moe) */
    int max_tokens;      /* largest n_tokens any call will pass (workspace size) */
    int n_heads;         /* attention q heads (decode step only, else 0) */
    int n_kv_heads;      /* attention kv heads, divides n_heads */
    int head_dim;        /* 128 for qwen3moe (a multiple of 64, <= 256) */
    int max_ctx;         /* KV-cache positions per layer, 1..262144 */
    float rope_base;     /* NEOX RoPE base */
    float rms_eps;       /* RMSNorm epsilon (all four norms) */
    void* stream;        /* cudaStream_t the work is enqueued on (NULL = legacy default) */
} qmoe_config;

/* Create a context on the current CUDA device and allocate its workspace
 * (router logits, expert ids / weights, per-expert pair lists, intermediate
 * activations, all sized by max_tokens).  Returns QMOE_ERR_NO_MEMORY with a
 * message giving the bytes needed and free, instead of failing later.
 * On success *out owns the workspace until qmoe_destroy. */
qmoe_status qmoe_create(const qmoe_config* cfg, qmoe_ctx** out);

/* Free the workspace (synchronises the context's stream first).  NULL is a no-op. */
void qmoe_destroy(qmoe_ctx* ctx);

/* Change the stream later calls enqueue on. */
qmoe_status qmoe_set_stream(qmoe_ctx* ctx, void* stream);

/* hidden_out = hidden_in + MoE(hidden_in) for n_tokens tokens.
 *  hidden_in, hidden_out : F32 [n_tokens][H] (device).  They may alias only
 *                          when n_tokens <= 8 (decode); otherwise -> INVALID_ARG.
 *  router_w              : F32 [E][H] (device), the ffn_gate_inp tensor.
 *  gate_exps, up_exps    : [E][F rows][H/256 superblocks], Q4_K (or Q6_K).
 *  down_exps             : [E][H rows][F/256 superblocks], Q6_K or Q4_K.
 *  All base pointers 16-byte aligned.  n_tokens in 1..max_tokens.
 * Expert ids are selected on the F32 logits, ties to the lower index. */
qmoe_status qmoe_forward(qmoe_ctx* ctx, const float* hidden_in, const float* router_w,
                         const void* gate_exps, const void* up_exps, const void* down_exps,
                         qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t,
                         int n_tokens, float* hidden_out);

/* General form:  out = residual + MoE(ffn_in), router logits += router_bias.
 *  residual     : F32 [n_tokens][H] or NULL (then residual = ffn_in).
 *  router_bias  : F32 [E] or NULL.
 *  ids_out      : int32 [n_tokens][k] or NULL -- selected experts, ordered by
 *                 descending logit (ties: lower index first).
 *  weights_out  : F32 [n_tokens][k] or NULL -- their routing weights.
 * out may alias residual (not ffn_in) when n_tokens <= 8. */
qmoe_status qmoe_forward_ex(qmoe_ctx* ctx, const float* ffn_in, const float* residual,
                            const float* router_bias, const float* router_w,
                            const void* gate_exps, const void* up_exps, const void* down_exps,
                            qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t,
                            int n_tokens, float* out, int32_t* ids_out, float* weights_out);

/* The same layer with 8-bit activations in every expert GEMV: the int8 (DP4A)
 * variant of the aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working
 * CUDA path" ("Gaps ... G8"; its R1 receipt measures it against FP32
 * activations).  hidden_out = hidden_in + MoE(hidden_in) where x (per token)
 * and the SwiGLU output (per selected expert) are first quantised to Q8_K
 * blocks of 256 values: fp32 scale d, int8 codes, the block's largest-magnitude
 * value (first on a tie) on code -128 (s = -128/v, q = min(127, rint(s*x)),
 * d = 1/s, fp32), and each weight row is dotted with the codes in integer form.
 * The router stays F32.  Arguments as qmoe_forward; ids_out / weights_out as
 * qmoe_forward_ex (nullable).  hidden_out may alias hidden_in.  Any n_tokens in
 * 1..max_tokens; hidden and ffn multiples of 256 (as for every entry point).
 * Argument errors are returned before any launch, as for qmoe_forward. */
qmoe_status qmoe_forward_q8k(qmoe_ctx* ctx, const float* hidden_in, const float* router_w,
                             const void* gate_exps, const void* up_exps, const void* down_exps,
                             qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t,
                             int n_tokens, float* hidden_out, int32_t* ids_out, float* weights_out);

/* The MoE layer over FP8 block-scaled experts with the F32 router (atlasinference
 * source page "spark_model/weight_loader/qwen3.rs", load_layers: experts kept as
 * FP8 with one scale per 128 x 128 block, FP8 weights against wider
 * activations, and the option of a full-precision router so that expert
 * selection is not decided by quantised logits).
 *   gate_exps / up_exps: E4M3 ("e4m3fn") codes [E][ffn][hidden], one byte each;
 *   down_exps: codes [E][hidden][ffn];
 *   gate_scale / up_scale: fp32 [E][ffn/128][hidden/128];
 *   down_scale: fp32 [E][hidden/128][ffn/128];
 *   weight (r, c) of expert e = e4m3(code) * scale[e][r/128][c/128].
 * Codes 0x7F / 0xFF (NaN) are not valid weights.  Up to 32 tokens the expert
 * GEMVs run on the CUDA cores with x, the SwiGLU output and every sum in fp32;
 * more tokens run as grouped GEMMs on the tensor cores (weights widened to fp16
 * as e4m3 * scale rounded once, x and the SwiGLU output rounded to fp16, fp32
 * accumulation), like the k-quant path of qmoe_forward.  hidden_out = hidden_in + MoE(hidden_in); it may alias
 * hidden_in for any n_tokens.  ids_out / weights_out as qmoe_forward_ex
 * (nullable).  Serves hidden/256 in {2, 4, 8, 16} and ffn/256 in 1..6
 * (QMOE_ERR_SHAPE otherwise).  Code and activation pointers 16-byte aligned,
 * scale pointers 4-byte aligned (QMOE_ERR_MISALIGNED).  Argument errors are
 * returned before any launch. */
qmoe_status qmoe_forward_fp8(qmoe_ctx* ctx, const float* hidden_in, const float* router_w,
                             const void* gate_exps, const float* gate_scale,
                             const void* up_exps, const float* up_scale,
                             const void* down_exps, const float* down_scale,
                             int n_tokens, float* hidden_out, int32_t* ids_out,
                             float* weights_out);

/* The MoE layer over NVFP4 experts with the F32 router (atlasinference source
 * page "spark_model/weight_loader/qwen3.rs", load_layers: weights quantised
 * from BF16 to NVFP4 at load).  NVFP4 (the public format): FP4 E2M1 elements,
 * two per byte with the even element in the low nibble, one E4M3 scale per 16
 * consecutive elements of a row, one fp32 scale per matrix:
 *   weight (r, c) of expert e = e2m1(code) * e4m3(bscale[e][r][c/16]) * global[e].
 *   gate_exps / up_exps: codes [E][ffn][hidden/2]; *_bscale [E][ffn][hidden/16];
 *   down_exps: codes [E][hidden][ffn/2]; down_bscale [E][hidden][ffn/16];
 *   *_global: fp32 [E].
 * Up to 32 tokens (and whenever a block-scale pointer is not 16-byte aligned)
 * the expert GEMVs run on the CUDA cores with x, the SwiGLU output and every
 * sum in fp32; more tokens run as grouped GEMMs on the tensor cores (weights
 * widened to fp16 as e2m1 * e4m3 * global rounded once, x and the SwiGLU
 * output rounded to fp16, fp32 accumulation).  hidden_out = hidden_in + MoE(hidden_in) and may alias
 * hidden_in.  ids_out / weights_out as qmoe_forward_ex (nullable).  Serves
 * hidden/512 in {1, 2, 4, 8} and ffn/256 in 1..6 (QMOE_ERR_SHAPE otherwise).
 * Code and activation pointers 16-byte aligned, block scales 2-byte, globals
 * 4-byte (QMOE_ERR_MISALIGNED).  Argument errors are returned before any launch. */
qmoe_status qmoe_forward_nvfp4(qmoe_ctx* ctx, const float* hidden_in, const float* router_w,
                               const void* gate_exps, const void* gate_bscale,
                               const float* gate_global, const void* up_exps,
                               const void* up_bscale, const float* up_global,
                               const void* down_exps, const void* down_bscale,
                               const float* down_global, int n_tokens, float* hidden_out,
                               int32_t* ids_out, float* weights_out);

/* Runtime quantisation of n_mats consecutive BF16 matrices [rows][cols] (device
 * memory, bit patterns) to NVFP4 (same page: a global-absmax pass, then the
 * per-block quantisation).  Per matrix, every decision in fp32:
 *   amax = max |x|; global = amax / 2688 (448 * 6);
 *   per 16 elements: s = E4M3 nearest to bmax / (6 * global) (ties to even,
 *   saturating at 448); d = e4m3(s) * global; code = E2M1 nearest to x / d
 *   (ties to even, saturating at 6; 0 where d = 0).
 * Outputs (device, caller-owned): codes [n_mats][rows][cols/2] (8-byte
 * aligned), bscale [n_mats][rows][cols/16], global [n_mats] (4-byte aligned).
 * x 16-byte aligned; cols a positive multiple of 16; n_mats in 1..1024.
 * Enqueued on the context's stream; uses a few bytes of its workspace, so it is
 * ordered with the context's other calls. */
qmoe_status qmoe_nvfp4_quantize(qmoe_ctx* ctx, const void* x_bf16, int n_mats, int rows, int cols,
                                void* codes, void* bscale, float* global);

/* Same as qmoe_forward, but hidden_in / hidden_out are HOST pointers (pinned
 * memory gives asynchronous copies).  Copies the activations to the device
 * workspace, runs the layer, copies the result back and synchronises the
 * stream before returning.  Weights stay device pointers. */
qmoe_status qmoe_forward_host(qmoe_ctx* ctx, const float* hidden_in_host, const float* router_w,
                              const void* gate_exps, const void* up_exps, const void* down_exps,
                              qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t,
                              int n_tokens, float* hidden_out_host);

/* Weights of one qwen3moe decoder layer (all device pointers). */
typedef struct {
    const float* attn_norm;  /* [H] input RMSNorm weight */
    const void* wq;          /* [n_heads*head_dim rows][H], Q4_K */
    const void* wk;          /* [n_kv*head_dim rows][H], Q4_K */
    const void* wv;          /* [n_kv*head_dim rows][H], Q4_K */
    const void* wo;          /* [H rows][n_heads*head_dim], Q4_K */
    const float* q_norm;     /* [head_dim] per-head Q RMSNorm weight */
    const float* k_norm;     /* [head_dim] per-head K RMSNorm weight */
    const float* ffn_norm;   /* [H] post-attention RMSNorm weight */
    const float* router_w;   /* [E][H] F32 */
    const void* gate_exps;   /* MoE experts as in qmoe_forward */
    const void* up_exps;
    const void* down_exps;
    qmoe_qtype down_t;       /* Q6_K or Q4_K (per layer) */
    void* k_cache;           /* fp16 [n_kv][max_ctx][head_dim]; slot pos is written */
    void* v_cache;           /* fp16 [n_kv][max_ctx][head_dim]; slot pos is written */
} qmoe_layer_weights;

/* One batch-1 decode step through n_layers qwen3moe decoder layers, in place on
 * hidden (F32 [H], device).  Per layer: x = RMSNorm(h)*attn_norm; q,k,v = Wq/Wk/Wv x;
 * per-head RMSNorm of q and k (q_norm, k_norm), then NEOX RoPE at position pos
 * (pairs (i, i + head_dim/2)); k, v rounded to fp16 into cache slot pos; GQA
 * attention of q head h over kv head h / (n_heads/n_kv_heads), positions
 * 0..pos, scale 1/sqrt(head_dim); h += Wo attn; h += MoE(RMSNorm(h)*ffn_norm).
 * Sources: aprender issue "Qwen3 GPU inference produces garbage output" (Fix
 * Applied), aprender PR "apply per-head Q/K RMSNorm in forward_qwen3_moe" (The
 * fix), SharpInference issue "Forward-pass divergence on Qwen3-Coder 30B-A3B"
 * (NEOX RoPE).  ids_out (nullable): int32 [n_layers][k] selected experts.
 * Requires the attention geometry in the config; 0 <= pos < max_ctx. */
qmoe_status qmoe_decode_step(qmoe_ctx* ctx, const qmoe_layer_weights* layers, int n_layers,
                             int pos, float* hidden, int32_t* ids_out);

/* Batched prefill: n_tokens tokens at positions pos0 .. pos0+n_tokens-1 through
 * n_layers qwen3moe decoder layers, in place on hidden (F32 [n_tokens][H],
 * device, 16-byte aligned).  Per layer it computes, for every token t, what
 * qmoe_decode_step computes for one token at position pos0 + t, with causal
 * attention: token t attends to the cache positions 0 .. pos0-1 as stored and
 * to the batch's tokens 0 .. t.  Within a layer a token's K and V depend only
 * on its own input, so this equals n_tokens decode steps in order (the
 * token-by-token prefill of the aprender issue "qwen3moe ... has NO working
 * CUDA path", later gap list, "Prefill is token-by-token", which names the
 * batched form as the fix).  Differences from the decode step: the Q/K/V and O
 * projections run as tensor-core GEMMs on fp16 rows of the normalised input and
 * of the attention output (fp32 accumulation), and for n_tokens > 8 the MoE is
 * the tensor-core grouped-GEMM path of qmoe_forward_ex (fp16 operands).
 *  layers   : n_layers qmoe_layer_weights, as for qmoe_decode_step; the cache
 *             slots pos0 .. pos0+n_tokens-1 of every layer are written (fp16),
 *             the other slots are only read.
 *  ids_out  : nullable, int32 [n_layers][n_tokens][k] selected experts.
 * Requires the attention geometry in the config with at most 8 q heads per kv
 * head and n_heads*head_dim, n_kv_heads*head_dim multiples of 128; otherwise
 * QMOE_ERR_SHAPE.  1 <= n_tokens <= max_tokens, 0 <= pos0, pos0 + n_tokens <=
 * max_ctx (else QMOE_ERR_SHAPE).  The context holds a scratch of
 * about 56 KiB per max_tokens token at the Qwen3-30B-A3B shape for this call. */
qmoe_status qmoe_prefill(qmoe_ctx* ctx, const qmoe_layer_weights* layers, int n_layers,
                         int n_tokens, int pos0, float* hidden, int32_t* ids_out);

/* Allocation-free variant of qmoe_forward for decode-sized calls.  The pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory: processes whose device memory is owned by their own
 * pool (a host framework's allocator, a plugin inside such a process), or
 * latency-critical loops that must not run a cudaMalloc, with its implicit
 * device synchronisation, after start-up.  It needs no context and allocates
 * nothing: its scratch (the tagged router logits, SwiGLU activations and down
 * outputs that the fused decode kernel passes between its CTAs, the "x staged"
 * marks, two control words and a status word) is one fixed device array inside
 * the library of 2 MiB + 256 B, which every GPU that loads the library holds
 * until the process exits.
 *  - Computes the same as qmoe_forward (hidden_out = hidden_in + MoE(hidden_in))
 *    with the same argument meaning, layout and alignment rules, on `stream`
 *    (a cudaStream_t; NULL = legacy default stream).
 *  - Served shapes: those of the fused single-kernel decode path (n_tokens
 *    <= 8, gate/up Q4_K, hidden in {256, 2048}, ffn in {256, 768}; see
 *    qmoe_fused_decode_available) whose buffers fit the array:
 *    8 * (n_tokens*n_experts + n_tokens*top_k*(ffn + hidden) + number of SMs)
 *    + 4 * top_k*ffn, each of the five parts rounded up to 256 B, at most 2 MiB.  At the
 *    Qwen3-30B-A3B shape that is every n_tokens <= 8 at top_k 8.  Anything
 *    else returns QMOE_ERR_SHAPE and enqueues nothing.
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress) and sets the kernel's shared-memory limit; make that
 *    first call before any stream capture.
 *  - All calls share the one scratch array and it keeps the last call's
 *    contents.  Its control words carry over from call to call (they count
 *    launches, so values left by an earlier call are never mistaken for this
 *    call's); the status word is cleared at the start of every call.  Calls
 *    whose execution overlaps on the GPU (other streams, other host threads)
 *    race on it and give wrong results: order them.
 *  - Returns launch / argument errors only; the device-side status of the call
 *    (a bounded wait that ran out) is read with qmoe_noalloc_status. */
qmoe_status qmoe_forward_noalloc(const float* hidden_in, const float* router_w,
                                 const void* gate_exps, const void* up_exps,
                                 const void* down_exps, qmoe_qtype gate_t, qmoe_qtype up_t,
                                 qmoe_qtype down_t, int hidden, int n_experts, int top_k,
                                 int ffn, int norm_topk_prob, int n_tokens, float* hidden_out,
                                 void* stream);

/* Device-side status of the last qmoe_forward_noalloc call on the current
 * device: synchronises `stream` (the stream that call used), reads the status
 * word of the shared scratch and clears it.  QMOE_OK, or QMOE_ERR_TIMEOUT /
 * QMOE_ERR_DEVICE_CHECK as for qmoe_get_status; QMOE_ERR_CUDA if the device
 * was never set up by a call. */
qmoe_status qmoe_noalloc_status(void* stream);

/* Synchronise the stream and read the device status word (bounded-wait
 * timeouts, device index checks).  A non-OK status is sticky until read:
 * reading it clears it. */
qmoe_status qmoe_get_status(qmoe_ctx* ctx);

/* One-line description of the last error on this context ("" if none).  The
 * string is owned by the context and valid until the next call on it.  With
 * ctx = NULL: why the last qmoe_create on this thread failed (for
 * QMOE_ERR_NO_MEMORY the bytes the workspace needs and the bytes free). */
const char* qmoe_last_error(qmoe_ctx* ctx);

/* Test hooks of the failure paths (no counterpart on the pages).
 * qmoe_debug_stall_next: the next fused decode launch on this context (a
 *   qmoe_forward / qmoe_forward_ex of n_tokens <= 8 at a fused shape) waits for
 *   router logits carrying a launch tag that no CTA writes, gives up after
 *   wait_ns, records QMOE_ERR_TIMEOUT in the status word and exits without
 *   computing (its outputs are left unwritten).  Later launches are normal:
 *   this is how a test shows that a timed-out launch leaves the context usable.
 * qmoe_debug_fail_alloc: the next n workspace allocations of qmoe_create, in
 *   any thread, fail as if the device were out of memory (QMOE_ERR_NO_MEMORY). */
qmoe_status qmoe_debug_stall_next(qmoe_ctx* ctx, uint64_t wait_ns);
void qmoe_debug_fail_alloc(int n);

/* Bytes of workspace a context with this config allocates (0 on bad config). */
size_t qmoe_workspace_bytes(const qmoe_config* cfg);

/* 1 when qmoe_forward / qmoe_forward_ex on this context would run a layer of
 * n_tokens tokens with these expert qtypes as the single fused decode kernel
 * (one launch: router, top-k, gate/up, SwiGLU, down and combine), 0 when it
 * would take the multi-kernel path (tensor-core prefill or the SIMT path).
 * Pure host query; no device work. */
int qmoe_fused_decode_available(const qmoe_ctx* ctx, int n_tokens, qmoe_qtype gate_t,
                                qmoe_qtype up_t, qmoe_qtype down_t);

/* Byte stride between consecutive experts of a 3-D expert tensor whose
 * matrices have `rows` outputs and `cols` inputs (0 on bad arguments). */
size_t qmoe_expert_stride(qmoe_qtype qtype, int rows, int cols);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H */
