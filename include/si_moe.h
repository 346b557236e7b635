/*
 * si_moe.h -- C ABI of libsimoe: a Q4_K-resident mixture-of-experts FFN
 * (router, top-k, dequant-on-read expert GEMVs, SwiGLU, weighted combine)
 * for single-stream decode and grouped prefill on one GB300 (sm_103a).
 *
 * What the library computes, per token x (H values):
 *   z = W_r x (+ bias); ids = k largest z (descending, equal z -> lower
 *   index); w_i = softmax(z)[ids_i] / sum_j softmax(z)[ids_j];
 *   h_i = silu(W_gate[ids_i] x) * (W_up[ids_i] x);  out = sum_i w_i W_down[ids_i] h_i;
 * or, for a pre-normed block (si_moe_layer.norm_weight), the same on
 * x * gamma / sqrt(mean(x^2) + eps) with x added to out.
 * Sources: sparkinfer README (luciferlive112116), opening section (experts
 * "quantized-resident, dequantized on-read", greedy bs=1 decode of a Q4_K_M
 * GGUF Qwen3-30B-A3B) and "Layout" table (kernels: "decode GEMV", "fused
 * quantized MoE expert FFN", "GGUF dequant"; moe: "sync-free MoE router +
 * expert dispatch (on-device counts, CUDA-graph-ready)"); SP-RKINFER README
 * (gittensor-ai-lab), "Benchmark - Qwen3.8-27B" prefill note (Q4_K is
 * dequantized into the GEMM operand on every prefill pass); the CuTe-DSL
 * sparkinfer README (local-inference-lab), "Using it" (host plan, views-only
 * bind, capture-safe run) for the shape of this interface.
 *
 * Conventions for every call:
 *  - Ownership: the caller owns every device buffer and the stream.  The
 *    library never allocates or frees device memory, never synchronises
 *    inside a forward call, and its forward calls can be captured in a CUDA
 *    graph; the one exception is si_moe_forward_decode_host, which takes
 *    host buffers and waits for its result.  A plan owns host memory only
 *    (for si_moe_forward_decode_host also its captured graphs and their
 *    page-locked staging).
 *  - Device pointers must be 16-byte aligned (SI_ERR_MISALIGNED otherwise).
 *  - Errors: no call throws.  Argument errors are reported before any
 *    launch.  A failed launch returns SI_ERR_CUDA.  Faults found on the
 *    device (a bounded wait that ran out) are recorded in the scratch status
 *    word and returned by si_moe_read_status.
 *  - Threading: calls on one plan are thread-safe when each thread uses its
 *    own scratch buffer.
 *  - Bounded waits: every device-side wait gives up after about one second
 *    and records SI_ERR_TIMEOUT.  Test mode: when the environment variable
 *    SI_FAULT_WAIT_BUDGET holds a decimal cycle count at si_moe_plan time,
 *    that plan's waits use it as their budget and its expert kernels first
 *    wait on a scratch word nothing writes, so the error path (record the
 *    status, skip the rest, let in-flight copies land, return) runs for
 *    certain.  After SI_ERR_TIMEOUT call si_moe_scratch_init again.
 *
 * Q4_K weights (GGUF's block format, unmodified): 144-byte super-blocks of
 * 256 weights {fp16 d, fp16 dmin, u8 scales[12], u8 qs[128]}, blocked along
 * each matrix's input dimension, expert-major:
 *   w_gate, w_up: [E][I rows][H/256 blocks]   (row r of expert e at byte
 *                 ((e*I + r) * H/256) * 144)
 *   w_down:       [E][H rows][I/256 blocks]
 * Q5_K weights (SI_WTYPE_Q5_K; another GGUF K-quant block type -- a Q4_K_M
 * or Q5_K_M file mixes K-quant types; the layout is GGUF's, a reading from
 * outside the pages): 176-byte super-blocks {fp16 d, fp16 dmin, u8
 * scales[12] as in Q4_K, u8 qh[32], u8 qs[128]}, code q = low four bits from
 * qs (arranged as Q4_K's) + 16 * bit j of qh[l] for weight l of sub-block j,
 * weight = d*sc_j*q - dmin*m_j; the same expert-major layout with 176 in
 * place of 144.  All three matrices of a layer have the plan's wtype.  Q5_K
 * layers are plain blocks (a norm_weight gives SI_ERR_UNSUPPORTED).
 */
#ifndef SI_MOE_H
#define SI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *si_stream_t;

typedef enum si_status {
    SI_OK = 0,
    SI_ERR_INVALID_ARG = 1,       /* null pointer, bad size, bad mode */
    SI_ERR_UNSUPPORTED = 2,       /* a shape the library has no kernel for */
    SI_ERR_MISALIGNED = 3,        /* a device pointer not 16-byte aligned */
    SI_ERR_SCRATCH_TOO_SMALL = 4, /* scratch_bytes below si_moe_scratch_bytes() */
    SI_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
    SI_ERR_TIMEOUT = 6,           /* a bounded device-side wait ran out */
    SI_ERR_DEVICE = 7,            /* another device-side check failed */
    SI_ERR_RANGE = 8              /* prefill: a value outside the fp16 range of its tensor-core operands */
} si_status;

#define SI_WTYPE_Q4_K 12          /* GGUF's type id of Q4_K */
#define SI_WTYPE_Q5_K 13          /* GGUF's type id of Q5_K: 176-byte super-blocks (see below) */
#define SI_WTYPE_NVFP4 100        /* NVFP4 super-blocks (see si_moe_layer.w_scale) */
/* si_moe_desc.flags: int8-activation mode of single-token decode (the dp4a
 * matrix-vector product on quantised weights that the sparkinfer README's
 * "Milestone 1" plans, with each activation vector quantised once).  x and h are quantised to int8 per 32
 * columns (q = round-half-even(v * 127/max|v|), scale max|v|/127) and dotted
 * with the 4-bit codes by dp4a; the Q4_K min term uses the exact 32-column
 * sums.  An approximation with its own, looser tolerance (measured against
 * the exact block: about 1e-3 .. 1e-2 rel-L2 per token on synthetic layers,
 * several 1e-2 for a token whose h has an outlier in some 32-column block),
 * reported separately from the default path.  Q4_K only, not with a
 * pre-normed block (SI_ERR_UNSUPPORTED).  It applies where single-token
 * decode runs on the cluster expert kernel (si_debug_decode_fused = 2);
 * batched decode and prefill keep their precision. */
#define SI_FLAG_ACT_INT8 1u
#define SI_MODE_DECODE 0
#define SI_MODE_PREFILL 1
#define SI_MODE_DECODE_HOST 2  /* si_moe_forward_decode_host: decode scratch + x and out staging */
#define SI_MAX_EXPERTS 256
#define SI_MAX_TOPK 16
#define SI_MAX_DECODE_TOKENS 4

/* Layer shape.  hidden and intermediate are multiples of 256 (one Q4_K
 * super-block); 1 <= top_k <= min(n_experts, SI_MAX_TOPK);
 * n_experts <= SI_MAX_EXPERTS; max_tokens bounds the prefill token count.
 * wtype is SI_WTYPE_Q4_K, SI_WTYPE_Q5_K or SI_WTYPE_NVFP4; flags is 0 or SI_FLAG_ACT_INT8
 * (other bits: SI_ERR_UNSUPPORTED). */
typedef struct si_moe_desc {
    int32_t hidden;
    int32_t intermediate;
    int32_t n_experts;
    int32_t top_k;
    int32_t max_tokens;
    int32_t wtype;
    uint32_t flags;
} si_moe_desc;

typedef struct si_moe_plan_s *si_moe_plan_t;

/* Validate desc for device cuda_device and choose launch shapes from its
 * properties (SM count, shared memory, L2).  Host memory only; no device
 * allocation.  *out receives a plan to free with si_moe_plan_destroy. */
si_status si_moe_plan(const si_moe_desc *desc, int cuda_device, si_moe_plan_t *out);
void si_moe_plan_destroy(si_moe_plan_t plan);

/* Bytes of caller-allocated device scratch one forward call of `mode`
 * needs for n_tokens tokens (SI_MODE_DECODE and SI_MODE_DECODE_HOST:
 * 1..SI_MAX_DECODE_TOKENS; SI_MODE_PREFILL: 1..max_tokens).  A buffer sized
 * for n tokens serves any smaller count. */
si_status si_moe_scratch_bytes(si_moe_plan_t plan, int mode, int32_t n_tokens, size_t *bytes);

/* Zero the scratch control block (status word and arrival counters),
 * stream-ordered.  Call once after allocating a scratch buffer, before its
 * first forward call. */
si_status si_moe_scratch_init(si_moe_plan_t plan, void *scratch, size_t scratch_bytes,
                              si_stream_t stream);

/* One layer's weights (device pointers, read only). */
typedef struct si_moe_layer {
    const void *w_gate;        /* Q4_K [E][I][H/256] */
    const void *w_up;          /* Q4_K [E][I][H/256] */
    const void *w_down;        /* Q4_K [E][H][I/256] */
    const float *router_w;     /* fp32 [E][H], row-major */
    const float *router_bias;  /* fp32 [E] added to the logits, or NULL */
    /* Optional pre-normed block (sparkinfer README, "Layout": an RMSNorm kernel
     * runs before the MoE block of each layer).  When norm_weight is non-NULL
     * the call computes out = x + MoE(x * norm_weight / sqrt(mean(x^2) + norm_eps))
     * for each token x: the MoE (router and experts) sees the normalised row,
     * the output gets the un-normalised x back as the residual.  The norm is
     * fused into the kernels that read x and the residual into the ones that
     * write out; no extra launch.  NULL: out = MoE(x). */
    const float *norm_weight;  /* fp32 [H] gain, 16-byte aligned, or NULL */
    float norm_eps;            /* >= 0 and finite (used only with norm_weight) */
    /* NVFP4 experts (wtype SI_WTYPE_NVFP4; sparkinfer README, "Milestone 2":
     * NVFP4 experts; SP-RKINFER README, "Native NVFP4 - two supported
     * checkpoints"; the CuTe-DSL README's moe row: a W4A16 mode with bf16
     * activations and inline FP4 weight dequant).  w_gate, w_up and w_down
     * then hold super-blocks of 256 weights in 144 bytes (the size of a Q4_K
     * block, so the same row layout): bytes 0-15 the FP8 E4M3 scales of
     * weights 16j .. 16j+15, bytes 16-143 the 4-bit E2M1 codes (byte 16 + l:
     * weight 2l in its low nibble, 2l+1 in its high nibble); a weight is
     * e2m1 * e4m3 * g with g the matrix's fp32 tensor scale, given here as
     * [E][3] (gate, up, down of each expert), 4-byte aligned.  NULL for Q4_K
     * (and required for NVFP4).  A checkpoint's separate code and scale
     * tensors are repacked into this layout once, losslessly. */
    const float *w_scale;
} si_moe_layer;

/* Optional routing outputs (device pointers; each may be NULL). */
typedef struct si_moe_route_out {
    int32_t *topk_ids;         /* [n][k] selected experts, descending logit */
    float *topk_w;             /* [n][k] renormalised softmax weights */
    int32_t *expert_counts;    /* [E] tokens (decode) or pairs (prefill) per expert */
    int32_t *expert_offsets;   /* [E+1] exclusive scan of counts (prefill only) */
    int32_t *perm;             /* [n*k] pair ids t*k+slot ordered by expert, then pair id (prefill only) */
    float *logits;             /* [n][E] fp32 router logits */
} si_moe_route_out;

/* Decode: n_tokens (1..SI_MAX_DECODE_TOKENS) independent tokens through one
 * layer.  x_bf16: [n][H] bf16; out: [n][H] fp32 (written, not accumulated).
 * With n_tokens > 1 each selected expert is read once per call and applied
 * to every token that chose it.  Stream-ordered, no host synchronisation. */
si_status si_moe_forward_decode(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                int32_t n_tokens, float *out, si_moe_route_out *route_out,
                                void *scratch, size_t scratch_bytes, si_stream_t stream);

/* Decode with x and out in host memory, for a caller that keeps no device
 * copy of them (a bs=1 generation loop that needs each output on the host
 * before it forms the next token).  x_bf16_host: [n][H] bf16; out_host:
 * [n][H] fp32; any host memory.  The call copies x into page-locked staging,
 * launches one CUDA graph on `stream` (the copy into the scratch, the decode
 * of si_moe_forward_decode, the copies of the result and of the device status
 * back into staging), waits for it, and copies the result into out_host:
 * out_host holds the output when the call returns.  The graph is captured on
 * the first call for a given (layer, route_out, scratch, n) and kept with the
 * plan (the four most recent; freed by si_moe_plan_destroy, with their
 * page-locked staging); the plan serialises these calls.  scratch holds
 * si_moe_scratch_bytes(plan, SI_MODE_DECODE_HOST, n) bytes (the decode scratch
 * followed by device copies of x and out) and was initialised with
 * si_moe_scratch_init; route_out, if given, holds device pointers as for
 * si_moe_forward_decode.  The call reads the device status as
 * si_moe_read_status does: SI_ERR_TIMEOUT or another device-side error is
 * returned (and cleared) by the call that observes it.  Argument errors are
 * returned before anything is queued.  Not usable inside stream capture. */
si_status si_moe_forward_decode_host(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16_host,
                                     int32_t n_tokens, float *out_host, si_moe_route_out *route_out,
                                     void *scratch, size_t scratch_bytes, si_stream_t stream);

/* Grouped prefill (SP⚡RKINFER README, "Benchmark · Qwen3.8-27B", prefill
 * paragraph: Q4_K dequantized into the GEMM operand; sparkinfer-k3 blog post,
 * "v0.2.2": a chunk of tokens shares one weight-tile read): T tokens
 * (1..max_tokens) routed top-k (fp32 logits, ties to the lower index,
 * renormalised softmax), counts per expert, offsets = exclusive scan, perm =
 * pair ids t*k+slot ordered by expert then pair id; per expert a 16-bit
 * tensor-core GEMM of the gathered tokens with the gate and up rows (Q4_K
 * dequantized to fp16, round-to-nearest-even, fp32 accumulation), h =
 * fp16(silu(g)*u), a second GEMM with the down rows, each row times its
 * routing weight (fp32), and out[t] = the sum of token t's k rows in slot
 * order (deterministic).  The tensor-core operands are fp16 (weights and h
 * rounded to nearest even, x converted exactly): bf16 weights cannot hold
 * the output tolerance.  An input, weight or h value beyond the fp16 range
 * is reported as SI_ERR_RANGE by si_moe_read_status (in a pre-normed block
 * the weight check is made before the norm gain is multiplied in, so a gain
 * that pushes a weight past 65504 is not reported).  x_bf16: [T][H] bf16; out: [T][H] fp32 (written).
 * route_out may return ids/weights [T][k], counts [E], offsets [E+1],
 * perm [T*k] and logits [T][E].  Needs H, I multiples of 256 (as every call)
 * and scratch of si_moe_scratch_bytes(plan, SI_MODE_PREFILL, T).  Returns
 * SI_ERR_UNSUPPORTED on a device without the tensor-memory MMA path.
 * Stream-ordered, no host synchronisation, no allocation. */
si_status si_moe_forward_prefill(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                 int32_t n_tokens, float *out, si_moe_route_out *route_out,
                                 void *scratch, size_t scratch_bytes, si_stream_t stream);

/* Synchronise `stream`, return the device status recorded in `scratch`
 * since the last read (SI_OK if none) and clear it. */
si_status si_moe_read_status(si_moe_plan_t plan, const void *scratch, si_stream_t stream);

const char *si_status_string(si_status status);

/* Decode without a caller scratch buffer, for callers that cannot allocate
 * device memory: for example a plug-in inside a host framework whose memory
 * pool owns all device memory and gives it no allocator, or a latency-
 * critical decode loop where cudaMalloc would synchronise the device.  (The
 * sparkinfer pages have no counterpart of this entry point.)
 * Same arguments and results as si_moe_forward_decode, minus the scratch
 * pointer and size, and the same argument errors, all returned before
 * anything is launched or written.  The scratch is one fixed device array of
 * SI_STATIC_SCRATCH_BYTES per GPU, part of the library's module image: every
 * GPU that loads the library holds it until the process exits.  A call whose
 * shape needs more scratch (si_moe_scratch_bytes) is rejected with
 * SI_ERR_SCRATCH_TOO_SMALL.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).  The first call on a device looks
 * up the array's device address with that device current; make that first
 * call before any stream capture.  After cudaDeviceReset the looked-up
 * address is stale and these entry points must not be used on that device.
 * Every call on a device shares the one array, which keeps the previous
 * call's contents; each call clears the words that must start at zero
 * (stream-ordered).  Calls that may overlap on the GPU (different streams, or
 * unordered host threads) race on the array: order them.  Device-side errors
 * (a bounded wait that ran out) are kept in the array's status word until
 * si_moe_read_status_noalloc reads them. */
#define SI_STATIC_SCRATCH_BYTES (1u << 20)
si_status si_moe_forward_decode_noalloc(si_moe_plan_t plan, const si_moe_layer *layer,
                                        const void *x_bf16, int32_t n_tokens, float *out,
                                        si_moe_route_out *route_out, si_stream_t stream);

/* Synchronise `stream` and return the device-side status that calls of
 * si_moe_forward_decode_noalloc on the current device recorded since the last
 * read (SI_OK if none), then clear it.  Like si_moe_read_status, but for the
 * fixed array of those calls; allocates nothing. */
si_status si_moe_read_status_noalloc(si_stream_t stream);

/* Test/bench export: which expert kernels decode of n_tokens tokens runs
 * after the router launch: 2 = the cluster kernel (one launch, n_tokens == 1),
 * 3 = the cluster kernel over the distinct experts (one launch, 2..4 tokens of
 * a block that is not pre-normed; a pre-normed block takes the next choice),
 * 1 = the grid-synchronised fused kernel (one launch), 0 = the generic
 * gate/up + down kernels (two launches); -1 on a bad argument. */
int si_debug_decode_fused(si_moe_plan_t plan, int32_t n_tokens);

/* Test/bench export: up to n plan facts into info[]: SM count, cluster path
 * usable (0/1), CTAs per cluster, clusters of that size resident at once,
 * clusters one token needs (top_k * intermediate/256), shared memory per CTA
 * (opt-in bytes).  Returns the number written, -1 on a bad argument. */
int si_debug_plan_info(si_moe_plan_t plan, int32_t *info, int32_t n);

/* Test exports.  si_debug_q4k_dequant decodes n_blocks Q4_K blocks into
 * out_f32 [n_blocks*256] and/or out_bf16 [n_blocks*256] (either may be
 * NULL): w = d*sc*q - dmin*m rounded once to fp32 (bf16: round-to-nearest-
 * even of that fp32 value).  si_debug_topk runs the decode top-k on given
 * fp32 logits [n][E] (n <= SI_MAX_DECODE_TOKENS) and fills route_out's
 * topk_ids, topk_w and expert_counts. */
si_status si_debug_q4k_dequant(const void *blocks, int64_t n_blocks, float *out_f32,
                               uint16_t *out_bf16, si_stream_t stream);
si_status si_debug_topk(const float *logits, int32_t n, const si_moe_desc *desc,
                        si_moe_route_out *route_out, si_stream_t stream);

/* Test export: the grouped prefill's own Q4_K -> fp16 operand conversion (the
 * device function its GEMM dequantization warps run; SP-RKINFER README,
 * "Benchmark - Qwen3.8-27B", prefill paragraph: Q4_K is dequantized into the
 * GEMM operand on every prefill pass) applied to n_blocks blocks.
 * out_f16[256*b + c] (fp16 bits) = round-to-nearest-even fp16 of the fp32
 * weight w = d*sc*q - dmin*m of column c of block b, or, when gamma
 * ([n_blocks*256] fp32, 16-byte aligned) is non-NULL, of the fp32 product
 * fp32(w) * gamma[256*b + c] (the gate/up operand of a pre-normed block).
 * blocks, out_f16 16-byte aligned.  Stream-ordered. */
si_status si_debug_q4k_dequant_f16(const void *blocks, int64_t n_blocks, const float *gamma, uint16_t *out_f16,
                                   si_stream_t stream);

/* Test export: the grouped prefill's Q5_K -> fp16 operand conversion (the
 * device function its GEMM dequantization warps run for SI_WTYPE_Q5_K)
 * applied to n_blocks 176-byte Q5_K blocks: out_f16[256*b + c] (fp16 bits) =
 * round-to-nearest-even fp16 of the fp32 weight of column c of block b, or,
 * when gamma is non-NULL, of fp32(w) * gamma[256*b + c].  blocks, out_f16
 * (and gamma) 16-byte aligned.  Stream-ordered. */
si_status si_debug_q5k_dequant_f16(const void *blocks, int64_t n_blocks, const float *gamma, uint16_t *out_f16,
                                   si_stream_t stream);

/* Test export: the grouped prefill's NVFP4 -> fp16 operand conversion (the
 * device function its GEMM dequantization warps run for SI_WTYPE_NVFP4)
 * applied to n_blocks NVFP4 super-blocks with tensor scale g.
 * out_f16[256*b + c] (fp16 bits) = round-to-nearest-even fp16 of the fp32
 * weight e2m1 * e4m3 * g (one rounding) of column c of block b.  blocks,
 * out_f16 16-byte aligned.  Stream-ordered. */
si_status si_debug_nvfp4_dequant_f16(const void *blocks, int64_t n_blocks, float g, uint16_t *out_f16,
                                     si_stream_t stream);

/* Timing export: si_moe_forward_decode that also records caller-created
 * cudaEvent_t handles on `stream` -- events[0] before the router kernel,
 * events[1] before the gate/up kernel, events[2] before the down kernel,
 * events[3] after it (any may be NULL).  Recorded as external events, so a
 * CUDA-graph capture keeps them as event-record nodes.  Same arguments,
 * errors and results as si_moe_forward_decode. */
si_status si_debug_decode_events(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                 int32_t n_tokens, float *out, si_moe_route_out *route_out,
                                 void *scratch, size_t scratch_bytes, void *const *events,
                                 si_stream_t stream);

/* Timing export: si_moe_forward_prefill that also records caller-created
 * events on `stream` -- events[0] before routing, [1] before the gate/up GEMM,
 * [2] before the down GEMM, [3] before the combine, [4] after it (any may be
 * NULL).  Same arguments, errors and results as si_moe_forward_prefill. */
si_status si_debug_prefill_events(si_moe_plan_t plan, const si_moe_layer *layer, const void *x_bf16,
                                  int32_t n_tokens, float *out, si_moe_route_out *route_out,
                                  void *scratch, size_t scratch_bytes, void *const *events,
                                  si_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SI_MOE_H */
