/*
 * moe.h -- C ABI of libmoe, a GB300 (sm_103a) implementation of the sparse
 * Mixture-of-Experts FFN sublayer of an LLM decoder.
 *
 * The layer takes the post-norm hidden state x [T][H] and returns the FFN
 * output [T][H] without the residual (the caller adds it):
 *
 *   l      = Wr x (+ b_r)                                        router logits
 *   (idx, w) = softmax -> top-k -> renormalise -> * scale        (mode 0), or
 *              top-k on l -> softmax over the k                  (mode 1)
 *   y_e    = W_down,e act(W_gate,e x, W_up,e x) (+ b_down,e)     each selected e
 *   out    = sum_j w_j y_{idx_j}  +  sigmoid(w_sh . x) * SwiGLU_shared(x)
 *
 * Passages defining the operation:
 *   - "Qwen3.5-MoE Model Implementation" (Pantheon), section "MoE routing":
 *     router [n_expert, n_embd] -> softmax -> top-8 -> norm_topk_prob
 *     renormalisation -> expert_weights_scale; SwiGLU experts; shared expert
 *     with scalar sigmoid gate [n_embd]; out = moe_out + shexp_out, residual
 *     by the caller.
 *   - "Phase 19: MoE -- gpt-oss-20b" (xserv), section 2, Router and Experts:
 *     logits with bias, top-4 then softmax over the 4; fused interleaved
 *     gate_up with bias (gate = even rows, up = odd rows), gate <= limit,
 *     -limit <= up <= limit, h = (up + 1) * gate * sigmoid(alpha * gate),
 *     down with bias.  Measured tensor layout: weights stored [out][in].
 *   - "Llama Forward Pass" (Pantheon), sections "Mixture of Experts
 *     (Mixtral)" and "Expert weight formats in GGUF": merged expert tensors
 *     gate/up [E][F][H], down [E][H][F].
 *   - "Engine" (cherenkov), section "Prefill": tokens grouped by expert,
 *     gathered, projected and scattered back.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major [out][in] (the input dimension contiguous).
 *   - All calls return a moe_status; on failure moe_last_error() describes it
 *     (a per-thread string, valid until the next call on that thread).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is asynchronous on it.
 *   - The library uses the CUDA device that is current when the layer is
 *     created; later calls on that layer must run with the same device
 *     current.
 *   - Public structs carry no build-dependent fields ("Llama Forward Pass",
 *     ABI note on pn_qweight.gpu).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 7

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,     /* bad pointer, size, alignment or config */
    MOE_ERR_UNSUPPORTED = -2,     /* valid but not implemented combination */
    MOE_ERR_OOM = -3,             /* device allocation failed at create */
    MOE_ERR_CUDA = -4,            /* a CUDA runtime call failed */
    MOE_ERR_TOO_MANY_TOKENS = -5, /* n_tokens > config.max_tokens */
    MOE_ERR_DEVICE_TIMEOUT = -6   /* a bounded device-side wait gave up */
} moe_status;

typedef enum {
    MOE_DT_F32 = 0,
    MOE_DT_BF16 = 1,
    /* w_dtype only: the routed experts' weights in MXFP4 ("Phase 19: MoE --
     * gpt-oss-20b", MXFP4 packing note under the measured tensor layout, and
     * section 3, MXFP4 dequantisation).  Each [out][in] matrix row is in/32
     * blocks of 16 bytes = 32 E2M1 codes (low nibble = even element, high
     * nibble = odd element; E2M1 as in the OCP Microscaling formats), blocks
     * along the input dimension, plus one E8M0 byte per block; an element is
     * e2m1(code) * 2^(e8m0 - 127).  gate_up_w / down_w then hold the blocks
     * ([E][2F][H/32][16] and [E][H][F/32][16] bytes) and gate_up_scales /
     * down_scales the scales ([E][2F][H/32], [E][H][F/32]); the router and the
     * biases are bf16 and act_dtype must be bf16.  Requires
     * gate_up_interleaved = 1, shared_ff = 0 and H, F multiples of 64.
     * The layer keeps only the codes and scales (repacked per 128-row,
     * 64-wide K block); both tensor-core paths (weight-streaming decode for up
     * to 16 tokens, grouped GEMMs above) widen them to bf16 on chip, exactly
     * for every E8M0 byte (an E2M1 value times a power of two has at most two
     * significant bits; products beyond the fp32 range are infinite, byte 255
     * is NaN).  The result equals the bf16 layer built from the dequantised
     * weights, up to rounding order.  MOE_PATH_STREAM and MOE_PATH_FUSED are
     * UNSUPPORTED for such a layer, and create is UNSUPPORTED on a device
     * without the tensor-core kernels. */
    MOE_DT_MXFP4 = 2,
    /* w_dtype only: the routed experts as Q4 records ("Engine" (cherenkov),
     * section "Prefill": Q4 expert GEMMs with half weights and float
     * accumulation; the record layout read as the ggml-Q4_0 rows named in
     * "Qwen3.5-MoE Model Implementation", KV Cache).  A record covers 32 consecutive K elements of
     * one row in 18 bytes: a little-endian binary16 scale d, then 16 bytes
     * whose byte j holds element j in its low nibble and element j + 16 in
     * its high nibble; element value = (code - 8) * d.  gate_up_w (or gate_w
     * and up_w), and down_w, hold the records ([E][2F][H/32][18], or
     * [E][F][H/32][18] each, and [E][H][F/32][18] bytes); the router and the
     * biases are bf16 and act_dtype must be bf16.  Requires shared_ff = 0
     * and H, F multiples of 64; gate_up_scales and down_scales stay NULL.
     * The layer keeps only the records, repacked per 128-row, 64-wide K
     * block (codes, then the scales); both tensor-core paths widen them on
     * chip to bf16, each weight (code - 8) * d computed exactly in fp32 and
     * rounded once to bf16 (round to nearest even), because the tensor
     * cores multiply the bf16 activations with operands of the same type.
     * The result equals the bf16 layer built from those rounded weights, up
     * to rounding order.  The paths and devices supported are those of
     * MOE_DT_MXFP4. */
    MOE_DT_Q4 = 3
} moe_dtype;

typedef enum {
    /* softmax over all experts -> top-k -> (renormalise) -> * weights_scale
     * ("Qwen3.5-MoE Model Implementation", MoE routing; "Llama Forward
     * Pass", Mixture of Experts) */
    MOE_ROUTER_SOFTMAX_TOPK = 0,
    /* top-k on the (biased) logits -> softmax over the k selected
     * ("Phase 19: MoE -- gpt-oss-20b", section 2, Router) */
    MOE_ROUTER_TOPK_SOFTMAX = 1
} moe_router_mode;

typedef enum {
    MOE_ACT_SWIGLU = 0,      /* h = silu(gate) * up */
    MOE_ACT_CLAMP_GLU = 1    /* gpt-oss: g = min(gate, limit), u = clamp(up, -limit, limit),
                                h = (u + 1) * g * sigmoid(alpha * g) */
} moe_act;

typedef struct {
    int32_t hidden;              /* H; multiple of 8 (64 for the tensor-core path) */
    int32_t n_expert;            /* E; 1 .. 1024 */
    int32_t top_k;               /* k; 1 .. min(E, 32) */
    int32_t expert_ff;           /* F; multiple of 8 (64 for the tensor-core path) */
    int32_t shared_ff;           /* Fs; 0 = no shared expert, else multiple of 8 (64 for tensor cores) */
    int32_t router_mode;         /* moe_router_mode */
    int32_t norm_topk_prob;      /* mode 0: 1 = divide the kept probabilities by their sum */
    float weights_scale;         /* mode 0: multiplier after renormalisation (1.0) */
    int32_t act;                 /* moe_act (the routed experts; the shared expert is SwiGLU) */
    float act_alpha;             /* MOE_ACT_CLAMP_GLU: 1.702 */
    float act_limit;             /* MOE_ACT_CLAMP_GLU: 7.0 */
    int32_t has_bias;            /* router [E], gate_up [E][2F], down [E][H] biases */
    int32_t gate_up_interleaved; /* 1: one [E][2F][H] gate_up tensor, gate = even rows */
    int32_t w_dtype;             /* moe_dtype of every weight and bias (MOE_DT_MXFP4, MOE_DT_Q4: see moe_dtype) */
    int32_t act_dtype;           /* moe_dtype of x; must equal w_dtype (bf16 with MOE_DT_MXFP4, MOE_DT_Q4) */
    int32_t out_dtype;           /* moe_dtype of out */
    int32_t max_tokens;          /* workspace is sized once for this many tokens */
    /* Expert residency ("Engine" (cherenkov), sections "Decode and expert
     * IO" and "Memory ownership": a bounded pool of resident experts, the
     * rest streamed in on demand, resident experts addressed through a
     * table).  0: every routed expert stays in device memory.  S in
     * [min(E, 16 * top_k), E): the routed experts' weights (after repacking)
     * live in pinned host memory, read by the GPU over the host link, and S
     * device slots hold the resident ones; every forward runs as chunks of
     * up to 16 tokens, each chunk selecting its experts, keeping resident
     * ones (hits) and copying the others from host memory into the least
     * recently used slots that no expert of the chunk needs (ties: lowest
     * slot), then running the weight-streaming tensor-core kernel through the
     * slot table.  Results are bitwise those of the fully resident layer.
     * Needs the weight-streaming tensor-core path (bf16, MXFP4 or Q4 experts;
     * H, F, Fs multiples of 64); slots start with experts 0 .. S - 1. */
    int32_t resident_experts;
} moe_config;

/* Weights: pointers to memory that cudaMemcpy can read (device memory, or
 * host memory under unified addressing), in w_dtype.  moe_layer_create copies
 * (and repacks) them into library-owned device memory; the caller may free its
 * copies when create returns.  Unused fields must be NULL. */
typedef struct {
    const void *router_w;    /* [E][H] */
    const void *router_b;    /* [E]            (has_bias) */
    const void *gate_w;      /* [E][F][H]      (!gate_up_interleaved) */
    const void *up_w;        /* [E][F][H]      (!gate_up_interleaved) */
    const void *gate_up_w;   /* [E][2F][H]     (gate_up_interleaved) */
    const void *gate_up_b;   /* [E][2F]        (has_bias): interleaved order when
                                gate_up_interleaved, else [gate F | up F] */
    const void *down_w;      /* [E][H][F] */
    const void *down_b;      /* [E][H]         (has_bias) */
    const void *sh_gate_w;   /* [Fs][H]        (shared_ff > 0) */
    const void *sh_up_w;     /* [Fs][H] */
    const void *sh_down_w;   /* [H][Fs] */
    const void *sh_gate_inp; /* [H] scalar-gate vector */
    const void *gate_up_scales; /* [E][2F][H/32] E8M0 bytes (w_dtype MOE_DT_MXFP4 only) */
    const void *down_scales;    /* [E][H][F/32] E8M0 bytes (w_dtype MOE_DT_MXFP4 only) */
} moe_weights;

typedef struct moe_layer moe_layer;

/* Validates the config, copies/repacks the weights and allocates all device
 * workspace for config.max_tokens.  Synchronous.  On failure *out is NULL and
 * nothing stays allocated.  Errors: INVALID_ARG (NULL pointer, inconsistent
 * config, a required weight missing), UNSUPPORTED (act_dtype != w_dtype,
 * sizes not multiples of 8), OOM, CUDA. */
moe_status moe_layer_create(const moe_config *config, const moe_weights *weights, moe_layer **out);

/* out[n_tokens][H] (out_dtype) = the layer applied to x[n_tokens][H]
 * (act_dtype).  x and out are caller-owned device pointers, 16-byte aligned,
 * non-overlapping.  Asynchronous on `stream`; allocates nothing and never
 * synchronises the host.  Results are bitwise reproducible for the same
 * inputs (fixed-order combine, no floating-point atomics).  n_tokens == 0 is
 * a no-op.  Errors: INVALID_ARG (NULL / misaligned / aliasing pointers,
 * n_tokens < 0), TOO_MANY_TOKENS (n_tokens > max_tokens), CUDA (launch
 * failure).  Device-side wait timeouts are reported by moe_get_status.
 * Calls on one layer must not overlap on the GPU (they share its workspace):
 * issue them on one stream or order them with events. */
moe_status moe_forward(moe_layer *layer, const void *x, int32_t n_tokens, void *out, void *stream);

/* Same as moe_forward with x and out in HOST memory (pinned memory makes the
 * copies asynchronous).  The copies in and out go through device staging
 * buffers allocated at create: x is copied in on a stream of the layer's own
 * (created at the first call), after the previous forward of this layer has
 * read the staging buffer, so that the copy overlaps the work still queued
 * on `stream`, which waits for it.  out is copied on `stream`, except for a
 * batch the weight-streaming decode kernels take (and with expert residency)
 * when out is pinned memory mapped into the device's address space: that
 * kernel then writes out directly.  The caller must synchronise `stream`
 * before reading out, and keep x valid until then. */
moe_status moe_forward_host(moe_layer *layer, const void *x_host, int32_t n_tokens, void *out_host,
                            void *stream);

/* Routing of the last forward: idx[n][k] (int32, descending weight, ties to
 * the lower expert index) and w[n][k] (fp32), n = that forward's n_tokens.
 * Device pointers; either may be NULL.  Asynchronous on `stream`. */
moe_status moe_get_routing(moe_layer *layer, int32_t *idx, float *w, void *stream);

/* Router logits of the last forward: logits[n][E] fp32 (router bias included)
 * and, with a shared expert, its gate logit sh[n] (w_sh . x).  Device
 * pointers; either may be NULL.  Asynchronous on `stream`. */
moe_status moe_get_logits(moe_layer *layer, float *logits, float *sh_logit, void *stream);

/* Number of token rows routed to each expert in the last forward:
 * counts[E] int32 (device pointer).  Asynchronous on `stream`. */
moe_status moe_get_expert_counts(moe_layer *layer, int32_t *counts, void *stream);

/* Intermediates of the last forward, for checking each step against a
 * reference ("Engine" (cherenkov), section "Prefill": tokens grouped by
 * expert, gathered, projected and scattered back).  Kept only by the grouped
 * paths (MOE_PATH_TC and MOE_PATH_STREAM); after a decode-path forward a
 * non-NULL dst returns UNSUPPORTED.  n = that forward's n_tokens, k = top_k.
 *   MOE_INTER_OFFSETS  int32 [E + 1]: exclusive prefix sum of the per-expert
 *                      row counts (expert e's rows start at offsets[e])
 *   MOE_INTER_PERM     int32 [n k]: the pair ids p = t k + slot in expert
 *                      order (a stable sort by expert: ascending p within one)
 *   MOE_INTER_H        [n k (+ n)][max(F, Fs)] in the weight dtype: the
 *                      activation act(gate, up) of each routed row in the
 *                      order of MOE_INTER_PERM, then the shared expert's rows
 *                      (token order) when the layer has one
 *   MOE_INTER_YS       fp32 [n][k + 1][H]: w_slot (W_down h + b_down) of every
 *                      (token, slot), and in slot k the gated shared-expert
 *                      output (zeros-free only when the layer has one)
 * *size (if non-NULL) receives the byte count; dst NULL only queries it.
 * dst is a device pointer of `capacity` bytes.  Asynchronous on `stream`. */
typedef enum {
    MOE_INTER_OFFSETS = 0,
    MOE_INTER_PERM = 1,
    MOE_INTER_H = 2,
    MOE_INTER_YS = 3
} moe_intermediate;
moe_status moe_get_intermediate(moe_layer *layer, int32_t which, void *dst, size_t capacity, size_t *size,
                                void *stream);

/* Kernel-path selection, for tests and benchmarks. */
typedef enum {
    MOE_PATH_AUTO = 0,     /* default: DECODE_TC, else FUSED, else TC, else STREAM (first that applies) */
    MOE_PATH_STREAM = 1,   /* weight-streaming CUDA-core kernels (any dtype) */
    MOE_PATH_TC = 2,       /* tcgen05 grouped GEMMs (bf16, H, F, Fs multiples of 64);
                              UNSUPPORTED otherwise */
    MOE_PATH_FUSED = 3,    /* the whole layer in one cooperative CUDA-core kernel, for up to 8
                              tokens (top_k * n_tokens <= 256, F a multiple of 16) */
    MOE_PATH_DECODE_TC = 4 /* weight-streaming tcgen05 kernels for up to 16 tokens (bf16, H, F,
                              Fs multiples of 64): weight rows are the MMA's M operand */
    /* While FUSED or DECODE_TC is forced, forward returns UNSUPPORTED for a
     * batch the path does not cover. */
} moe_path;
moe_status moe_set_path(moe_layer *layer, int32_t path);

/* Per-kernel timing (tracing).  While enabled, each forward records a CUDA
 * event before and after every kernel it launches, on the forward's stream
 * (events created here, once; nothing is allocated per forward).  Up to
 * `max_forwards` forwards are recorded between two moe_timing_read calls; later
 * ones are not recorded.  max_forwards = 0 disables timing and frees the
 * events.  Errors: INVALID_ARG (max_forwards < 0 or > 4096), CUDA. */
moe_status moe_timing_enable(moe_layer *layer, int32_t max_forwards);

/* Kernel kinds reported by moe_timing_read, in this order. */
typedef enum {
    MOE_KERNEL_ROUTER = 0,   /* router logits */
    MOE_KERNEL_SELECT = 1,   /* softmax / top-k / weights */
    MOE_KERNEL_GROUP = 2,    /* grouping by expert */
    MOE_KERNEL_UP = 3,       /* gate/up projection + activation */
    MOE_KERNEL_DOWN = 4,     /* down projection + routing weight */
    MOE_KERNEL_COMBINE = 5,  /* fixed-order combine */
    MOE_KERNEL_GATHER = 6,   /* token-row gather (tensor-core path) */
    MOE_KERNEL_FUSED = 7,    /* whole layer in one kernel (fused decode path) */
    MOE_KERNEL_EXPERTS = 8,  /* selection, gate/up and down in one persistent kernel
                                (weight-streaming tensor-core decode path) */
    MOE_KERNEL_EXPERTS_MXFP4 = 9, /* the same kernel streaming MXFP4 codes and scales */
    MOE_KERNEL_EXPERTS_Q4 = 10,   /* the same kernel streaming Q4 records */
    MOE_KERNEL_RESIDENCY = 11,    /* expert residency: slot assignment and the copies from host memory */
    MOE_KERNEL_COUNT = 12
} moe_kernel_kind;

/* Synchronises the device, then writes, per kernel kind, the summed device
 * time in milliseconds (total_ms[MOE_KERNEL_COUNT]) and the number of
 * launches (launches[MOE_KERNEL_COUNT]) of the forwards recorded since the
 * last read, and starts a new recording window.  Errors: INVALID_ARG (timing
 * not enabled, NULL pointer), CUDA. */
moe_status moe_timing_read(moe_layer *layer, float *total_ms, int32_t *launches);

/* Synchronises the device and reports a device-side error recorded by the
 * layer's kernels (MOE_ERR_DEVICE_TIMEOUT), then clears it and resets the
 * layer's inter-block counters so that the next forward starts clean (the
 * output of the forward that failed is not valid).  MOE_OK if none. */
moe_status moe_get_status(moe_layer *layer);

/* Expert residency (config.resident_experts > 0).  Synchronises the device
 * and writes, when non-NULL: expert_of[S] = the expert each slot holds (-1:
 * none yet), and stats[3] = hits, misses (experts copied from host memory)
 * and bytes copied, counted over every chunk since create.  Errors:
 * INVALID_ARG (NULL layer), UNSUPPORTED (no residency on this layer), CUDA. */
moe_status moe_get_residency(moe_layer *layer, int32_t *expert_of, int64_t *stats);

/* Bound, in nanoseconds, of every wait of the layer's kernels on work of
 * another thread block (a grid barrier, another block's activations, the
 * injected wait below); ns <= 0 restores the default of one second, values
 * under 1000 become 1000.  A wait that runs out records
 * MOE_ERR_DEVICE_TIMEOUT for moe_get_status, and the kernel stops issuing
 * work, waits for its own copies and tensor-core operations in flight and
 * returns.  Waits inside one block's pipeline keep the one-second bound.
 * Takes effect at the next forward.  Errors: INVALID_ARG (ns above 10 s). */
moe_status moe_set_wait_limit(moe_layer *layer, int64_t ns);

/* Test-only fault injection ("Qwen3.5-MoE Model Implementation", Gotchas and
 * Fragile Spots: failures must not be silent).  While on, every forward makes
 * its kernels wait for a condition that nothing satisfies -- a grid barrier
 * one arrival short (fused decode path), a group's activations one tile short
 * (weight-streaming decode path), a device word that stays zero (tensor-core
 * GEMMs) -- so that the wait runs out after the wait limit, the output is not
 * valid and moe_get_status reports MOE_ERR_DEVICE_TIMEOUT.  No GPU fault is
 * involved.  Off by default. */
moe_status moe_set_fault_injection(moe_layer *layer, int32_t on);

/* Number of kernel launches the last forward issued. */
int32_t moe_last_launch_count(const moe_layer *layer);

/* n_tokens of the last forward that returned MOE_OK (0 before the first, or
 * for a NULL layer): the row count n that moe_get_routing, moe_get_logits and
 * moe_get_intermediate write, so that a caller can size its buffers. */
int32_t moe_last_token_count(const moe_layer *layer);

/* Device bytes owned by the layer (weights + workspace). */
size_t moe_device_bytes(const moe_layer *layer);

/* Frees everything the layer owns.  Synchronises the device first.  NULL is
 * a no-op. */
void moe_destroy(moe_layer *layer);

/* Routing without any device allocation: router logits, top-k selection with
 * routing weights, and per-expert token counts, for callers that must not call
 * cudaMalloc (an application that owns all device memory through its own pool,
 * a process whose allocator is frozen after start-up, a real-time loop where
 * an allocation and the synchronisation it can bring are not allowed).  The
 * pages have no counterpart of this entry point; it computes the routing that
 * moe_forward reports (moe_get_routing / moe_get_expert_counts) without a
 * layer, with the same selection routine: the logits are fp32 dot products
 * whose rounding order may differ from the layer's router kernels, so a token
 * whose k-th and (k+1)-th logits nearly tie may pick differently.
 *
 * x [n_tokens][hidden], router_w [n_expert][hidden] and the optional router_b
 * [n_expert] are device pointers in `dtype` (x and router_w 16-byte aligned);
 * outputs are device pointers: idx [n_tokens][top_k] int32 (descending weight,
 * ties to the lower expert index), w [n_tokens][top_k] fp32, counts [n_expert]
 * int32 (zeroed by the call).  router_mode, norm_topk_prob and weights_scale
 * mean what they mean in moe_config.  Asynchronous on `stream`.
 *
 * The logits are kept in a static device array of 262144 floats (1 MiB) that
 * every GPU holding the library keeps until the process exits:
 * n_tokens * n_expert above 262144 returns MOE_ERR_TOO_MANY_TOKENS.  All calls
 * on a device share that array and it keeps the last call's contents, so calls
 * that overlap on the GPU race; order them (one stream, or events).  The first
 * call on each device looks the array's address up (cudaGetSymbolAddress) with
 * that device current, and looks it up again when the device's CUDA context
 * has changed since (after cudaDeviceReset, say); make that first call before
 * any stream capture.  Other
 * errors: INVALID_ARG (NULL or misaligned pointer, bad size, mode or dtype),
 * UNSUPPORTED (top_k > 32, n_expert > 1024, hidden not a multiple of 8, device
 * ordinal >= 64), CUDA. */
moe_status moe_route_noalloc(const void *x, const void *router_w, const void *router_b, int32_t n_tokens,
                             int32_t hidden, int32_t n_expert, int32_t top_k, int32_t router_mode,
                             int32_t norm_topk_prob, float weights_scale, int32_t dtype, int32_t *idx, float *w,
                             int32_t *counts, void *stream);

/* Expert parallelism: index arithmetic (host pointers, int32; no device work).
 * The pages list expert parallelism as not done ("Phase 19: MoE --
 * gpt-oss-20b", section 6); the split builds on the grouping step ("Engine"
 * (cherenkov), section "Prefill").  n_ranks ranks, rank g owns the experts
 * [first_expert[g], first_expert[g+1]) (ascending, first_expert[0] = 0,
 * first_expert[n_ranks] = n_expert).  Each rank routes its own tokens and
 * orders its (token, slot) pairs by expert (MOE_INTER_PERM), which groups them
 * by owning rank.
 *
 * moe_ep_send_plan: counts[n_expert] = the local pairs per expert ->
 *   send_counts[g], send_displs[g]: the rows of the expert-ordered pairs that
 *   go to rank g (one all-to-all of token rows dispatches them).
 * moe_ep_recv_plan: counts_from[n_ranks][n_local] = what each rank sends this
 *   one per local expert (an all-to-all of the count rows) -> recv_counts[g],
 *   recv_displs[g] of the arriving rows (source-major), order[n_recv]: the
 *   arriving row at position i of the local expert-major order (expert
 *   ascending, then source rank, then the source's order), group_offsets
 *   [n_local + 1] of each local expert in that order.  The experts' outputs go
 *   back in arrival order (the inverse all-to-all), so each source gets them in
 *   its own expert order and scatters them to (token, slot) for the fixed
 *   slot-order combine.
 * Errors: INVALID_ARG (NULL pointer, bad ranges, negative counts, more than
 * 2^31 - 1 rows). */
moe_status moe_ep_send_plan(int32_t n_expert, int32_t n_ranks, const int32_t *first_expert, const int32_t *counts,
                            int32_t *send_counts, int32_t *send_displs);
moe_status moe_ep_recv_plan(int32_t n_ranks, int32_t n_local, const int32_t *counts_from, int32_t *recv_counts,
                            int32_t *recv_displs, int32_t *order, int32_t *group_offsets);

/* Description of the last error on this thread ("" if none). */
const char *moe_last_error(void);

/* MOE_ABI_VERSION of the loaded library. */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
