/*
 * moe_oracle.h -- plain, slow, double-precision CPU oracle for the sparse
 * Mixture-of-Experts FFN sublayer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no source with the CUDA path.
 *
 * What it computes (per token t, independently):
 *   1. router logits  l[e] = sum_i Wr[e][i] * x[i]  (+ b_r[e] when has_bias)
 *        - "Qwen3.5-MoE Model Implementation", section "MoE routing" (Router)
 *        - "Phase 19: MoE -- gpt-oss-20b", section 2, Router (logits = x W^T + b)
 *        - "Llama Forward Pass", section "Mixture of Experts (Mixtral)"
 *   2. selection + weights
 *        mode 0: p = softmax(l); top-k of p; w = p_sel / sum(p_sel) (if
 *                norm_topk_prob); w *= weights_scale
 *                ("Qwen3.5-MoE Model Implementation", "MoE routing";
 *                 "Llama Forward Pass", "Mixture of Experts (Mixtral)")
 *        mode 1: top-k of l (bias included); w = softmax over the k selected
 *                ("Phase 19: MoE -- gpt-oss-20b", section 2, Router)
 *        ties: the lower expert index wins; output order is descending weight.
 *   3. each selected expert
 *        act 0 (SwiGLU): h = silu(Wg x) * (Wu x); y = Wd h
 *                ("Llama Forward Pass", "SwiGLU FFN" and "Mixture of Experts")
 *        act 1 (gpt-oss): z = Wgu x + b_gu; gate = z[2j] (even), up = z[2j+1]
 *                (odd); gate = min(gate, limit); up = clamp(up, -limit, limit);
 *                h = (up + 1) * gate * sigmoid(alpha * gate); y = Wd h + b_d
 *                ("Phase 19: MoE -- gpt-oss-20b", section 2, Experts)
 *   4. moe_out = sum_j w_j * y_j
 *   5. shared expert (shared_ff > 0):
 *        out = moe_out + sigmoid(w_sh . x) * Wsd (silu(Wsg x) * (Wsu x))
 *      ("Qwen3.5-MoE Model Implementation", "MoE routing": shared expert with
 *       scalar sigmoid gate, combine; the residual is the caller's)
 *
 * All matrices are [out][in], row-major (the input dimension contiguous):
 * gate/up [E][F][H], down [E][H][F], interleaved gate_up [E][2F][H]
 * ("Llama Forward Pass", "Expert weight formats in GGUF"; "Phase 19",
 * measured tensor layout: rows = out, cols = in).
 * Every value is read as the exact fp32 or bf16 number stored and converted to
 * double; all arithmetic is double.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_ROUTER_SOFTMAX_TOPK = 0, ORC_ROUTER_TOPK_SOFTMAX = 1 };
enum { ORC_ACT_SWIGLU = 0, ORC_ACT_CLAMP_GLU = 1 };

typedef struct {
    int hidden;          /* H */
    int n_expert;        /* E */
    int top_k;           /* k */
    int expert_ff;       /* F */
    int shared_ff;       /* Fs, 0 = no shared expert */
    int router_mode;     /* ORC_ROUTER_* */
    int norm_topk_prob;  /* mode 0: divide by the selected sum */
    double weights_scale;
    int act;             /* ORC_ACT_* */
    double act_alpha;    /* 1.702 for gpt-oss */
    double act_limit;    /* 7.0 for gpt-oss */
    int has_bias;        /* router bias [E], gate_up bias [E][2F], down bias [E][H] */
    int gate_up_interleaved; /* 1: one [E][2F][H] tensor, gate = even rows */
    int w_dtype;         /* ORC_F32 / ORC_BF16: all weights and biases */
    int x_dtype;         /* ORC_F32 / ORC_BF16: the input activations */
} orc_config;

typedef struct {
    const void *router_w;    /* [E][H] */
    const void *router_b;    /* [E] (has_bias) */
    const void *gate_w;      /* [E][F][H] (not interleaved) */
    const void *up_w;        /* [E][F][H] (not interleaved) */
    const void *gate_up_w;   /* [E][2F][H] (interleaved) */
    const void *gate_up_b;   /* [E][2F] (has_bias); interleaved order when
                                gate_up_interleaved, else [gate F | up F] */
    const void *down_w;      /* [E][H][F] */
    const void *down_b;      /* [E][H] (has_bias) */
    const void *sh_gate_w;   /* [Fs][H] */
    const void *sh_up_w;     /* [Fs][H] */
    const void *sh_down_w;   /* [H][Fs] */
    const void *sh_gate_inp; /* [H] scalar-gate vector */
} orc_weights;

/* 0 on success, negative on a bad argument. */
int orc_check_config(const orc_config *c);

/* Router logits for T tokens: logits [T][E]; sh_logit [T] (may be NULL;
 * only written when shared_ff > 0). */
int orc_router_logits(const orc_config *c, const orc_weights *w, const void *x,
                      int n_tokens, double *logits, double *sh_logit);

/* Selection for one token from its logits row: idx[k], wt[k]. */
int orc_select(const orc_config *c, const double *logits_row, int *idx, double *wt);

/* Routing weights that a given selection (idx[k]) would receive, from the
 * token's own logits (used to score the alternatives of a near tie). */
int orc_weights_for_selection(const orc_config *c, const double *logits_row,
                              const int *idx, double *wt);

/* One routed expert on one token: h[F] (activation), y[H] (down output,
 * bias included, not yet weighted).  x_row is double. */
int orc_expert(const orc_config *c, const orc_weights *w, int e,
               const double *x_row, double *h, double *y);

/* Shared expert on one token: h[Fs], y[H] (ungated) and the gate sigmoid. */
int orc_shared(const orc_config *c, const orc_weights *w, const double *x_row,
               double *h, double *y, double *gate);

/* Whole layer for one token with a given selection and weights. */
int orc_token_output(const orc_config *c, const orc_weights *w, const double *x_row,
                     const int *idx, const double *wt, double *out_row);

/* Whole layer for the tokens listed in rows[n_rows] (NULL = all 0..T-1) of x.
 * Writes out[n_rows][H], idx[n_rows][k], wt[n_rows][k] (idx / wt may be NULL).
 * n_threads <= 0 uses the OpenMP default. */
int orc_forward(const orc_config *c, const orc_weights *w, const void *x,
                int n_tokens, const int *rows, int n_rows, double *out,
                int *idx, double *wt, int n_threads);

/* Number of OpenMP threads the library would use (1 without OpenMP). */
int orc_max_threads(void);

/* MXFP4 expert weights ("Phase 19: MoE -- gpt-oss-20b", the MXFP4 packing
 * note under the measured tensor layout, and section 3, MXFP4 dequantisation):
 * each row of an [out][in] matrix is stored as in/32 blocks of 16 bytes = 32
 * four-bit E2M1 codes (low nibble = even element, high nibble = odd element),
 * blocks running along the input dimension, with one E8M0 byte per block;
 * value = e2m1(code) * 2^(e8m0 - 127).  E2M1 (OCP Microscaling formats): bit 3
 * sign, bits 2..1 exponent with bias 1, bit 0 mantissa; exponent 0 encodes
 * 0 or 0.5 (subnormal), otherwise 1.m * 2^(exponent - 1).  E8M0 255 is NaN.
 *
 * orc_e2m1_value: the value of one code (0..15).
 * orc_e8m0_scale: the scale of one E8M0 byte.
 * orc_mxfp4_dequant: out[rows][cols] (float; every value is exact in float)
 *   from blocks [rows][cols/32][16] and scales [rows][cols/32]; cols must be
 *   a positive multiple of 32.  Returns 0, or -1 on a bad argument. */
double orc_e2m1_value(unsigned code);
double orc_e8m0_scale(unsigned e8m0);
int orc_mxfp4_dequant(const uint8_t *blocks, const uint8_t *scales, int64_t rows, int cols, float *out);

/* Q4 records ("Engine" (cherenkov), section "Prefill"; the ggml-Q4_0 rows of
 * "Qwen3.5-MoE Model Implementation", KV Cache): a row of cols elements is
 * cols/32 blocks of 18 bytes -- a binary16 scale d (little-endian), then 16
 * bytes whose byte j holds element j (low nibble) and element j + 16 (high
 * nibble); element = (code - 8) * d.
 * orc_fp16_value: the value of one binary16 bit pattern (exact).
 * orc_q4_dequant: out[rows][cols] (every value is exact in float: a 4-bit
 * integer times an 11-bit significand). */
double orc_fp16_value(unsigned h);
int orc_q4_dequant(const uint8_t *blocks, int64_t rows, int cols, float *out);

#ifdef __cplusplus
}
#endif
#endif
