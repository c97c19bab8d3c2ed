/*
 * Reference oracle for the expert-major chunked MoE prefill layer: plain, slow, float64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls this library; only the tests, the
 * smoke check and the benchmark's CPU-baseline leg do. It shares no code, header or table with the CUDA library.
 *
 * Sources. The layer is described by four pull-request pages of one inference engine:
 *   [DP-a] "deep prefill" draft, slice 3 of 7: sections "What", "Exactness", and the maintainer review ("To land").
 *   [DP-b] "EXL3 Flash Next: deep prefill (3/8)": sections "What this changes", "Device results", "Checklist".
 *   [DP-c] "Flash Next EXL3: exact deep prefill": introduction, "Completed final functional audit",
 *          "Independent numerical-phase audit".
 *   [UMB]  umbrella draft PR #1113: "What it adds", "Memory and execution split", "Latest prefill efficiency
 *          candidate", "Latest measured follow-up".
 * The pages name the steps (routed experts plus a resident shared expert, expert-major chunks, per-expert member
 * lists, gate/up and down projections, a canonical fixed-order reduction of the routed contributions) but print no
 * formula for any of them. Where they are silent this oracle takes the plainest reading, stated at each function.
 *
 * Parity pins (the tests): bf16 rounding against closed-form midpoint cases and a library conversion; router
 * logits against a library matmul; top-k against routing invariants and planted ties; the FFN against a textbook
 * numpy SwiGLU; the whole layer against a numpy dense masked evaluation (every expert) and a hand-worked example;
 * the permutation against a stable library sort; the fp32 combine against hand-built exact and midpoint cases; the
 * float64 tree combine against a hand-worked example (order, signed zeros, the float32 step) and exact integer sums.
 *
 * Conventions: BF16 values are passed as their uint16 bit patterns and decoded exactly. Row-major layouts.
 * All functions return 0 on success and -1 on a bad argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t hidden;        /* H */
  int32_t n_experts;     /* E, routed experts */
  int32_t inter;         /* I, routed expert intermediate size */
  int32_t top_k;         /* k */
  int32_t shared_inter;  /* I_s, 0 = no shared expert */
} oracle_dims;

int oracle_num_threads(void);

/* Exact bfloat16 -> double. */
double oracle_bf16_to_double(uint16_t b);
/* double -> bfloat16, round to nearest, ties to even, in ONE rounding step (no pass through float). */
uint16_t oracle_bf16_from_double(double v);
int oracle_bf16_round_array(const double* in, uint16_t* out, int64_t n);

/* Router logits l[t][e] = sum_i x[t][i] * w_router[e][i], float64, i ascending from 0.0. */
int oracle_router_logits(const uint16_t* x, const uint16_t* w_router, int64_t n_tokens, int32_t hidden,
                         int32_t n_experts, double* logits /* [n_tokens][E] */);

/* Top-k by (logit desc, expert id asc); ids written in ascending id order; weights = softmax over the k selected
   logits (renormalised). */
int oracle_topk(const double* logits, int64_t n_tokens, int32_t n_experts, int32_t top_k,
                int32_t* topk_id /* [n][k] */, double* topk_w /* [n][k] */);

/* One SwiGLU expert on one token: g = x.Wgu[0:I]^T, u = x.Wgu[I:2I]^T, h = bf16(silu(g)*u), y = h.Wdown^T. */
int oracle_swiglu_ffn(const uint16_t* x_row, const uint16_t* w_gu /* [2I][H] */, const uint16_t* w_down /* [H][I] */,
                      int32_t hidden, int32_t inter, double* y /* [H] */, uint16_t* h_bf16 /* [I] or NULL */);

/* The whole layer on a set of tokens. token_idx lists the tokens to evaluate (NULL = all n_tokens, in order).
   Outputs are per evaluated token: out_ref (float64, before the final rounding), out_bf16 (bf16 RNE of out_ref),
   topk_id / topk_w (may be NULL). */
int oracle_moe_forward(const oracle_dims* dims, const uint16_t* x, const uint16_t* w_router,
                       const uint16_t* w_gu, const uint16_t* w_down, const uint16_t* ws_gu, const uint16_t* ws_down,
                       int64_t n_tokens, const int64_t* token_idx, int64_t n_eval,
                       double* out_ref, uint16_t* out_bf16, int32_t* topk_id, double* topk_w);

/* Per-chunk member lists: chunk c covers tokens [c*chunk, min((c+1)*chunk, T)). Rows of a chunk are ordered by
   (expert asc, token asc). expert_offsets [n_chunks][E+1] (chunk-local), row_token [T*k] (row j of chunk c at
   c*chunk*k + j, holding the global token id), token_row [T][k] (chunk-local row of each (token, slot)). */
int oracle_permutation(const int32_t* topk_id, int64_t n_tokens, int32_t top_k, int32_t n_experts, int32_t chunk,
                       int32_t* expert_offsets, int32_t* row_token, int32_t* token_row);

/* Weighted combine in float64: out_ref[t] = sum_s w[t][s]*y[token_row[t][s]] (s ascending) + s_shared[t]. */
int oracle_combine_f64(const float* y, const float* w, const int32_t* token_row, const float* s_shared,
                       int64_t n, int32_t top_k, int32_t hidden, double* out_ref, uint16_t* out_bf16);

/* The same combine as the fixed-order float32 reduction: acc = +0.0f; per slot acc = acc + (w*y) with each multiply
   and add rounded to float32 (no contraction); then acc = acc + s_shared; out = bf16 RNE of acc. */
int oracle_combine_f32_canonical(const float* y, const float* w, const int32_t* token_row, const float* s_shared,
                                 int64_t n, int32_t top_k, int32_t hidden, uint16_t* out_bf16);

/*
 * Expert-parallel combine with float64 partials ([DP-b] "What this changes", "Checklist"). The routed contributions
 * of one output element are the leaves of a complete binary tree over the expert ids 0 .. Ep-1 (Ep = the least power
 * of two >= n_experts): leaf e = (double)w * (double)y for the slot routed to expert e (exact: a product of two
 * floats fits in a double), +0.0 for every expert the token did not choose; each inner node = left + right in
 * float64, round to nearest. An expert-parallel split has n_parts aligned blocks of Ep/n_parts ids (n_parts a power
 * of two, 1 <= n_parts <= Ep): part p holds the experts [p*Ep/n_parts, (p+1)*Ep/n_parts), i.e. one subtree.
 *
 * Partial: partial[t][o] = value of part `part`'s subtree. topk_id [n][k]: the slots' expert ids, distinct within a
 * token, in any order; token_row is read only for slots whose expert is in the part.
 */
int oracle_combine_tree_partial_f64(const float* y, const float* w, const int32_t* token_row, const int32_t* topk_id,
                                    int64_t n, int32_t top_k, int32_t hidden, int32_t n_experts, int32_t n_parts,
                                    int32_t part, double* partial);

/* Finish: the parts' values [n_parts][n][H] summed in the same tree (float64), then + s_shared[t][o] (float64),
   then ONE rounding to float32 (out_f32), then that float rounded to bf16, ties to even (out_bf16). Either output
   may be NULL; s_shared may be NULL. */
int oracle_combine_tree_finish_f64(const double* partials, int32_t n_parts, const float* s_shared, int64_t n,
                                   int32_t hidden, float* out_f32, uint16_t* out_bf16);

/*
 * Block-scaled FP8 expert weights (MXFP8): each weight is an E4M3 code (1 sign bit, 4 exponent bits with bias 7,
 * 3 fraction bits; exponent field 0 holds the subnormals m/8 * 2^-6; codes 0x7F / 0xFF are NaN, there is no
 * infinity) times the power of two 2^(s - 127) given by an E8M0 scale byte s (255 is NaN) shared by a block of 32
 * consecutive weights along K (OCP Microscaling Formats v1.0). The pages quantise prompt-tile weights (the
 * deep-prefill draft's review, "To land": NVFP4 prompt tiles that reproduce the decode bytes); this is the 8-bit
 * block-scaled member of that family.
 * codes [R][K], scales [K/32][R] (one plane per 32-wide K block), K a multiple of 32. out_bf16 [R][K]: the exact
 * value of each weight as bf16 bits. Returns -1 for a NaN code or scale, or a value that bf16 cannot hold exactly.
 */
int oracle_dequant_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K, uint16_t* out_bf16);

/*
 * Block-scaled FP4 expert weights (NVFP4, the format the deep-prefill review names for prompt tiles): each weight
 * is an E2M1 code (1 sign bit, 2 exponent bits with bias 1, 1 fraction bit; exponent field 0 holds 0 and 0.5) times
 * an E4M3 scale shared by a block of 16 consecutive weights along K. No tensor-wide scale (it is taken as 1).
 * codes [R][K/2], two codes per byte, element 2j in the low nibble of byte j, element 2j+1 in the high nibble;
 * scales [K/16][R] (one plane per 16-wide K block), K a multiple of 16. out_bf16 [R][K]: the exact value of each
 * weight as bf16 bits (a product of a 2-bit and a 4-bit significand always fits bf16 here). Returns -1 for a NaN
 * scale (0x7F / 0xFF).
 */
int oracle_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K, uint16_t* out_bf16);

#ifdef __cplusplus
}
#endif
#endif
