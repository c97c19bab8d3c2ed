/*
 * Reference oracle for the expert-major chunked MoE prefill layer (float64, CPU). TEST INFRASTRUCTURE ONLY.
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC (no contraction, IEEE order).
 * Page references use the tags defined in oracle.h.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * Plainest reading for every BF16 store of the layer ("BF16 layer"): round to nearest, ties to even, straight from
 * the exact value. |v| lies in [2^(e-1), 2^e) with e from frexp; a bf16 normal number there has 8 significant bits,
 * so its spacing is 2^(e-8); below the smallest normal 2^-126 the spacing is fixed at 2^-133. Dividing by a power of
 * two is exact, rint() rounds ties to even, and the rounded value is exactly representable in float, whose top 16
 * bits are the bf16 pattern.
 */
uint16_t oracle_bf16_from_double(double v) {
  if (isnan(v)) return (uint16_t)0x7FC0;
  uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  (void)frexp(a, &e);
  int qexp = e - 8;
  if (qexp < -133) qexp = -133;
  double q = ldexp(1.0, qexp);
  double r = rint(a / q) * q;
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80); /* rounds past the largest bf16: infinity */
  float f = (float)r;                                          /* exact */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

int oracle_bf16_round_array(const double* in, uint16_t* out, int64_t n) {
  if (!in || !out || n < 0) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_double(in[i]);
  return 0;
}

static double bf(const uint16_t* p, int64_t i) { return oracle_bf16_to_double(p[i]); }

/*
 * Router logits. [UMB] "What it adds" / "Memory and execution split": routed experts 0..E-1 chosen per token by a
 * router on the dense side; the pages give no router formula. Plainest reading: a bias-free linear router,
 * l[t][e] = <x_t, w_e>, summed in float64 over i ascending from 0.0 (each bf16 x bf16 product is exact in double).
 */
static double router_logit(const uint16_t* x_row, const uint16_t* w_row, int32_t H) {
  double acc = 0.0;
  for (int32_t i = 0; i < H; ++i) acc += bf(x_row, i) * bf(w_row, i);
  return acc;
}

int oracle_router_logits(const uint16_t* x, const uint16_t* w_router, int64_t n_tokens, int32_t hidden,
                         int32_t n_experts, double* logits) {
  if (!x || !w_router || !logits || n_tokens < 0 || hidden <= 0 || n_experts <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_tokens; ++t)
    for (int32_t e = 0; e < n_experts; ++e)
      logits[t * n_experts + e] = router_logit(x + t * (int64_t)hidden, w_router + (int64_t)e * hidden, hidden);
  return 0;
}

/*
 * Top-k selection and weights for one token. The pages only say "routed experts" with per-expert member lists
 * ([UMB] "Latest prefill efficiency candidate"); plainest reading: the k largest logits, an exact tie going to the
 * lower expert id; the weights are the softmax of the selected logits, i.e. the full softmax renormalised over the
 * selected experts. Selected ids are listed in ascending id order, which is the order the canonical reduction of
 * [DP-c] (introduction: "canonical routed-expert reduction") walks.
 */
static void topk_one(const double* l, int32_t E, int32_t k, unsigned char* chosen, int32_t* ids, double* w) {
  memset(chosen, 0, (size_t)E);
  for (int32_t s = 0; s < k; ++s) {
    int32_t best = -1;
    for (int32_t e = 0; e < E; ++e) {
      if (chosen[e]) continue;
      if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower id on an exact tie */
    }
    chosen[best] = 1;
  }
  int32_t j = 0;
  for (int32_t e = 0; e < E; ++e)
    if (chosen[e]) ids[j++] = e;
  double lmax = l[ids[0]];
  for (int32_t s = 1; s < k; ++s)
    if (l[ids[s]] > lmax) lmax = l[ids[s]];
  double denom = 0.0;
  for (int32_t s = 0; s < k; ++s) denom += exp(l[ids[s]] - lmax);
  for (int32_t s = 0; s < k; ++s) w[s] = exp(l[ids[s]] - lmax) / denom;
}

int oracle_topk(const double* logits, int64_t n_tokens, int32_t n_experts, int32_t top_k, int32_t* topk_id,
                double* topk_w) {
  if (!logits || !topk_id || !topk_w || n_tokens < 0 || n_experts <= 0 || top_k < 1 || top_k > n_experts) return -1;
#pragma omp parallel
  {
    unsigned char* chosen = (unsigned char*)malloc((size_t)n_experts);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < n_tokens; ++t)
      topk_one(logits + t * n_experts, n_experts, top_k, chosen, topk_id + t * top_k, topk_w + t * top_k);
    free(chosen);
  }
  return 0;
}

/*
 * One SwiGLU expert. [DP-a] maintainer review names the two expert kernels, a gate/up projection ("gu") and a down
 * projection; [DP-c] "Independent numerical-phase audit" says the gate/up kernel writes complete scratch bytes that
 * the down kernel reads. Plainest reading for a BF16 layer: g = x.Wg^T, u = x.Wu^T with the gate rows first in the
 * fused [2I][H] matrix, h = silu(g)*u stored as BF16 (the one storage rounding between the two projections),
 * y = h.Wd^T kept unrounded. silu(z) = z / (1 + exp(-z)).
 */
int oracle_swiglu_ffn(const uint16_t* x_row, const uint16_t* w_gu, const uint16_t* w_down, int32_t hidden,
                      int32_t inter, double* y, uint16_t* h_bf16) {
  if (!x_row || !w_gu || !w_down || !y || hidden <= 0 || inter <= 0) return -1;
  double* h = (double*)malloc(sizeof(double) * (size_t)inter);
  if (!h) return -1;
  for (int32_t j = 0; j < inter; ++j) {
    double g = 0.0, u = 0.0;
    const uint16_t* wg = w_gu + (int64_t)j * hidden;
    const uint16_t* wu = w_gu + (int64_t)(inter + j) * hidden;
    for (int32_t i = 0; i < hidden; ++i) g += bf(x_row, i) * bf(wg, i);
    for (int32_t i = 0; i < hidden; ++i) u += bf(x_row, i) * bf(wu, i);
    double silu = g / (1.0 + exp(-g));
    uint16_t hb = oracle_bf16_from_double(silu * u);
    if (h_bf16) h_bf16[j] = hb;
    h[j] = oracle_bf16_to_double(hb);
  }
  for (int32_t o = 0; o < hidden; ++o) {
    double acc = 0.0;
    const uint16_t* wd = w_down + (int64_t)o * inter;
    for (int32_t j = 0; j < inter; ++j) acc += h[j] * bf(wd, j);
    y[o] = acc;
  }
  free(h);
  return 0;
}

/*
 * The whole layer for one token. [DP-c] introduction: the routed-expert contributions of a token are reduced in one
 * canonical order so that every row is independent of the chunk size; [UMB] "Memory and execution split": the
 * shared expert is resident and indexed after the routed experts. Plainest reading: acc = 0; for the selected
 * experts in ascending id order acc += w_s * y_s; then acc += y_shared (ungated, weight 1); out = bf16(acc).
 */
int oracle_moe_forward(const oracle_dims* d, const uint16_t* x, const uint16_t* w_router, const uint16_t* w_gu,
                       const uint16_t* w_down, const uint16_t* ws_gu, const uint16_t* ws_down, int64_t n_tokens,
                       const int64_t* token_idx, int64_t n_eval, double* out_ref, uint16_t* out_bf16,
                       int32_t* topk_id, double* topk_w) {
  if (!d || !x || !w_router || !w_gu || !w_down || n_tokens < 0 || n_eval < 0) return -1;
  const int32_t H = d->hidden, E = d->n_experts, I = d->inter, k = d->top_k, Is = d->shared_inter;
  if (H <= 0 || E <= 0 || I <= 0 || k < 1 || k > E || Is < 0) return -1;
  if (Is > 0 && (!ws_gu || !ws_down)) return -1;
  if (!token_idx && n_eval != n_tokens) return -1;
  for (int64_t j = 0; token_idx && j < n_eval; ++j)
    if (token_idx[j] < 0 || token_idx[j] >= n_tokens) return -1;
  int bad = 0;
#pragma omp parallel
  {
    double* l = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* chosen = (unsigned char*)malloc((size_t)E);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!l || !chosen || !ids || !w || !y || !acc) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_eval; ++j) {
      if (bad) continue;
      const int64_t t = token_idx ? token_idx[j] : j;
      const uint16_t* xr = x + t * H;
      for (int32_t e = 0; e < E; ++e) l[e] = router_logit(xr, w_router + (int64_t)e * H, H);
      topk_one(l, E, k, chosen, ids, w);
      for (int32_t o = 0; o < H; ++o) acc[o] = 0.0;
      for (int32_t s = 0; s < k; ++s) {
        const int64_t e = ids[s];
        oracle_swiglu_ffn(xr, w_gu + e * 2 * I * (int64_t)H, w_down + e * (int64_t)H * I, H, I, y, NULL);
        for (int32_t o = 0; o < H; ++o) acc[o] += w[s] * y[o];
      }
      if (Is > 0) {
        oracle_swiglu_ffn(xr, ws_gu, ws_down, H, Is, y, NULL);
        for (int32_t o = 0; o < H; ++o) acc[o] += y[o];
      }
      for (int32_t o = 0; o < H; ++o) {
        if (out_ref) out_ref[j * H + o] = acc[o];
        if (out_bf16) out_bf16[j * H + o] = oracle_bf16_from_double(acc[o]);
      }
      for (int32_t s = 0; s < k; ++s) {
        if (topk_id) topk_id[j * k + s] = ids[s];
        if (topk_w) topk_w[j * k + s] = w[s];
      }
    }
    free(l); free(chosen); free(ids); free(w); free(y); free(acc);
  }
  return bad ? -1 : 0;
}

/*
 * Member lists. [DP-c] introduction: "expert-major deep-prefill chunks"; [UMB] "Latest prefill efficiency
 * candidate": per-expert member lists are built for each chunk. Plainest reading: a chunk covers consecutive tokens;
 * its (token, slot) pairs are grouped by expert in ascending id order and, within an expert, by ascending token
 * (a stable counting sort). Offsets and rows are local to the chunk; row_token holds global token ids.
 */
int oracle_permutation(const int32_t* topk_id, int64_t n_tokens, int32_t top_k, int32_t n_experts, int32_t chunk,
                       int32_t* expert_offsets, int32_t* row_token, int32_t* token_row) {
  if (!topk_id || n_tokens < 0 || top_k < 1 || n_experts < 1 || chunk < 1) return -1;
  const int64_t n_chunks = (n_tokens + chunk - 1) / chunk;
  int32_t* count = (int32_t*)calloc((size_t)n_experts, sizeof(int32_t));
  int32_t* next = (int32_t*)calloc((size_t)n_experts, sizeof(int32_t));
  if (!count || !next) { free(count); free(next); return -1; }
  int rc = 0;
  for (int64_t c = 0; c < n_chunks && rc == 0; ++c) {
    const int64_t t0 = c * chunk;
    const int64_t t1 = (t0 + chunk < n_tokens) ? t0 + chunk : n_tokens;
    memset(count, 0, sizeof(int32_t) * (size_t)n_experts);
    for (int64_t t = t0; t < t1; ++t)
      for (int32_t s = 0; s < top_k; ++s) {
        int32_t e = topk_id[t * top_k + s];
        if (e < 0 || e >= n_experts) { rc = -1; break; }
        count[e] += 1;
      }
    if (rc) break;
    int32_t run = 0;
    for (int32_t e = 0; e < n_experts; ++e) {
      if (expert_offsets) expert_offsets[c * (n_experts + 1) + e] = run;
      next[e] = run;
      run += count[e];
    }
    if (expert_offsets) expert_offsets[c * (n_experts + 1) + n_experts] = run;
    for (int32_t e = 0; e < n_experts; ++e)
      for (int64_t t = t0; t < t1; ++t)
        for (int32_t s = 0; s < top_k; ++s)
          if (topk_id[t * top_k + s] == e) {
            int32_t row = next[e]++;
            if (row_token) row_token[t0 * top_k + row] = (int32_t)t;
            if (token_row) token_row[t * top_k + s] = row;
          }
  }
  free(count);
  free(next);
  return rc;
}

/* Weighted combine in float64 (the tolerance reference for the float32 reduction). */
int oracle_combine_f64(const float* y, const float* w, const int32_t* token_row, const float* s_shared, int64_t n,
                       int32_t top_k, int32_t hidden, double* out_ref, uint16_t* out_bf16) {
  if (!y || !w || !token_row || n < 0 || top_k < 1 || hidden < 1) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t)
    for (int32_t o = 0; o < hidden; ++o) {
      double acc = 0.0;
      for (int32_t s = 0; s < top_k; ++s)
        acc += (double)w[t * top_k + s] * (double)y[(int64_t)token_row[t * top_k + s] * hidden + o];
      if (s_shared) acc += (double)s_shared[t * hidden + o];
      if (out_ref) out_ref[t * hidden + o] = acc;
      if (out_bf16) out_bf16[t * hidden + o] = oracle_bf16_from_double(acc);
    }
  return 0;
}

/*
 * The canonical reduction as a float32 computation. [DP-c] introduction: one canonical, fixed-order reduction of the
 * routed contributions makes the rows independent of the chunk size; [DP-b] "Checklist": no precision traded for
 * speed, and a changed summation is named. Reading: float32 accumulation from +0.0f, slots in ascending expert id,
 * each product and each sum rounded to float32, the shared expert added last, one final BF16 rounding.
 */
int oracle_combine_f32_canonical(const float* y, const float* w, const int32_t* token_row, const float* s_shared,
                                 int64_t n, int32_t top_k, int32_t hidden, uint16_t* out_bf16) {
  if (!y || !w || !token_row || !out_bf16 || n < 0 || top_k < 1 || hidden < 1) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t)
    for (int32_t o = 0; o < hidden; ++o) {
      volatile float acc = 0.0f;
      for (int32_t s = 0; s < top_k; ++s) {
        volatile float prod = w[t * top_k + s] * y[(int64_t)token_row[t * top_k + s] * hidden + o];
        acc = acc + prod;
      }
      if (s_shared) acc = acc + s_shared[t * hidden + o];
      out_bf16[t * hidden + o] = oracle_bf16_from_double((double)acc);
    }
  return 0;
}

/*
 * Expert-parallel combine with float64 partials. [DP-b] "What this changes": the tensor-parallel prefill partials
 * are float64; "Checklist": they are summed in float64 and rounded once, to float32, at the finish, so a two-GPU
 * split reproduces the one-GPU sum. The pages leave the order inside a partial open. Reading: a complete binary
 * tree over the expert ids, evaluated densely here (every expert a leaf, +0.0 where the token has no slot), so that
 * each aligned block of ids is a subtree and a split into such blocks changes no operation.
 */
static double tree_sum_f64(const double* v, int64_t len) {
  if (len == 1) return v[0];
  const double left = tree_sum_f64(v, len / 2);
  const double right = tree_sum_f64(v + len / 2, len / 2);
  return left + right;
}

static int32_t least_pow2_at_least(int32_t v) {
  int32_t p = 1;
  while (p < v) p *= 2;
  return p;
}

static int is_pow2(int32_t v) { return v > 0 && (v & (v - 1)) == 0; }

int oracle_combine_tree_partial_f64(const float* y, const float* w, const int32_t* token_row, const int32_t* topk_id,
                                    int64_t n, int32_t top_k, int32_t hidden, int32_t n_experts, int32_t n_parts,
                                    int32_t part, double* partial) {
  if (!w || !topk_id || !partial || n < 0 || top_k < 1 || hidden < 1 || n_experts < 1) return -1;
  const int32_t Ep = least_pow2_at_least(n_experts);
  if (!is_pow2(n_parts) || n_parts > Ep || part < 0 || part >= n_parts) return -1;
  const int32_t block = Ep / n_parts;
  const int32_t lo = part * block;
  for (int64_t i = 0; i < n * top_k; ++i)
    if (topk_id[i] < 0 || topk_id[i] >= n_experts) return -1;
  for (int64_t t = 0; t < n; ++t)
    for (int32_t a = 0; a < top_k; ++a)
      for (int32_t b = a + 1; b < top_k; ++b)
        if (topk_id[t * top_k + a] == topk_id[t * top_k + b]) return -1;
  if (n > 0 && !y && block > 0) {
    for (int64_t i = 0; i < n * top_k; ++i)
      if (topk_id[i] >= lo && topk_id[i] < lo + block) return -1;
  }
  int rc = 0;
#pragma omp parallel
  {
    double* leaves = (double*)malloc(sizeof(double) * (size_t)block);
    if (!leaves) {
#pragma omp atomic write
      rc = -1;
    }
#pragma omp for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
      if (!leaves) continue;
      for (int32_t o = 0; o < hidden; ++o) {
        for (int32_t e = 0; e < block; ++e) leaves[e] = 0.0;
        for (int32_t s = 0; s < top_k; ++s) {
          const int32_t e = topk_id[t * top_k + s];
          if (e < lo || e >= lo + block) continue;
          const int64_t row = token_row[t * top_k + s];
          leaves[e - lo] = (double)w[t * top_k + s] * (double)y[row * hidden + o];
        }
        partial[t * hidden + o] = tree_sum_f64(leaves, block);
      }
    }
    free(leaves);
  }
  return rc;
}

int oracle_combine_tree_finish_f64(const double* partials, int32_t n_parts, const float* s_shared, int64_t n,
                                   int32_t hidden, float* out_f32, uint16_t* out_bf16) {
  if (!partials || !is_pow2(n_parts) || n < 0 || hidden < 1) return -1;
  const int64_t plane = n * hidden;
  int rc = 0;
#pragma omp parallel
  {
    double* parts = (double*)malloc(sizeof(double) * (size_t)n_parts);
    if (!parts) {
#pragma omp atomic write
      rc = -1;
    }
#pragma omp for schedule(static)
    for (int64_t i = 0; i < plane; ++i) {
      if (!parts) continue;
      for (int32_t p = 0; p < n_parts; ++p) parts[p] = partials[p * plane + i];
      double v = tree_sum_f64(parts, n_parts);
      if (s_shared) v = v + (double)s_shared[i];
      const float f = (float)v;
      if (out_f32) out_f32[i] = f;
      if (out_bf16) out_bf16[i] = oracle_bf16_from_double((double)f);
    }
    free(parts);
  }
  return rc;
}

/* E4M3 code -> exact value, from the format's definition (sign, 4-bit exponent with bias 7, 3-bit fraction). */
static int e4m3_value(uint8_t code, double* v) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return -1; /* NaN */
  const double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  *v = sign ? -mag : mag;
  return 0;
}

int oracle_dequant_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K, uint16_t* out_bf16) {
  if (!codes || !scales || !out_bf16 || rows < 0 || K < 0 || K % 32 != 0) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t s = scales[(k / 32) * rows + r];
      if (s == 255) return -1;
      double v;
      if (e4m3_value(codes[r * K + k], &v) != 0) return -1;
      v = ldexp(v, (int)s - 127);
      const uint16_t b = oracle_bf16_from_double(v);
      if (oracle_bf16_to_double(b) != v) return -1; /* not exactly representable in bf16 */
      if (v == 0.0 && signbit(v) != ((b >> 15) & 1)) return -1;
      out_bf16[r * K + k] = b;
    }
  return 0;
}

/* E2M1 code (low 4 bits) -> exact value: sign, 2-bit exponent with bias 1, 1-bit fraction; exponent 0 gives m/2. */
static double e2m1_value(uint8_t nib) {
  const int sign = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  const double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -mag : mag;
}

int oracle_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K, uint16_t* out_bf16) {
  if (!codes || !scales || !out_bf16 || rows < 0 || K < 0 || K % 16 != 0) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      double sv;
      if (e4m3_value(scales[(k / 16) * rows + r], &sv) != 0) return -1;
      const uint8_t byte = codes[r * (K / 2) + k / 2];
      const double v = e2m1_value((k % 2 == 0) ? (byte & 15) : (byte >> 4)) * sv;
      const uint16_t b = oracle_bf16_from_double(v);
      if (oracle_bf16_to_double(b) != v) return -1;
      if (v == 0.0 && signbit(v) != ((b >> 15) & 1)) return -1;
      out_bf16[r * K + k] = b;
    }
  return 0;
}
