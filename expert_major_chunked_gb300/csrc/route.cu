// Routing of one chunk: top-k selection with weights, then the per-chunk member lists (histogram, exclusive scan,
// permutation) and the tile lists of the two grouped GEMMs. No atomics: every count and every row index is a
// function of the chunk's top-k ids alone, so the member lists are identical run to run.
//
// Umbrella PR #1113 ("Latest prefill efficiency candidate") builds per-expert member lists for each chunk on the
// host; here they are built on the device. Reading of the order (pages silent): rows of a chunk are grouped by
// ascending expert id and, inside an expert, by ascending token.
#include "internal.h"

#include <cuda_bf16.h>
#include <cfloat>
#include <algorithm>
#include <climits>

namespace moe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ double bf16d_lo(uint32_t w) { return static_cast<double>(bf16_lo(w)); }
__device__ __forceinline__ double bf16d_hi(uint32_t w) { return static_cast<double>(bf16_hi(w)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of squares of a bf16 row in fp32 (8 elements per lane per step; H is a multiple of 64). The loads of up to 8
// steps are issued before their arithmetic, so a row costs about one memory round trip, not one per step.
__device__ __forceinline__ float row_sumsq(const uint16_t* row, int H, int lane) {
  float ss = 0.0f;
  for (int i0 = lane * 8; i0 < H; i0 += 8 * 256) {
    uint4 q[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int i = i0 + 256 * m;
      q[m] = i < H ? __ldg(reinterpret_cast<const uint4*>(row + i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t w[4] = {q[m].x, q[m].y, q[m].z, q[m].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
  }
  return warp_sum(ss);
}

// Router logit in float64, summed over i ascending from 0.0: every bf16 x bf16 product is exact in double, so
// rounding only the additions reproduces the plain sequential float64 dot product bit for bit.
__device__ double exact_logit(const uint16_t* x, const uint16_t* w, int H) {
  double acc = 0.0;
  for (int i = 0; i < H; i += 8) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(x + i));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(w + i));
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc = __dadd_rn(acc, __dmul_rn(bf16d_lo(aw[j]), bf16d_lo(bw[j])));
      acc = __dadd_rn(acc, __dmul_rn(bf16d_hi(aw[j]), bf16d_hi(bw[j])));
    }
  }
  return acc;
}

// Scratch of one warp for the float64 recheck of the ambiguous places of one token.
constexpr int kMaxCand = 64;
struct BandScratch {
  double val[kMaxCand];
  double sabs[kMaxCand];
  int32_t id[kMaxCand];
  int32_t chosen[kMaxCand];
};

// bf16 -> double by bit manipulation on the integer pipe (GB300's fp64 pipe is 1/64 of fp32): exact for every bf16.
__device__ __forceinline__ double bf16_bits_to_double(uint32_t b16) {
  const uint32_t sign = b16 >> 15, ex = (b16 >> 7) & 0xFFu, man = b16 & 0x7Fu;
  if (ex == 0u) return static_cast<double>(__uint_as_float(b16 << 16));  // zero / subnormal: rare, exact cast
  if (ex == 0xFFu) return static_cast<double>(__uint_as_float(b16 << 16));
  const uint64_t bits = (static_cast<uint64_t>(sign) << 63) | (static_cast<uint64_t>(ex - 127u + 1023u) << 52) |
                        (static_cast<uint64_t>(man) << 45);
  return __longlong_as_double(static_cast<long long>(bits));
}

template <typename T>
__device__ __forceinline__ T bf16_as(uint32_t b16);
template <>
__device__ __forceinline__ float bf16_as<float>(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}
template <>
__device__ __forceinline__ double bf16_as<double>(uint32_t b16) {
  return bf16_bits_to_double(b16);
}

// Logits of the candidates in precision T (float or double), the whole warp on one candidate at a time. Lane l
// owns elements 256 m + 8 l + j (j < 8, m = 0, 1, ...); slot j keeps its own running sum over m (fused multiply-
// add of exact products), the 8 slot sums are added pairwise, then a butterfly adds the 32 lanes. Every bf16 x bf16
// product is exact in float and in double, so each value differs from the exact dot product by at most
// depth * u * S, depth = ceil(H/256) + 8 roundings on any path and S = sum |x_i w_i| (returned in B.sabs as a
// float sum, which the bound inflates by 1%). All loads of a row segment are issued before its arithmetic.
template <typename T>
__device__ void band_values(BandScratch& B, int ncand, const uint16_t* xrow, const uint16_t* w_router, int H,
                            int lane, bool with_sabs) {
  for (int c = 0; c < ncand; ++c) {
    const uint16_t* wrow = w_router + static_cast<int64_t>(B.id[c]) * H;
    T acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = T(0);
    float sab = 0.0f;
    for (int i0 = lane * 8; i0 < H; i0 += 256 * 8) {
      uint4 xa[8], wa[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int i = i0 + 256 * m;
        if (i < H) {
          xa[m] = __ldg(reinterpret_cast<const uint4*>(xrow + i));
          wa[m] = __ldg(reinterpret_cast<const uint4*>(wrow + i));
        } else {
          xa[m] = make_uint4(0, 0, 0, 0);
          wa[m] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t aw[4] = {xa[m].x, xa[m].y, xa[m].z, xa[m].w};
        const uint32_t bw[4] = {wa[m].x, wa[m].y, wa[m].z, wa[m].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const T x0 = bf16_as<T>(aw[q] & 0xFFFFu), x1 = bf16_as<T>(aw[q] >> 16);
          const T w0 = bf16_as<T>(bw[q] & 0xFFFFu), w1 = bf16_as<T>(bw[q] >> 16);
          acc[2 * q] = fma(x0, w0, acc[2 * q]);
          acc[2 * q + 1] = fma(x1, w1, acc[2 * q + 1]);
          if (with_sabs) {
            sab += fabsf(bf16_lo(aw[q]) * bf16_lo(bw[q]));
            sab += fabsf(bf16_hi(aw[q]) * bf16_hi(bw[q]));
          }
        }
      }
    }
    T v = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (with_sabs) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sab += __shfl_xor_sync(0xffffffffu, sab, o);
    }
    if (lane == 0) {
      B.val[c] = static_cast<double>(v);
      if (with_sabs) B.sabs[c] = static_cast<double>(sab) * 1.01;
    }
  }
  __syncwarp();
}

// Lane 0 only: marks the `need` best candidates by (value desc, id asc) in B.chosen. When beta >= 0 the values are
// estimates within beta of the sequential float64 sums (per candidate: beta_c = bound * S_c, bound passed in), and
// the function returns 1 only when the choice provably equals the choice on those sums: the worst chosen estimate
// beats the best unchosen one by more than twice the largest beta.
__device__ int band_select(BandScratch& B, int ncand, int need, double bound) {
  for (int c = 0; c < ncand; ++c) B.chosen[c] = 0;
  double worst_in = DBL_MAX;
  for (int r = 0; r < need; ++r) {
    int best = -1;
    for (int c = 0; c < ncand; ++c) {
      if (B.chosen[c]) continue;
      if (best < 0 || B.val[c] > B.val[best] || (B.val[c] == B.val[best] && B.id[c] < B.id[best])) best = c;
    }
    if (best < 0) break;
    B.chosen[best] = 1;
    worst_in = fmin(worst_in, B.val[best]);
  }
  if (bound < 0.0 || need <= 0 || need >= ncand) return 1;
  double best_out = -DBL_MAX, smax = 0.0;
  for (int c = 0; c < ncand; ++c) {
    smax = fmax(smax, B.sabs[c]);
    if (!B.chosen[c]) best_out = fmax(best_out, B.val[c]);
  }
  // products that underflow float contribute at most 2^-149 each: an absolute term covers them
  const double beta = bound * smax + 0x1p-140;
  return (worst_in - best_out > 2.0 * beta) ? 1 : 0;
}

__global__ void __launch_bounds__(256) router_norms_kernel(const uint16_t* w, int E, int H, float* wnorm,
                                                           WsHeader* hdr) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = blockIdx.x * 8 + warp;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->err = 0;
    hdr->band_tokens = 0;
    hdr->chunks_done = 0;
    for (int i = 0; i < 4; ++i) hdr->band_levels[i] = 0;
    hdr->experts_copied = 0;
    hdr->experts_skipped = 0;
    hdr->experts_hot = 0;
  }
  if (e >= E) return;
  const float ss = row_sumsq(w + static_cast<int64_t>(e) * H, H, lane);
  // fp32 rounding of the sum of squares is far below 1e-3 relative: the inflated value is an upper bound
  if (lane == 0) wnorm[e] = sqrtf(ss) * 1.001f;
}

// Top-k selection of one token per warp. The selection follows the float64 logits: the fp32 tensor-core logits are
// trusted only when the gap between the k-th and (k+1)-th largest exceeds twice the error bound tau; otherwise the
// token is flagged and band_kernel decides its last places (see there). Both kernels write the outputs the same way.
template <int EPL>
__device__ __forceinline__ void load_logits(const float* lrow, int E, int lane, float (&v)[EPL]) {
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    v[j] = (e < E) ? lrow[e] : -FLT_MAX;
  }
}

// A float's bits as an unsigned key with the same order (for non-NaN values; -0 is taken as +0 first, so the two
// zeros tie as they compare equal).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// (rounds) rounds of warp argmax by (value desc, id asc); marks the first k in *sel, returns the k-th and (k+1)-th.
// Each round: every lane offers its best unselected value; the warp takes the largest key (redux max), then the
// smallest id among the lanes holding it (redux min).
template <int EPL>
__device__ __forceinline__ void select_top(const float (&v)[EPL], int E, int k, int lane, uint32_t* sel, float* vk,
                                           float* vk1) {
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) key[j] = order_key(v[j]);
  uint32_t s = 0;
  float a = 0.0f, b = -FLT_MAX;
  const int rounds = (k + 1 < E) ? k + 1 : E;
  for (int r = 0; r < rounds; ++r) {
    uint32_t bk = 0;
    int bid = INT_MAX;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = j * 32 + lane;
      if (e < E && !((s >> j) & 1u) && (bid == INT_MAX || key[j] > bk)) {
        bk = key[j];
        bid = e;
      }
    }
    // lanes with nothing left offer key 0 and id INT_MAX; a real key is never 0 (it would be a NaN's)
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bid == INT_MAX ? 0u : bk);
    const int wid = static_cast<int>(
        __reduce_min_sync(0xffffffffu, (bid != INT_MAX && bk == wk) ? static_cast<uint32_t>(bid) : 0x7FFFFFFFu));
    const float wv = wid == INT_MAX ? -FLT_MAX : key_value(wk);
    if (r < k) {
      if (wid != INT_MAX && (wid & 31) == lane) s |= 1u << (wid >> 5);
      if (r == k - 1) a = wv;
    } else {
      b = wv;
    }
  }
  *sel = s;
  *vk = a;
  *vk1 = b;
}

// Ids of the selected experts in ascending order and their weights: softmax over the selected fp32 logits (equal to
// the full softmax renormalised over the selection).
template <int EPL>
__device__ __forceinline__ void write_selection(const RouteParams& p, int t, int lane, uint32_t sel,
                                                const float (&v)[EPL]) {
  const int k = p.k;
  float fmax_sel = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if ((sel >> j) & 1u) fmax_sel = fmaxf(fmax_sel, v[j]);
  fmax_sel = warp_max(fmax_sel);
  float ex[EPL];
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    ex[j] = ((sel >> j) & 1u) ? expf(v[j] - fmax_sel) : 0.0f;
    s += ex[j];
  }
  s = warp_sum(s);
  int pos = 0;
  int32_t* ids_out = p.topk_id + static_cast<int64_t>(t) * k;
  float* w_out = p.topk_w + static_cast<int64_t>(t) * k;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const bool mine = (sel >> j) & 1u;
    const uint32_t b = __ballot_sync(0xffffffffu, mine);
    if (mine) {
      const int slot = pos + __popc(b & lt);
      if (slot < k) {
        ids_out[slot] = j * 32 + lane;
        w_out[slot] = __fdiv_rn(ex[j], s);
      }
    }
    pos += __popc(b);
  }
  if (pos != k) {
    // cannot happen for finite logits; keep every slot a valid expert id so later kernels stay in bounds
    if (lane >= pos && lane < k) {
      ids_out[lane] = 0;
      w_out[lane] = 0.0f;
    }
    if (lane == 0) atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, t));
  }
}

// Candidates of a flagged token: experts whose fp32 logit lies in [v_k - 2 tau, v_{k+1} + 2 tau]. Those above the
// band are certainly among the k largest float64 logits, those below certainly not. Fills B.id in ascending id order
// (when at most kMaxCand) and returns the number of candidates; *need = places left for them.
template <int EPL>
__device__ __forceinline__ int band_candidates(const float (&v)[EPL], int E, int k, int lane, double tau, double vk,
                                               double vk1, BandScratch& B, uint32_t* sure_out, uint32_t* cand_out,
                                               int (&cidx)[EPL], int* need) {
  const double hi = vk1 + 2.0 * tau;
  const double lo = vk - 2.0 * tau;
  uint32_t sure = 0, cand = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    if (e >= E) continue;
    const double dv = static_cast<double>(v[j]);
    if (dv > hi)
      sure |= 1u << j;
    else if (dv >= lo)
      cand |= 1u << j;
  }
  *need = k - warp_sum_i(__popc(sure));
  int ncand = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const bool mine = (cand >> j) & 1u;
    const uint32_t b = __ballot_sync(0xffffffffu, mine);
    cidx[j] = ncand + __popc(b & ((1u << lane) - 1u));
    ncand += __popc(b);
  }
  if (ncand <= kMaxCand) {
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if ((cand >> j) & 1u) B.id[cidx[j]] = j * 32 + lane;
  }
  __syncwarp();
  *sure_out = sure;
  *cand_out = cand;
  return ncand;
}

template <int EPL>
__device__ __forceinline__ uint32_t chosen_mask(const BandScratch& B, uint32_t cand, const int (&cidx)[EPL]) {
  uint32_t chosen = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if (((cand >> j) & 1u) && B.chosen[cidx[j]]) chosen |= 1u << j;
  return chosen;
}

// Bounds of the band estimates: an estimate summed with tree depth d is within d u S of the exact dot product and the
// sequential float64 sum within (H - 1) u64 S of it (S = sum |x_i w_i|); 1% covers the rounding of S itself.
__device__ __forceinline__ double band_bound(int H, double u) {
  const double depth = static_cast<double>((H + 255) / 256 + 8);
  return 1.01 * (depth * u + static_cast<double>(H) * 0x1p-53);
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(RouteParams p) {
  __shared__ float wm_warp[8];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * 8 + warp;
  const int E = p.E, k = p.k, H = p.H;
  // max_e ||w_e|| once per block (every thread of the block loads a few norms at once)
  float wm = 0.0f;
  for (int e = threadIdx.x; e < E; e += 256) wm = fmaxf(wm, p.wnorm[e]);
  wm = warp_max(wm);
  if (lane == 0) wm_warp[warp] = wm;
  __syncthreads();
  wm = wm_warp[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) wm = fmaxf(wm, wm_warp[i]);
  if (t >= p.n) return;
  float v[EPL];
  load_logits(p.logits + static_cast<int64_t>(t) * E, E, lane, v);
  const uint16_t* xrow = p.x + static_cast<int64_t>(t) * H;
  const float xnorm = sqrtf(row_sumsq(xrow, H, lane)) * 1.001f;
  const double tau = static_cast<double>(p.tau_coef) * static_cast<double>(xnorm) * static_cast<double>(wm);
  uint32_t sel;
  float vk, vk1;
  select_top(v, E, k, lane, &sel, &vk, &vk1);
  int flag = 0;
  if ((k < E) && !(static_cast<double>(vk) - static_cast<double>(vk1) > 2.0 * tau)) {
    // not certain: band_kernel decides the last places of this token
    flag = 2;
    if (lane == 0) p.band_info[t] = BandInfo{tau, static_cast<double>(vk), static_cast<double>(vk1), 0.0};
  }
  if (flag != 2) write_selection(p, t, lane, sel, v);
  if (lane == 0) p.band_flag[t] = static_cast<uint8_t>(flag);
}

// Tokens whose fp32 selection was not certain (flag 2): their last places are decided on float sums of the exact
// products, then, when those cannot separate them, on double sums, and finally on the sequential float64 sums
// themselves (the reference definition, bit for bit). A grid of one CTA per SM strides over the chunk's tokens, so
// the few flagged tokens (a few percent) are spread over every SM and the top-k kernel stays light.
template <int EPL>
__global__ void __launch_bounds__(256) band_kernel(RouteParams p) {
  __shared__ BandScratch band_scratch[8];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int E = p.E, k = p.k, H = p.H;
  // the warp's tokens t0 + i * stride; their flags are read 32 at a time (one load per lane, then a ballot) instead
  // of one dependent load per token
  const int stride = gridDim.x * 8;
  for (int t0 = blockIdx.x * 8 + warp; t0 < p.n; t0 += 32 * stride) {
    const int tl = t0 + lane * stride;
    uint32_t todo = __ballot_sync(0xffffffffu, tl < p.n && p.band_flag[tl] == 2);
    while (todo != 0u) {
      const int t = t0 + (__ffs(todo) - 1) * stride;
      todo &= todo - 1u;
      float v[EPL];
      load_logits(p.logits + static_cast<int64_t>(t) * E, E, lane, v);
      const uint16_t* xrow = p.x + static_cast<int64_t>(t) * H;
      const BandInfo bi = p.band_info[t];
      BandScratch& B = band_scratch[warp];
      uint32_t sure, cand;
      int cidx[EPL];
      int need;
      const int ncand = band_candidates(v, E, k, lane, bi.tau, bi.vk, bi.vk1, B, &sure, &cand, cidx, &need);
      uint32_t chosen = 0;
      if (ncand <= kMaxCand) {
        // level 0: float sums of the exact products (also S for every level's bound)
        band_values<float>(B, ncand, xrow, p.w_router, H, lane, true);
        int certified = 0;
        if (lane == 0) certified = band_select(B, ncand, need, band_bound(H, 0x1p-24));
        certified = __shfl_sync(0xffffffffu, certified, 0);
        int level = 0;
        if (!certified) {
          // level 1: double sums
          level = 1;
          band_values<double>(B, ncand, xrow, p.w_router, H, lane, false);
          if (lane == 0) certified = band_select(B, ncand, need, band_bound(H, 0x1p-53));
          certified = __shfl_sync(0xffffffffu, certified, 0);
        }
        if (!certified) {
          level = 2;
          for (int c = lane; c < ncand; c += 32)
            B.val[c] = exact_logit(xrow, p.w_router + static_cast<int64_t>(B.id[c]) * H, H);
          __syncwarp();
          if (lane == 0) band_select(B, ncand, need, -1.0);
        }
        __syncwarp();
        if (lane == 0) atomicAdd(&p.hdr->band_levels[level], 1);  // diagnostic counter only
        chosen = chosen_mask(B, cand, cidx);
      } else {
        // more candidates than the scratch list holds (e.g. all-zero tokens): sequential float64 sums per lane
        if (lane == 0) atomicAdd(&p.hdr->band_levels[3], 1);  // diagnostic counter only
        double d[EPL];
  #pragma unroll
        for (int j = 0; j < EPL; ++j) {
          d[j] = 0.0;
          if ((cand >> j) & 1u) d[j] = exact_logit(xrow, p.w_router + static_cast<int64_t>(j * 32 + lane) * H, H);
        }
        for (int r = 0; r < need; ++r) {
          double bv = -DBL_MAX;
          int bid = INT_MAX;
  #pragma unroll
          for (int j = 0; j < EPL; ++j) {
            if (((cand & ~chosen) >> j) & 1u) {
              if (bid == INT_MAX || d[j] > bv) {
                bv = d[j];
                bid = j * 32 + lane;
              }
            }
          }
  #pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
            if (ov > bv || (ov == bv && oid < bid)) {
              bv = ov;
              bid = oid;
            }
          }
          if (bid != INT_MAX && (bid & 31) == lane) chosen |= 1u << (bid >> 5);
        }
      }
      write_selection(p, t, lane, sure | chosen, v);
      __syncwarp();
    }
  }
}

// Histogram of 32-token blocks, one warp per block: for every expert, the bit mask of the block's tokens that
// selected it. Slot by slot, __match_any_sync groups the lanes (tokens) that picked the same expert and the
// group's lowest lane ORs the group into that expert's mask; the experts of one slot are distinct writers, so the
// masks need no atomics and do not depend on timing.
constexpr int kCountWarps = 8;
__global__ void __launch_bounds__(kCountWarps * 32) count_kernel(PermuteParams p) {
  extern __shared__ uint32_t cmask[];  // [kCountWarps][E]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int E = p.E, k = p.k;
  const int b = blockIdx.x * kCountWarps + warp;
  if (b >= p.nblk) return;
  uint32_t* m = cmask + warp * E;
  for (int e = lane; e < E; e += 32) m[e] = 0;
  __syncwarp();
  const int t = b * 32 + lane;
  const bool valid = t < p.n;
  for (int s = 0; s < k; ++s) {
    int e = valid ? p.topk_id[static_cast<int64_t>(t) * k + s] : -1;
    if (e >= E) e = -1;
    const uint32_t g = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(g) - 1) m[e] |= g;
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) {
    const uint32_t v = m[e];
    p.masks[static_cast<int64_t>(b) * E + e] = v;
    p.counts[static_cast<int64_t>(b) * E + e] = __popc(v);
  }
  const uint32_t bb = __ballot_sync(0xffffffffu, valid && p.band_flag[valid ? t : 0] != 0);
  if (lane == 0) p.block_band[b] = __popc(bb);
}

// Exclusive scan across the block (blockDim.x a multiple of 32, at most 1024); returns the thread's exclusive prefix,
// *total gets the sum.
__device__ int block_exclusive_scan(int v, int* total, int* smem32) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nwarps = blockDim.x / 32;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) smem32[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < nwarps ? smem32[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    smem32[lane] = wi - ws;  // exclusive prefix of warp sums
    if (lane == 31) smem32[32] = wi;
  }
  __syncthreads();
  const int r = incl - v + smem32[warp];
  *total = smem32[32];
  __syncthreads();
  return r;
}

// Per expert, its total rows in the chunk and, for every 32-token block, the rows of that expert in the blocks before
// it (the block's base relative to the expert's first row). ceil(E/32) CTAs of 1024 threads: lane l handles expert
// 32 x CTA + l (consecutive experts: the counts rows load coalesced), warp w the w-th of 32 contiguous ranges of
// blocks; the 32 range sums of an expert meet in shared memory. Each thread walks at most ceil(nblk / 32) blocks.
constexpr int kBaseWarps = 32;
__global__ void __launch_bounds__(kBaseWarps * 32) block_bases_kernel(PermuteParams p) {
  __shared__ int part[kBaseWarps][33];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = blockIdx.x * 32 + lane;
  const int E = p.E, nblk = p.nblk;
  const int per = (nblk + kBaseWarps - 1) / kBaseWarps;
  const int b0 = min(nblk, warp * per), b1 = min(nblk, b0 + per);
  int sum = 0;
  if (e < E) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) sum += p.counts[static_cast<int64_t>(b) * E + e];
  }
  part[warp][lane] = sum;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += part[w][lane];
  if (e < E) {
    if (warp == kBaseWarps - 1) p.totals[e] = before + sum;
    int run = before;
    for (int b = b0; b < b1; ++b) {
      const int64_t be = static_cast<int64_t>(b) * E + e;
      const int c = p.counts[be];
      p.base[be] = run;
      run += c;
    }
  }
}

// One CTA of 512 threads; thread i owns expert i and, when E > 512, expert i + 512: expert offsets (an exclusive
// scan of the totals block_bases_kernel left), and the tile lists of the gate/up and down GEMMs (expert-major:
// expert, then N tile, then M tile; or, for grouped_pair_kernel, expert, then weight block, then token tile of
// pair_tile_width rows). 512 threads of at most 64 registers leave room on an SM for a GEMM CTA beside it: this
// kernel runs while the previous chunk's GEMMs hold every SM.
constexpr int kScanThreads = 512;

// Row tiles of an expert with `rows` member rows: 128-row tiles (grouped_gemm_kernel) or pair_tile_width-row tiles
// (grouped_pair_kernel).
__device__ __forceinline__ int row_tiles(int rows, int pair) {
  return pair ? pair_tile_count(rows) : (rows + kBlockM - 1) / kBlockM;
}
__device__ __forceinline__ int row_tile_width(int rows, int pair) { return pair ? pair_tile_width(rows) : kBlockM; }

__global__ void __launch_bounds__(kScanThreads, 2) scan_tiles_kernel(PermuteParams p) {
  __shared__ int sm[33];
  const int E = p.E, nblk = p.nblk;
  const int halves = (E + kScanThreads - 1) / kScanThreads;  // 1, or 2 for E > 512
  int tot[2] = {0, 0}, off[2] = {0, 0}, gu_base[2] = {0, 0}, dn_base[2] = {0, 0};
  int R = 0, n_gu = 0, n_dn = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (h >= halves) break;
    const int e = static_cast<int>(threadIdx.x) + h * kScanThreads;
    if (e < E) tot[h] = p.totals[e];
    // exclusive scans over the experts of this half, after those of the half before
    int sum = 0;
    off[h] = R + block_exclusive_scan(tot[h], &sum, sm);
    R += sum;
    const int mt_gu = (e < E) ? row_tiles(tot[h], p.pair_gu) : 0;
    const int mt_dn = (e < E) ? row_tiles(tot[h], p.pair_dn) : 0;
    gu_base[h] = n_gu + block_exclusive_scan(mt_gu * p.nt_gu, &sum, sm);
    n_gu += sum;
    dn_base[h] = n_dn + block_exclusive_scan(mt_dn * p.nt_down, &sum, sm);
    n_dn += sum;
  }
  if (threadIdx.x == 0) {
    p.offsets[E] = R;
    if (p.offsets_out) p.offsets_out[E] = R;
    p.tile_base[E] = n_gu;
    p.tile_base[E + 1 + E] = n_dn;
  }
  const int mts_gu = row_tiles(p.n, p.pair_gu), mts_dn = row_tiles(p.n, p.pair_dn);
  const int swid_gu = row_tile_width(p.n, p.pair_gu), swid_dn = row_tile_width(p.n, p.pair_dn);
  const int n_gu_all = n_gu + (p.nt_gu_shared > 0 ? mts_gu * p.nt_gu_shared : 0);
  const int n_dn_all = n_dn + (p.nt_down_shared > 0 ? mts_dn * p.nt_down_shared : 0);
  const bool fits = n_gu_all <= p.cap_gu && n_dn_all <= p.cap_down;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = static_cast<int>(threadIdx.x) + h * kScanThreads;
    if (h >= halves || e >= E) continue;
    p.offsets[e] = off[h];
    if (p.offsets_out) p.offsets_out[e] = off[h];
    p.tile_base[e] = gu_base[h];
    p.tile_base[E + 1 + e] = dn_base[h];
    if (!fits) continue;
    // an expert with a single row tile is the only reader of its weight tiles: mark them for streaming
    {
      const int mt = row_tiles(tot[h], p.pair_gu), wid = row_tile_width(tot[h], p.pair_gu);
      const int stream = (mt == 1) ? static_cast<int>(1u << 31) : 0;
      for (int nn = 0; nn < p.nt_gu; ++nn)
        for (int m = 0; m < mt; ++m)
          p.tiles_gu[gu_base[h] + nn * mt + m] =
              make_int4(e | (nn << 16) | stream, off[h] + m * wid, min(wid, tot[h] - m * wid), off[h] + m * wid);
    }
    {
      const int mt = row_tiles(tot[h], p.pair_dn), wid = row_tile_width(tot[h], p.pair_dn);
      const int stream = (mt == 1) ? static_cast<int>(1u << 31) : 0;
      for (int nn = 0; nn < p.nt_down; ++nn)
        for (int m = 0; m < mt; ++m)
          p.tiles_down[dn_base[h] + nn * mt + m] =
              make_int4(e | (nn << 16) | stream, off[h] + m * wid, min(wid, tot[h] - m * wid), off[h] + m * wid);
    }
  }
  if (fits) {
    // shared expert (class 1): gate/up reads the chunk's rows of X, down reads the shared h rows
    for (int i = threadIdx.x; i < mts_gu * p.nt_gu_shared; i += blockDim.x) {
      const int nn = i / mts_gu, m = i % mts_gu;
      p.tiles_gu[n_gu + i] = make_int4((1 << 15) | (nn << 16), static_cast<int>(p.token0) + m * swid_gu,
                                       min(swid_gu, p.n - m * swid_gu), m * swid_gu);
    }
    for (int i = threadIdx.x; i < mts_dn * p.nt_down_shared; i += blockDim.x) {
      const int nn = i / mts_dn, m = i % mts_dn;
      p.tiles_down[n_dn + i] =
          make_int4((1 << 15) | (nn << 16), m * swid_dn, min(swid_dn, p.n - m * swid_dn), m * swid_dn);
    }
  }
  if (threadIdx.x == 0) {
    p.num_tiles[0] = fits ? n_gu_all : 0;
    p.num_tiles[1] = fits ? n_dn_all : 0;
    if (!fits) atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, 0));
    p.hdr->chunks_done += 1;
  }
  int nb_band = 0;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) nb_band += p.block_band[b];
  int band_total = 0;
  (void)block_exclusive_scan(nb_band, &band_total, sm);
  if (threadIdx.x == 0) p.hdr->band_tokens += band_total;
}

// Row index of every (token, slot), the inverse map, and the gathered copy of X in expert-major row order.
// One warp per token: lane s < k computes the row of slot s from the block's row base of its expert plus the
// number of earlier tokens of the block that selected the same expert (popcount of the mask below the token).
constexpr int kPermuteWarps = 8;
__global__ void __launch_bounds__(kPermuteWarps * 32) permute_kernel(PermuteParams p) {
  __shared__ int32_t rows_sm[kPermuteWarps][32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * kPermuteWarps + warp;
  if (t >= p.n) return;
  const int k = p.k, E = p.E, H = p.H;
  const int b = t >> 5, i = t & 31;
  if (lane < k) {
    int e = p.topk_id[static_cast<int64_t>(t) * k + lane];
    if (e < 0 || e >= E) {
      atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, t));
      e = 0;
    }
    const int64_t be = static_cast<int64_t>(b) * E + e;
    int row = p.offsets[e] + p.base[be] + __popc(p.masks[be] & ((1u << i) - 1u));
    if (row < 0 || row >= p.n * k) {
      atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, t));
      row = 0;
    }
    rows_sm[warp][lane] = row;
    p.token_row[static_cast<int64_t>(t) * k + lane] = row;
    if (p.row_token) p.row_token[row] = static_cast<int32_t>(p.token0 + t);
  }
  __syncwarp();
  const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(t) * H);
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 val = __ldg(src + c);
    for (int s = 0; s < k; ++s) reinterpret_cast<uint4*>(p.xp + static_cast<int64_t>(rows_sm[warp][s]) * H)[c] = val;
  }
}

}  // namespace

cudaError_t launch_router_norms(const uint16_t* w_router, int E, int H, float* wnorm, WsHeader* hdr,
                                cudaStream_t stream) {
  router_norms_kernel<<<(E + 7) / 8, 256, 0, stream>>>(w_router, E, H, wnorm, hdr);
  return cudaGetLastError();
}

template <int EPL>
cudaError_t launch_topk_epl(const RouteParams& p, int grid, cudaStream_t stream) {
  topk_kernel<EPL><<<grid, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  band_kernel<EPL><<<std::min(grid, p.band_grid), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_topk(const RouteParams& p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  const int grid = (p.n + 7) / 8;
  const int epl = (p.E + 31) / 32;
  if (epl <= 1) return launch_topk_epl<1>(p, grid, stream);
  if (epl <= 2) return launch_topk_epl<2>(p, grid, stream);
  if (epl <= 4) return launch_topk_epl<4>(p, grid, stream);
  if (epl <= 8) return launch_topk_epl<8>(p, grid, stream);
  if (epl <= 16) return launch_topk_epl<16>(p, grid, stream);
  return launch_topk_epl<32>(p, grid, stream);
}

cudaError_t launch_count(const PermuteParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kCountWarps) * p.E * sizeof(uint32_t);
  count_kernel<<<(p.nblk + kCountWarps - 1) / kCountWarps, kCountWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_block_bases(const PermuteParams& p, cudaStream_t stream) {
  block_bases_kernel<<<(p.E + 31) / 32, kBaseWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scan_tiles(const PermuteParams& p, cudaStream_t stream) {
  scan_tiles_kernel<<<1, kScanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t stream) {
  permute_kernel<<<(p.n + kPermuteWarps - 1) / kPermuteWarps, kPermuteWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
