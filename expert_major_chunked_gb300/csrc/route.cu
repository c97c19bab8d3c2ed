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

// Sum of squares of a bf16 row in fp32 (8 elements per lane per step; H is a multiple of 64).
__device__ __forceinline__ float row_sumsq(const uint16_t* row, int H, int lane) {
  float ss = 0.0f;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + i));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
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

__global__ void __launch_bounds__(256) router_norms_kernel(const uint16_t* w, int E, int H, float* wnorm,
                                                           WsHeader* hdr) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = blockIdx.x * 8 + warp;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->err = 0;
    hdr->band_tokens = 0;
    hdr->chunks_done = 0;
  }
  if (e >= E) return;
  const float ss = row_sumsq(w + static_cast<int64_t>(e) * H, H, lane);
  // fp32 rounding of the sum of squares is far below 1e-3 relative: the inflated value is an upper bound
  if (lane == 0) wnorm[e] = sqrtf(ss) * 1.001f;
}

// Top-k of one token per warp. Selection follows the float64 logits: the fp32 tensor-core logits are trusted only
// when the gap between the k-th and (k+1)-th value exceeds twice the error bound tau; otherwise the experts inside
// the ambiguity band are recomputed in float64 (the same sum the CPU reference uses) and decide the last places.
template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(RouteParams p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * 8 + warp;
  if (t >= p.n) return;
  const int E = p.E, k = p.k, H = p.H;
  const float* lrow = p.logits + static_cast<int64_t>(t) * E;
  float v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    v[j] = (e < E) ? lrow[e] : -FLT_MAX;
  }
  const uint16_t* xrow = p.x + static_cast<int64_t>(t) * H;
  const float xnorm = sqrtf(row_sumsq(xrow, H, lane)) * 1.001f;
  float wm = 0.0f;
  for (int e = lane; e < E; e += 32) wm = fmaxf(wm, p.wnorm[e]);
  wm = warp_max(wm);
  const double tau = static_cast<double>(p.tau_coef) * static_cast<double>(xnorm) * static_cast<double>(wm);

  // (k+1) rounds of warp argmax by (value desc, id asc)
  uint32_t sel = 0;
  float vk = 0.0f, vk1 = -FLT_MAX;
  const int rounds = (k + 1 < E) ? k + 1 : E;
  for (int r = 0; r < rounds; ++r) {
    float bv = -FLT_MAX;
    int bid = INT_MAX;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = j * 32 + lane;
      if (e < E && !((sel >> j) & 1u) && (bid == INT_MAX || v[j] > bv)) {
        bv = v[j];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (ov > bv || (ov == bv && oid < bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if (r < k) {
      if (bid != INT_MAX && (bid & 31) == lane) sel |= 1u << (bid >> 5);
      if (r == k - 1) vk = bv;
    } else {
      vk1 = bv;
    }
  }

  bool band = false;
  if (k < E) band = !(static_cast<double>(vk) - static_cast<double>(vk1) > 2.0 * tau);
  if (band) {
    const double hi = static_cast<double>(vk1) + 2.0 * tau;  // above: certainly among the k largest
    const double lo = static_cast<double>(vk) - 2.0 * tau;   // below: certainly not
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
    const int need = k - warp_sum_i(__popc(sure));
    double d[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      d[j] = 0.0;
      if ((cand >> j) & 1u) d[j] = exact_logit(xrow, p.w_router + static_cast<int64_t>(j * 32 + lane) * H, H);
    }
    uint32_t chosen = 0;
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
    sel = sure | chosen;
  }

  // weights: softmax over the selected fp32 logits (= full softmax renormalised over the selection)
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
  if (pos < k) {
    // cannot happen for finite logits; keep every slot a valid expert id so later kernels stay in bounds
    if (lane >= pos && lane < k) {
      ids_out[lane] = 0;
      w_out[lane] = 0.0f;
    }
    if (lane == 0) atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, t));
  }
  if (lane == 0) p.band_flag[t] = band ? 1 : 0;
}

// Histogram of a block of 32 tokens: for every expert, a bit mask of the block's tokens that selected it.
__global__ void __launch_bounds__(256) count_kernel(PermuteParams p) {
  __shared__ int32_t ids[32 * 32];
  const int b = blockIdx.x;
  const int t0 = b * 32;
  const int nt = min(32, p.n - t0);
  const int k = p.k, E = p.E;
  for (int i = threadIdx.x; i < 32 * k; i += blockDim.x) {
    const int tok = i / k;
    ids[i] = (tok < nt) ? p.topk_id[static_cast<int64_t>(t0 + tok) * k + (i % k)] : -1;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t m = 0;
    for (int tok = 0; tok < nt; ++tok) {
      const int32_t* r = ids + tok * k;
      for (int s = 0; s < k; ++s)
        if (r[s] == e) m |= 1u << tok;
    }
    p.masks[static_cast<int64_t>(b) * E + e] = m;
    p.counts[static_cast<int64_t>(b) * E + e] = __popc(m);
  }
  if (threadIdx.x < 32) {
    const int f = (static_cast<int>(threadIdx.x) < nt) ? p.band_flag[t0 + threadIdx.x] : 0;
    const uint32_t bb = __ballot_sync(0xffffffffu, f != 0);
    if (threadIdx.x == 0) p.block_band[b] = __popc(bb);
  }
}

// Exclusive scan across a block of 1024 threads; returns the thread's exclusive prefix, *total gets the sum.
__device__ int block_exclusive_scan(int v, int* total, int* smem32) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
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
    const int ws = smem32[lane];
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

// One CTA of 1024 threads, thread e = expert e: per-expert totals, expert offsets, per-(block, expert) row bases,
// and the tile lists of the gate/up and down GEMMs (expert-major: expert, then N tile, then M tile).
__global__ void __launch_bounds__(1024) scan_tiles_kernel(PermuteParams p) {
  __shared__ int sm[33];
  const int e = threadIdx.x;
  const int E = p.E, nblk = p.nblk;
  int total = 0;
  if (e < E)
    for (int b = 0; b < nblk; ++b) total += p.counts[static_cast<int64_t>(b) * E + e];
  int R = 0;
  const int off = block_exclusive_scan(e < E ? total : 0, &R, sm);
  if (e < E) {
    p.offsets[e] = off;
    if (p.offsets_out) p.offsets_out[e] = off;
    int run = off;
    for (int b = 0; b < nblk; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      p.base[i] = run;
      run += p.counts[i];
    }
  }
  if (e == 0) {
    p.offsets[E] = R;
    if (p.offsets_out) p.offsets_out[E] = R;
  }
  const int mt = (e < E) ? (total + kBlockM - 1) / kBlockM : 0;
  int n_gu = 0, n_dn = 0;
  const int gu_base = block_exclusive_scan(mt * p.nt_gu, &n_gu, sm);
  const int dn_base = block_exclusive_scan(mt * p.nt_down, &n_dn, sm);
  const int mts = (p.n + kBlockM - 1) / kBlockM;
  const int n_gu_all = n_gu + (p.nt_gu_shared > 0 ? mts * p.nt_gu_shared : 0);
  const int n_dn_all = n_dn + (p.nt_down_shared > 0 ? mts * p.nt_down_shared : 0);
  const bool fits = n_gu_all <= p.cap_gu && n_dn_all <= p.cap_down;
  if (fits && e < E) {
    for (int nn = 0; nn < p.nt_gu; ++nn)
      for (int m = 0; m < mt; ++m)
        p.tiles_gu[gu_base + nn * mt + m] =
            make_int4(e | (nn << 16), off + m * kBlockM, min(kBlockM, total - m * kBlockM), off + m * kBlockM);
    for (int nn = 0; nn < p.nt_down; ++nn)
      for (int m = 0; m < mt; ++m)
        p.tiles_down[dn_base + nn * mt + m] =
            make_int4(e | (nn << 16), off + m * kBlockM, min(kBlockM, total - m * kBlockM), off + m * kBlockM);
  }
  if (fits) {
    // shared expert (class 1): gate/up reads the chunk's rows of X, down reads the shared h rows
    for (int i = threadIdx.x; i < mts * p.nt_gu_shared; i += blockDim.x) {
      const int nn = i / mts, m = i % mts;
      p.tiles_gu[n_gu + i] = make_int4((1 << 15) | (nn << 16), static_cast<int>(p.token0) + m * kBlockM,
                                       min(kBlockM, p.n - m * kBlockM), m * kBlockM);
    }
    for (int i = threadIdx.x; i < mts * p.nt_down_shared; i += blockDim.x) {
      const int nn = i / mts, m = i % mts;
      p.tiles_down[n_dn + i] =
          make_int4((1 << 15) | (nn << 16), m * kBlockM, min(kBlockM, p.n - m * kBlockM), m * kBlockM);
    }
  }
  if (threadIdx.x == 0) {
    p.num_tiles[0] = fits ? n_gu_all : 0;
    p.num_tiles[1] = fits ? n_dn_all : 0;
    if (!fits) atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, 0));
    int band = 0;
    for (int b = 0; b < nblk; ++b) band += p.block_band[b];
    p.hdr->band_tokens += band;
    p.hdr->chunks_done += 1;
  }
}

// Row index of every (token, slot), the inverse map, and the gathered copy of X in expert-major row order.
__global__ void __launch_bounds__(256) permute_kernel(PermuteParams p) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t0 = b * 32;
  const int nt = min(32, p.n - t0);
  const int k = p.k, E = p.E, H = p.H;
  __shared__ int32_t rows_sm[8][32];
  for (int i = warp; i < nt; i += 8) {
    const int t = t0 + i;
    if (lane < k) {
      int e = p.topk_id[static_cast<int64_t>(t) * k + lane];
      if (e < 0 || e >= E) {
        atomicCAS(&p.hdr->err, 0, dev_error_code(kDevErrBounds, kSiteRouting, t));
        e = 0;
      }
      const int64_t be = static_cast<int64_t>(b) * E + e;
      int row = p.base[be] + __popc(p.masks[be] & ((1u << i) - 1u));
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
      for (int s = 0; s < k; ++s)
        reinterpret_cast<uint4*>(p.xp + static_cast<int64_t>(rows_sm[warp][s]) * H)[c] = val;
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_router_norms(const uint16_t* w_router, int E, int H, float* wnorm, WsHeader* hdr,
                                cudaStream_t stream) {
  router_norms_kernel<<<(E + 7) / 8, 256, 0, stream>>>(w_router, E, H, wnorm, hdr);
  return cudaGetLastError();
}

cudaError_t launch_topk(const RouteParams& p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  const int grid = (p.n + 7) / 8;
  const int epl = (p.E + 31) / 32;
  if (epl <= 1)
    topk_kernel<1><<<grid, 256, 0, stream>>>(p);
  else if (epl <= 2)
    topk_kernel<2><<<grid, 256, 0, stream>>>(p);
  else if (epl <= 4)
    topk_kernel<4><<<grid, 256, 0, stream>>>(p);
  else if (epl <= 8)
    topk_kernel<8><<<grid, 256, 0, stream>>>(p);
  else if (epl <= 16)
    topk_kernel<16><<<grid, 256, 0, stream>>>(p);
  else
    topk_kernel<32><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_count(const PermuteParams& p, cudaStream_t stream) {
  count_kernel<<<p.nblk, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scan_tiles(const PermuteParams& p, cudaStream_t stream) {
  scan_tiles_kernel<<<1, 1024, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t stream) {
  permute_kernel<<<p.nblk, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
