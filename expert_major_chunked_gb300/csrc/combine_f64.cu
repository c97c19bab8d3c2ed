// Routed combine with float64 partials, for an expert-parallel split whose result equals the unsplit one.
// "EXL3 Flash Next: deep prefill (3/8)", "What this changes": the tensor-parallel prefill partials are float64;
// "Checklist": they are summed in float64 and rounded once, to float32, at the finish, so two GPUs give the bits of
// one. The order inside a partial is not given there; this file fixes it as a complete binary tree over the expert
// ids 0 .. Ep-1 (Ep = least power of two >= E): leaf e = w*y of the slot routed to expert e (exact in float64),
// +0.0 for an expert the token did not choose, each inner node the float64 sum of its children. A part of the split
// is an aligned block of ids, i.e. a subtree, and the finish sums the parts in the same tree, so splitting changes
// no operation.
//
// Only the token's own slots are touched: the sparse tree over its sorted ids is evaluated as a post-order program,
// built once per token by one thread and run by every thread on its columns. Where a node has an empty sibling the
// dense tree adds +0.0, which changes a value only by turning -0.0 into +0.0; the program applies that as a bit test
// instead of an addition.
//
// The float64 pipe is the bound (on GB300 it is a small fraction of the float32 rate), and float <-> double
// conversions and float64 multiplies run on it too. So only the additions use it: a leaf product w*y of two normal
// floats is formed exactly on the integer pipe (24-bit x 24-bit significands give at most 48 bits, which a double
// holds), and the exact widening of a normal float and the rounding of a double whose float result is normal are
// done with integer operations (IEEE 754 binary32/binary64 layouts; other values take the float64 instructions).
#include "internal.h"

#include <cuda_bf16.h>

#include <algorithm>

namespace moe {
namespace {

constexpr int kTreeThreads = 128;
constexpr int kTreeSlots = 10;  // stored nodes: at most log2(1024) - 1 wait for a right sibling
constexpr uint8_t kNoLeaf = 0xFF;
constexpr uint8_t kOpPlusZero = 1;  // the node has an empty sibling below it: turn -0.0 into +0.0
constexpr uint8_t kOpPush = 2;      // store the current value to stack slot p (no arithmetic)

// MERGE: cur = left + right, left = raw leaf `la` (its exact product w*y) or stack slot p, right = raw leaf `lb`
// or the current value (the previous merge's result). PUSH: stack[p] = cur.
struct TreeOp {
  uint8_t p, la, lb, flags;
};

struct TreeProgram {
  int m;          // leaves (the token's slots inside the part), ascending expert id
  int nops;
  int root_pz;    // the root has an empty sibling below the part's top
  int32_t row[32];
  float w[32];
  TreeOp op[64];
};

__device__ __forceinline__ double plus_zero(double v) {
  return __double_as_longlong(v) == static_cast<long long>(0x8000000000000000ull) ? 0.0 : v;
}

// Exact float -> double. Normal floats by their bit layout; zeros, subnormals, inf and NaN by the instruction.
__device__ __forceinline__ double widen(float f) {
  const uint32_t b = __float_as_uint(f);
  const uint32_t mag = b & 0x7FFFFFFFu;
  if (mag - 0x00800000u < 0x7F000000u) {
    const uint32_t hi = (b & 0x80000000u) | ((mag >> 3) + (896u << 20));  // exponent bias 127 -> 1023
    return __hiloint2double(static_cast<int>(hi), static_cast<int>(b << 29));
  }
  return static_cast<double>(f);
}

// double -> float, round to nearest, ties to even. Results with a normal float exponent (before rounding) by the
// bit layout: keep 23 of the 52 fraction bits and round on the 29 dropped ones (a carry into the exponent is the
// correct result, up to infinity). Everything else by the instruction.
__device__ __forceinline__ float narrow_rn(double v) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  const uint32_t hi = static_cast<uint32_t>(b >> 32);
  const uint32_t e = (hi >> 20) & 0x7FFu;
  if (e - 897u < 254u) {
    const uint32_t keep = static_cast<uint32_t>(b >> 29) & 0x7FFFFFu;
    const uint32_t rest = static_cast<uint32_t>(b) & 0x1FFFFFFFu;
    uint32_t out = (hi & 0x80000000u) | ((e - 896u) << 23) | keep;
    out += (rest > 0x10000000u || (rest == 0x10000000u && (keep & 1u))) ? 1u : 0u;
    return __uint_as_float(out);
  }
  return __double2float_rn(v);
}

// Exact w*y as a double. For normal floats the product of the two 24-bit significands (at most 48 bits) is formed
// with one 32x32->64 integer multiply and packed with the summed exponents; it is never subnormal or infinite in
// double. Zeros, subnormals, inf and NaN take the float64 multiply, also exact.
__device__ __forceinline__ double exact_product(float a, float b) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const uint32_t ea = (ua >> 23) & 0xFFu, eb = (ub >> 23) & 0xFFu;
  if (ea - 1u < 254u && eb - 1u < 254u) {
    const uint64_t p = static_cast<uint64_t>((ua & 0x7FFFFFu) | 0x800000u) * ((ub & 0x7FFFFFu) | 0x800000u);
    const uint32_t top = static_cast<uint32_t>(p >> 47);                // leading one at bit 46 + top
    const uint64_t frac = (p << (6u - top)) & 0x000FFFFFFFFFFFFFull;    // the bits below it, as 52 fraction bits
    const uint64_t expo = static_cast<uint64_t>(ea + eb + 769u + top);  // (46 + top) + (ea - 150) + (eb - 150) + 1023
    const uint64_t sign = static_cast<uint64_t>((ua ^ ub) & 0x80000000u) << 32;
    return __longlong_as_double(static_cast<long long>(sign | (expo << 52) | frac));
  }
  return __dmul_rn(static_cast<double>(a), static_cast<double>(b));
}

__device__ __forceinline__ int bit_length(uint32_t v) { return v == 0 ? 0 : 32 - __clz(v); }

// One thread, operands already in shared memory: sort the slots inside [lo, lo + 2^block_log2) by expert id and
// emit the post-order program of the sparse tree (a binary radix tree: two neighbours in id order meet at the
// level of the highest bit in which their ids differ).
__device__ void build_program(TreeProgram& P, const int32_t* ids, const float* w, const int32_t* rows, int k, int lo,
                              int block_log2) {
  int e_sorted[32];
  int m = 0;
  const int block = 1 << block_log2;
  for (int s = 0; s < k; ++s) {
    const int e = ids[s];
    if (e < lo || e >= lo + block) continue;
    int j = m;
    bool dup = false;
    while (j > 0 && e_sorted[j - 1] >= e) {
      if (e_sorted[j - 1] == e) dup = true;
      --j;
    }
    if (dup) continue;  // a repeated id counts once, in its first slot
    for (int q = m; q > j; --q) {
      e_sorted[q] = e_sorted[q - 1];
      P.row[q] = P.row[q - 1];
      P.w[q] = P.w[q - 1];
    }
    e_sorted[j] = e;
    P.row[j] = rows[s];
    P.w[j] = w[s];
    ++m;
  }
  P.m = m;
  P.nops = 0;
  P.root_pz = 0;
  if (m == 0) return;
  // Stack entries: raw leaf index (or -1 for a stored node), node height, merge level to the right. The levels on
  // the stack fall strictly from bottom to top and lie in 1..block_log2, so at most block_log2 entries wait.
  int st_leaf[kTreeSlots + 1], st_h[kTreeSlots + 1], st_gap[kTreeSlots + 1];
  int sp = 0, nops = 0;
  for (int i = 0; i < m; ++i) {
    int cur_leaf = i, cur_h = 0;
    const int right_gap = (i + 1 < m) ? bit_length(static_cast<uint32_t>(e_sorted[i] ^ e_sorted[i + 1])) : 127;
    while (sp > 0 && st_gap[sp - 1] < right_gap) {
      --sp;
      const int L = st_gap[sp];
      TreeOp o;
      o.p = static_cast<uint8_t>(sp);
      o.la = st_leaf[sp] >= 0 ? static_cast<uint8_t>(st_leaf[sp]) : kNoLeaf;
      o.lb = cur_leaf >= 0 ? static_cast<uint8_t>(cur_leaf) : kNoLeaf;
      o.flags = (st_h[sp] < L - 1 || cur_h < L - 1) ? kOpPlusZero : 0;
      P.op[nops++] = o;
      cur_leaf = -1;
      cur_h = L;
    }
    if (cur_leaf < 0 && i + 1 < m) {  // a computed node waits on the stack for its right sibling
      TreeOp o;
      o.p = static_cast<uint8_t>(sp);
      o.la = kNoLeaf;
      o.lb = kNoLeaf;
      o.flags = kOpPush;
      P.op[nops++] = o;
    }
    st_leaf[sp] = cur_leaf;
    st_h[sp] = cur_h;
    st_gap[sp] = right_gap;
    ++sp;
  }
  P.nops = nops;
  P.root_pz = st_h[0] < block_log2 ? 1 : 0;
}

// One block per token; each thread runs the program on two adjacent columns at a time. The current value lives in
// registers; the leaves' y values yl[k][threads] and the stack stk[kTreeSlots][threads] live in shared memory,
// indexed [slot][thread] so that a warp's accesses fall in distinct banks.
// MODE 0: write the part's float64 value to `partial`. MODE 1: finish in place (+ s, float32, bf16).
template <int MODE>
__global__ void __launch_bounds__(kTreeThreads) combine_tree_kernel(CombineTreeParams a) {
  extern __shared__ __align__(16) unsigned char tree_smem[];
  __shared__ TreeProgram P;
  __shared__ int32_t s_ids[32], s_rows[32];
  __shared__ float s_w[32];
  float2* yl = reinterpret_cast<float2*>(tree_smem);                                           // [k][threads]
  double2* stk = reinterpret_cast<double2*>(tree_smem + a.k * kTreeThreads * sizeof(float2));  // [slots][threads]
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < a.k) {  // the token's slots, loaded in parallel
    s_ids[tid] = a.topk_id[t * a.k + tid];
    s_w[tid] = a.w[t * a.k + tid];
    s_rows[tid] = a.token_row[t * a.k + tid];
  }
  __syncthreads();
  if (tid == 0) build_program(P, s_ids, s_w, s_rows, a.k, a.lo, a.block_log2);
  __syncthreads();
  const int m = P.m, nops = P.nops;
  // The first kPrefetch leaves of the next column pair are loaded into registers while the current pair is summed
  // (one memory round trip per pair, hidden behind the additions); leaves beyond kPrefetch load on the spot.
  constexpr int kPrefetch = 16;
  const int step = 2 * kTreeThreads;
  float2 nxt[kPrefetch];
  if (2 * tid < a.H) {
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j)
      if (j < m) nxt[j] = __ldg(reinterpret_cast<const float2*>(a.y + static_cast<int64_t>(P.row[j]) * a.H + 2 * tid));
  }
  for (int c = 2 * tid; c < a.H; c += step) {
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j)
      if (j < m) yl[j * kTreeThreads + tid] = nxt[j];
    for (int j = kPrefetch; j < m; ++j)
      yl[j * kTreeThreads + tid] = __ldg(reinterpret_cast<const float2*>(a.y + static_cast<int64_t>(P.row[j]) * a.H + c));
    if (c + step < a.H) {
#pragma unroll
      for (int j = 0; j < kPrefetch; ++j)
        if (j < m)
          nxt[j] = __ldg(reinterpret_cast<const float2*>(a.y + static_cast<int64_t>(P.row[j]) * a.H + c + step));
    }
    double2 cur = make_double2(0.0, 0.0);
    if (m == 1) {
      const float2 yv = yl[tid];
      cur.x = exact_product(P.w[0], yv.x);
      cur.y = exact_product(P.w[0], yv.y);
    }
    for (int j = 0; j < nops; ++j) {
      const TreeOp o = P.op[j];
      if (o.flags & kOpPush) {
        stk[o.p * kTreeThreads + tid] = cur;
        continue;
      }
      double2 b;
      if (o.lb != kNoLeaf) {
        const float2 yv = yl[o.lb * kTreeThreads + tid];
        const float wb = P.w[o.lb];
        b.x = exact_product(wb, yv.x);
        b.y = exact_product(wb, yv.y);
      } else {
        b = cur;
      }
      double2 av;
      if (o.la != kNoLeaf) {
        const float2 yv = yl[o.la * kTreeThreads + tid];
        const float wa = P.w[o.la];
        av.x = exact_product(wa, yv.x);
        av.y = exact_product(wa, yv.y);
      } else {
        av = stk[o.p * kTreeThreads + tid];
      }
      cur.x = __dadd_rn(av.x, b.x);
      cur.y = __dadd_rn(av.y, b.y);
      if (o.flags & kOpPlusZero) {
        cur.x = plus_zero(cur.x);
        cur.y = plus_zero(cur.y);
      }
    }
    if (P.root_pz) {
      cur.x = plus_zero(cur.x);
      cur.y = plus_zero(cur.y);
    }
    const int64_t at = t * a.H + c;
    if (MODE == 0) {
      *reinterpret_cast<double2*>(a.partial + at) = cur;
    } else {
      if (a.s != nullptr) {
        const float2 sv = __ldg(reinterpret_cast<const float2*>(a.s + at));
        cur.x = __dadd_rn(cur.x, widen(sv.x));
        cur.y = __dadd_rn(cur.y, widen(sv.y));
      }
      const float2 f = make_float2(narrow_rn(cur.x), narrow_rn(cur.y));
      *reinterpret_cast<__nv_bfloat162*>(a.out + at) = __floats2bfloat162_rn(f.x, f.y);
      if (a.out_f32 != nullptr) *reinterpret_cast<float2*>(a.out_f32 + at) = f;
    }
  }
}

// Elementwise finish over n*H values: the parts summed pairwise in the tree, + s, float32, bf16.
__global__ void __launch_bounds__(256) combine_finish_kernel(CombineFinishParams a) {
  const int64_t total2 = a.count / 2;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total2;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    double2 v[kMaxFinishParts];
#pragma unroll
    for (int p = 0; p < kMaxFinishParts; ++p)
      v[p] = p < a.n_parts ? __ldg(reinterpret_cast<const double2*>(a.part[p]) + i) : make_double2(0.0, 0.0);
#pragma unroll
    for (int width = kMaxFinishParts; width > 1; width /= 2) {
      if (width <= a.n_parts) {
#pragma unroll
        for (int p = 0; p < width / 2; ++p) {
          v[p].x = __dadd_rn(v[2 * p].x, v[2 * p + 1].x);
          v[p].y = __dadd_rn(v[2 * p].y, v[2 * p + 1].y);
        }
      }
    }
    double2 r = v[0];
    if (a.s != nullptr) {
      const float2 sv = __ldg(reinterpret_cast<const float2*>(a.s) + i);
      r.x = __dadd_rn(r.x, widen(sv.x));
      r.y = __dadd_rn(r.y, widen(sv.y));
    }
    const float2 f = make_float2(narrow_rn(r.x), narrow_rn(r.y));
    reinterpret_cast<__nv_bfloat162*>(a.out)[i] = __floats2bfloat162_rn(f.x, f.y);
    if (a.out_f32 != nullptr) reinterpret_cast<float2*>(a.out_f32)[i] = f;
  }
}

}  // namespace

size_t combine_tree_smem_bytes(int k) {
  return static_cast<size_t>(k) * kTreeThreads * sizeof(float2) + kTreeSlots * kTreeThreads * sizeof(double2);
}

cudaError_t launch_combine_tree(const CombineTreeParams& a, bool finish, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  const size_t smem = combine_tree_smem_bytes(a.k);
  const void* fn = finish ? reinterpret_cast<const void*>(combine_tree_kernel<1>)
                          : reinterpret_cast<const void*>(combine_tree_kernel<0>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (finish)
    combine_tree_kernel<1><<<static_cast<unsigned>(a.n), kTreeThreads, smem, stream>>>(a);
  else
    combine_tree_kernel<0><<<static_cast<unsigned>(a.n), kTreeThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine_finish(const CombineFinishParams& a, int num_sms, cudaStream_t stream) {
  if (a.count <= 0) return cudaSuccess;
  const int64_t pairs = a.count / 2;
  const int64_t want = (pairs + 255) / 256;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, static_cast<int64_t>(num_sms) * 8));
  combine_finish_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
