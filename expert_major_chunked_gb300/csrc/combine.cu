// Canonical weighted combine. "Flash Next EXL3: exact deep prefill" (introduction) reduces the routed-expert
// contributions of a token in one canonical order, which makes every output row independent of the chunk size;
// "EXL3 Flash Next: deep prefill (3/8)" (Checklist) asks that a changed summation be named. The order used here:
// float32 accumulation from +0.0f over the token's slots in ascending expert id, each product w*y and each sum
// rounded to float32 (no fused multiply-add), then the shared expert's output, then one BF16 rounding (ties to
// even).
#include "internal.h"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ uint2 pack4_bf16(float4 a) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// One block per token; each thread owns 4 consecutive columns per step.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ y,
                                                                  const float* __restrict__ w,
                                                                  const int32_t* __restrict__ token_row,
                                                                  const float* __restrict__ s, int k, int H,
                                                                  uint16_t* __restrict__ out) {
  __shared__ int32_t rows[32];
  __shared__ float wts[32];
  const int64_t t = blockIdx.x;
  if (threadIdx.x < static_cast<unsigned>(k)) {
    rows[threadIdx.x] = token_row[t * k + threadIdx.x];
    wts[threadIdx.x] = w[t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 4; c < H; c += kCombineThreads * 4) {
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // slots in groups of 8: issue the group's loads first (memory-level parallelism), then add them in order
    for (int s0 = 0; s0 < k; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < k) v[j] = __ldg(reinterpret_cast<const float4*>(y + static_cast<int64_t>(rows[s0 + j]) * H + c));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j < k) {
          const float ws = wts[s0 + j];
          acc.x = __fadd_rn(acc.x, __fmul_rn(ws, v[j].x));
          acc.y = __fadd_rn(acc.y, __fmul_rn(ws, v[j].y));
          acc.z = __fadd_rn(acc.z, __fmul_rn(ws, v[j].z));
          acc.w = __fadd_rn(acc.w, __fmul_rn(ws, v[j].w));
        }
      }
    }
    if (s != nullptr) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(s + t * H + c));
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    *reinterpret_cast<uint2*>(out + t * H + c) = pack4_bf16(acc);
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* w, const int32_t* token_row, const float* s, int64_t n,
                           int k, int H, uint16_t* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  combine_kernel<<<static_cast<unsigned>(n), kCombineThreads, 0, stream>>>(y, w, token_row, s, k, H, out);
  return cudaGetLastError();
}

}  // namespace moe
