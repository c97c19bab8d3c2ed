// The SwiGLU of the gate/up epilogues (grouped_gemm_kernel and grouped_pair_kernel), in one place so that both
// kernels round it identically.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace moe {

__device__ __forceinline__ float swiglu(float g, float u) {
  // silu(g) * u with silu(z) = z / (1 + exp(-z)); IEEE-rounded division and products.
  const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  return __fmul_rn(s, u);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace moe
