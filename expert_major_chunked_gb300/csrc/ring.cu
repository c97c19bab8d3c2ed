// Device-planned staging of offloaded experts. The umbrella PR #1113 ("Memory and execution split") keeps expert
// banks in pinned host memory and lets device-planned paths fill expert lines with GPU kernels that read the mapped
// host banks; "Latest measured follow-up" names expert-transfer volume as the cost and accounts the copied bytes by
// category. Here a kernel stages one window of experts of one chunk into the HBM ring, reading the pinned banks
// through their device-accessible addresses, and copies only the experts that the chunk's member lists route rows
// to (an expert without gate/up tiles is skipped). The decision is taken on the device, from the chunk's tile
// bases, so no count travels to the host and nothing waits on it.
//
// On GB300 the host link, not the SMs, bounds this copy: a few dozen CTAs reach the same rate as the copy engines,
// so the kernel runs on a small grid beside the expert GEMMs.
#include "internal.h"

namespace moe {
namespace {

constexpr int kRingThreads = 256;
constexpr int kRingBlocks = 64;

__device__ __forceinline__ void copy16(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {  // four independent loads in flight per thread
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

__global__ void __launch_bounds__(kRingThreads) ring_copy_kernel(RingCopyParams p) {
  int copied = 0, hot = 0;
  for (int e = p.e0; e < p.e0 + p.count; ++e) {
    if (p.tile_base[e + 1] <= p.tile_base[e]) continue;  // no row of this chunk goes to expert e
    if (p.slot_map != nullptr && p.slot_map[e] >= p.slots) {  // resident in the hot set
      ++hot;
      continue;
    }
    ++copied;
    const int64_t slot = e % p.slots;
    copy16(p.bank_gu + e * p.gu16, p.ring_gu + slot * p.gu16, p.gu16);
    copy16(p.bank_down + e * p.dn16, p.ring_down + slot * p.dn16, p.dn16);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    atomicAdd(&p.hdr->experts_copied, copied);
    atomicAdd(&p.hdr->experts_skipped, p.count - copied - hot);
    atomicAdd(&p.hdr->experts_hot, hot);
  }
}

}  // namespace

cudaError_t launch_ring_copy(const RingCopyParams& p, cudaStream_t stream) {
  if (p.count <= 0) return cudaSuccess;
  ring_copy_kernel<<<kRingBlocks, kRingThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
