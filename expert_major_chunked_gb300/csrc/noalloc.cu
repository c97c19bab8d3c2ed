// The layer for callers that must not allocate device memory.
//
// moe_prefill_run needs a scratch workspace that the caller allocates. Some callers cannot do that at the point
// where they run the layer: code whose device memory is owned by another allocator or memory pool (calling
// cudaMalloc behind its back breaks its accounting and can fail when it has reserved nearly all of the GPU), code
// running under a strict no-allocation-after-start-up rule (latency-critical serving loops, where cudaMalloc and
// cudaFree synchronise the device), and code that is only handed raw input and output pointers by a host framework.
// moe_prefill_run_noalloc gives them the same computation with the scratch held in a fixed array inside this
// library instead.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <cstdio>
#include <mutex>

namespace {

// The scratch. Every GPU that loads this library holds these bytes until the process exits. All calls on a device
// share them, so two calls whose work overlaps on the GPU (for example on two streams) race on this memory.
static __device__ __align__(256) unsigned char g_noalloc_workspace[MOE_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

thread_local char g_msg[256];

// Device address of the array on the current device, looked up once per device (host code cannot use the
// symbol's name as an address: on the host it names a stand-in, not device memory).
cudaError_t scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace

namespace moe {
size_t plan_workspace_bytes(moe_plan_t plan);  // defined in moe_prefill.cu
}

extern "C" moe_status moe_prefill_run_noalloc(moe_plan_t plan, const void* x, int64_t T, int32_t chunk, void* out,
                                              int32_t* topk_id, float* topk_w, int32_t* expert_offsets,
                                              int32_t* row_token, int32_t* device_status, moe_stream_t stream) {
  if (!plan) {
    // Report through moe_prefill_run so that moe_prefill_last_error() carries the message.
    return moe_prefill_run(nullptr, x, T, chunk, nullptr, 0, out, topk_id, topk_w, expert_offsets, row_token,
                           stream, nullptr);
  }
  const size_t need = moe::plan_workspace_bytes(plan);
  if (need > static_cast<size_t>(MOE_NOALLOC_WORKSPACE_BYTES)) {
    snprintf(g_msg, sizeof g_msg,
             "moe_prefill_run_noalloc: this plan needs %zu bytes of scratch, more than the built-in %zu; use a "
             "smaller max_chunk or moe_prefill_run with a workspace",
             need, static_cast<size_t>(MOE_NOALLOC_WORKSPACE_BYTES));
    moe::set_last_error(g_msg);
    return MOE_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof g_msg, "moe_prefill_run_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    moe::set_last_error(g_msg);
    return MOE_ERR_CUDA;
  }
  // The run itself resets the status word and counters at the head of the scratch before any other work, and writes
  // every per-run byte whose value can reach an output earlier in the same run (stale bytes are read only as padding
  // rows of a GEMM tile, whose results are never stored). The bytes an offloaded plan keeps between runs (its hot
  // set's slots and slot map) are tracked per workspace address by moe_prefill_run: since every call here passes
  // the same address, a plan that was not the last one to run on the array stages them again.
  moe_status st = moe_prefill_run(plan, x, T, chunk, scratch, MOE_NOALLOC_WORKSPACE_BYTES, out, topk_id, topk_w,
                                  expert_offsets, row_token, stream, nullptr);
  if (st != MOE_OK || !device_status) return st;
  if (T == 0) {
    e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream));
  } else {
    e = cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        reinterpret_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof g_msg, "moe_prefill_run_noalloc: status copy failed: %s", cudaGetErrorString(e));
    moe::set_last_error(g_msg);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
