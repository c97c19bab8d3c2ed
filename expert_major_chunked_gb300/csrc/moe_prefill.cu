// Host side of the C ABI declared in include/moe_prefill.h: validation, workspace layout, TMA descriptors and the
// chunk loop. All arithmetic runs in the kernels of gemm.cu, gemm_pair.cu, route.cu, combine.cu, combine_f64.cu and
// ring.cu.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

using namespace moe;

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                            \
  do {                                                                                            \
    cudaError_t e_ = (expr);                                                                      \
    if (e_ != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));   \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_log2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ TMA descriptor encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 matrix [rows][cols] (row-major), boxes of box_rows x 64 elements, 128-byte swizzle, zero fill out of range.
moe_status encode_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu x %llu] matrix, box %u rows", (int)r,
                (unsigned long long)rows, (unsigned long long)cols, box_rows);
  return MOE_OK;
}

// Fused gate/up weights of `groups` groups, each [2][half_rows][cols] bf16 (its gate rows, then its up rows), as
// the 3-D tensor (cols, half_rows, 2 x groups): a box of 64 x box_rows x 2 at (k, j, 2g) holds rows j..j+box_rows-1
// of group g's gate half followed by the same rows of its up half. 128-byte swizzle, zero fill out of range.
moe_status encode_bf16_halves(CUtensorMap* m, const void* ptr, uint64_t groups, uint64_t half_rows, uint64_t cols,
                              uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {cols, half_rows, 2 * groups};
  const cuuint64_t strides[2] = {cols * 2, half_rows * cols * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llu groups of 2 x [%llu x %llu], box %u rows",
                (int)r, (unsigned long long)groups, (unsigned long long)half_rows, (unsigned long long)cols, box_rows);
  return MOE_OK;
}

// The same fused gate/up weights with the 64-wide K block as the outermost dimension: (64, half_rows, 2 x groups,
// cols / 64), strides (cols x 2, half_rows x cols x 2, 128) bytes. A box of 64 x box_rows x 2 x kb at
// (0, j, 2g, k block) holds, for each of kb consecutive K blocks in turn, box_rows gate rows then the same up rows.
moe_status encode_bf16_halves_kb(CUtensorMap* m, const void* ptr, uint64_t groups, uint64_t half_rows, uint64_t cols,
                                 uint32_t box_rows, uint32_t kb) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kBlockK), half_rows, 2 * groups, cols / kBlockK};
  const cuuint64_t strides[3] = {cols * 2, half_rows * cols * 2, static_cast<cuuint64_t>(kBlockK) * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBlockK), box_rows, 2, kb};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llu groups of 2 x [%llu x %llu] by K blocks",
                (int)r, (unsigned long long)groups, (unsigned long long)half_rows, (unsigned long long)cols);
  return MOE_OK;
}

// bf16 matrix [rows][cols] (row-major) with the 64-wide K block as the outermost dimension: (64, rows, cols / 64),
// strides (cols x 2, 128) bytes; a box of 64 x box_rows x kb holds box_rows rows of each of kb consecutive K blocks.
moe_status encode_bf16_rows_kb(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                               uint32_t kb) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBlockK), rows, cols / kBlockK};
  const cuuint64_t strides[2] = {cols * 2, static_cast<cuuint64_t>(kBlockK) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), box_rows, kb};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu x %llu] matrix by K blocks, box %u rows",
                (int)r, (unsigned long long)rows, (unsigned long long)cols, box_rows);
  return MOE_OK;
}

// fp32 output matrix [rows][cols] with row stride ld elements (ld % 4 == 0), written by TMA stores of 32 x 32
// blocks staged with 128-byte swizzle; stores past rows or cols are clipped.
moe_status encode_f32_out(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols, uint64_t ld) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu x %llu] fp32 output", (int)r,
                (unsigned long long)rows, (unsigned long long)cols);
  return MOE_OK;
}

// uint8 tensor of `rank` dimensions (dims[0] innermost, strides in bytes for dims 1..rank-1), no swizzle, zero fill.
moe_status encode_u8_nd(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                        const cuuint32_t* box, const char* what) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %s", (int)r, what);
  return MOE_OK;
}

// Codes of fused gate/up weights, `groups` groups of [2][half_rows][row_bytes], as (row_bytes, half_rows, 2 x groups):
// a box of step_bytes x box_rows x 2 holds box_rows gate code rows, then the same up rows.
moe_status encode_u8_halves(CUtensorMap* m, const void* ptr, uint64_t groups, uint64_t half_rows, uint64_t row_bytes,
                            uint32_t box_rows, uint32_t step_bytes) {
  const cuuint64_t dims[3] = {row_bytes, half_rows, 2 * groups};
  const cuuint64_t strides[2] = {row_bytes, half_rows * row_bytes};
  const cuuint32_t box[3] = {step_bytes, box_rows, 2};
  return encode_u8_nd(m, ptr, 3, dims, strides, box, "gate/up code halves");
}

// Scale planes [groups][planes][2 x half_rows] of fused gate/up weights as (half_rows, 2, planes, groups): a box of
// box_rows x 2 x blocks x 1 holds, for each of `blocks` planes in turn, box_rows gate scales then the same up scales.
moe_status encode_u8_scales_gu(CUtensorMap* m, const void* ptr, uint64_t groups, uint64_t planes, uint64_t half_rows,
                               uint32_t box_rows, uint32_t blocks) {
  const cuuint64_t dims[4] = {half_rows, 2, planes, groups};
  const cuuint64_t strides[3] = {half_rows, 2 * half_rows, planes * 2 * half_rows};
  const cuuint32_t box[4] = {box_rows, 2, blocks, 1};
  return encode_u8_nd(m, ptr, 4, dims, strides, box, "gate/up scale planes");
}

// Scale planes [groups][planes][rows] as (rows, planes, groups): a box of box_rows x blocks x 1.
moe_status encode_u8_scales(CUtensorMap* m, const void* ptr, uint64_t groups, uint64_t planes, uint64_t rows,
                            uint32_t box_rows, uint32_t blocks) {
  const cuuint64_t dims[3] = {rows, planes, groups};
  const cuuint64_t strides[2] = {rows, planes * rows};
  const cuuint32_t box[3] = {box_rows, blocks, 1};
  return encode_u8_nd(m, ptr, 3, dims, strides, box, "down scale planes");
}

// Code matrix [rows][cols] of bytes (row-major), boxes of box_rows x box_bytes, no swizzle (the decoder warps read
// the rows densely), zero fill out of range.
moe_status encode_u8_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                        uint32_t box_bytes) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu x %llu] code matrix, box %u rows",
                (int)r, (unsigned long long)rows, (unsigned long long)cols, box_rows);
  return MOE_OK;
}

// ------------------------------------------------------------------ device checks
moe_status check_device(int* device, int* num_sms) {
  CUDA_TRY(cudaGetDevice(device));
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, *device));
  if (prop.major != 10 || prop.minor != 3)
    return fail(MOE_ERR_ARCH, "device %d is sm_%d%d; the kernels are built for sm_103a", *device, prop.major,
                prop.minor);
  *num_sms = prop.multiProcessorCount;
  static std::mutex mu;
  static std::vector<int> prepared;
  std::lock_guard<std::mutex> lock(mu);
  if (std::find(prepared.begin(), prepared.end(), *device) == prepared.end()) {
    cudaError_t e = prepare_gemm_kernels();
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
      return fail(MOE_ERR_ARCH, "kernels do not load on device %d: %s", *device, cudaGetErrorString(e));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    // CTA pairs: without room for a cluster of two (pair_cluster_slots() == 0) plans use the single-CTA kernel
    e = prepare_pair_kernels();
    if (e == cudaErrorInvalidConfiguration) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "CTA-pair kernel setup: %s", cudaGetErrorString(e));
    prepared.push_back(*device);
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ workspace layout
struct Layout {
  size_t hdr, wnorm, logits, topk_id, topk_w, band, band_info, masks, counts, base, totals, block_band, offsets, h, hs,
      y, s, total;
  // two sets (chunk parity): the member lists of chunk c+1 are built while chunk c's GEMMs still read chunk c's
  size_t token_row[2], num_tiles[2], tiles_gu[2], tiles_down[2], xp[2], tile_base[2];
  size_t ring_gu, ring_down;  // offloaded experts: the HBM ring of expert slots, then the hot set's slots
  size_t slot_map;            // offloaded experts: slot of each expert [E] (used with a hot set)
  int cap_gu, cap_down;
};

// Routing (router GEMM, top-k, float64 recheck) is per token, so it runs once per span of whole chunks, up to
// kRouteSpan tokens (or max_chunk when larger); the expert-major GEMMs and the combine run per chunk.
constexpr int kRouteSpan = 16384;

struct Shape {
  int H, E, I, k, Is, C, span_cap, slots, window;
  int hot;     // offloaded experts kept resident in slots [slots, slots + hot) (moe_prefill_set_hot_experts)
  int fmt;     // routed expert weights: kFmtBf16, kFmtMxfp8 or kFmtNvfp4
  int cb64;    // bytes per 64 weights along K: 128 (bf16), 64 (MXFP8 codes), 32 (NVFP4 codes)
  int gu_half, gu_half_s, bn_down, bn_router_narrow, bn_router_wide;
  int nt_gu, nt_gu_s, nt_down;
};

Shape make_shape(const moe_dims& d) {
  Shape s;
  s.H = d.hidden;
  s.E = d.n_experts;
  s.I = d.inter;
  s.k = d.top_k;
  s.Is = d.shared_inter;
  s.C = d.max_chunk;
  s.span_cap = std::max(s.C, kRouteSpan);
  s.slots = d.offload_slots;
  s.hot = 0;
  s.fmt = kFmtBf16;
  s.cb64 = 128;
  s.window = d.offload_slots / 2;
  s.gu_half = (s.I % 128 == 0) ? 128 : 64;
  s.gu_half_s = (s.Is % 128 == 0) ? 128 : 64;
  s.bn_down = (s.H % 256 == 0) ? 256 : (s.H % 128 == 0 ? 128 : 64);
  s.bn_router_narrow = std::min(64, s.E);  // short spans: narrow N tiles give more CTAs
  s.bn_router_wide = std::min(256, s.E);   // long spans: wide N tiles read each X tile fewer times
  s.nt_gu = s.I / s.gu_half;
  s.nt_gu_s = s.Is > 0 ? s.Is / s.gu_half_s : 0;
  s.nt_down = s.H / s.bn_down;
  return s;
}

Layout make_layout(const Shape& s) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  const size_t C = static_cast<size_t>(s.C), E = s.E, k = s.k, H = s.H, I = s.I, Is = s.Is;
  const size_t SP = static_cast<size_t>(s.span_cap);
  const size_t R = C * k;
  const size_t nblk = (C + 31) / 32;
  const size_t mts = (C + kBlockM - 1) / kBlockM;
  const size_t routed_mt = (R + kBlockM - 1) / kBlockM + std::min(E, R);
  L.cap_gu = static_cast<int>(routed_mt * s.nt_gu + (Is > 0 ? mts * s.nt_gu_s : 0));
  L.cap_down = static_cast<int>(routed_mt * s.nt_down + (Is > 0 ? mts * s.nt_down : 0));
  L.hdr = take(sizeof(WsHeader));
  L.wnorm = take(E * 4);
  L.logits = take(SP * E * 4);
  L.topk_id = take(SP * k * 4);
  L.topk_w = take(SP * k * 4);
  L.band = take(SP);
  L.band_info = take(SP * 32);
  L.masks = take(nblk * E * 4);
  L.counts = take(nblk * E * 4);
  L.base = take(nblk * E * 4);
  L.totals = take(E * 4);
  L.block_band = take(nblk * 4);
  L.offsets = take((E + 1) * 4);
  for (int b = 0; b < 2; ++b) {
    L.token_row[b] = take(C * k * 4);
    L.num_tiles[b] = take(16);
    L.tiles_gu[b] = take(static_cast<size_t>(L.cap_gu) * 16);
    L.tiles_down[b] = take(static_cast<size_t>(L.cap_down) * 16);
    L.xp[b] = take(R * H * 2);
    L.tile_base[b] = take(2 * (E + 1) * 4);
  }
  const size_t S = static_cast<size_t>(s.slots) + static_cast<size_t>(s.hot);
  L.ring_gu = take(S * 2 * I * H / 64 * s.cb64);
  L.ring_down = take(S * H * I / 64 * s.cb64);
  L.slot_map = take(s.slots > 0 ? E * 4 : 0);
  L.h = take(R * I * 2);
  L.hs = take(Is > 0 ? C * Is * 2 : 0);
  L.y = take(R * H * 4);
  L.s = take(Is > 0 ? C * H * 4 : 0);
  L.total = off;
  return L;
}

// ------------------------------------------------------------------ what a workspace holds between runs
// Layers may share one workspace (one scratch for a whole stack of layers, or the library's built-in array of
// moe_prefill_run_noalloc), so what a run leaves in it for later runs belongs to the workspace, not to a plan: the
// hot set's slots and the slot map (valid only for the plan, and the hot-set version of that plan, that staged
// them), the ring's first window staged ahead by moe_prefill_prefetch, and the points on the GPU after which the
// last run no longer reads the ring (for a prefetch that overlaps the end of that run). One record per (device,
// workspace address), created by the first run or prefetch that names the workspace.
struct RingSig {  // where the ring's first window lies in a plan's layout
  size_t ring_gu, ring_down, gu_bytes, dn_bytes;
  int window;
  bool operator==(const RingSig& o) const {
    return ring_gu == o.ring_gu && ring_down == o.ring_down && gu_bytes == o.gu_bytes && dn_bytes == o.dn_bytes &&
           window == o.window;
  }
};

struct WsRecord {
  uint64_t owner = 0;        // id of the plan whose run was enqueued last on the workspace (0: none known)
  uint64_t owner_hot = 0;    // that plan's hot-set version at that run (the hot slots and slot map it left)
  bool owner_offload = false;
  RingSig owner_ring{};      // that run's ring layout (offloaded plans)
  cudaEvent_t ev_end = nullptr;    // end of that run (all of its work, every stream)
  cudaEvent_t ev_ring0 = nullptr;  // that run's last release of the ring's first half (offloaded plans)
  bool ring0_recorded = false;
  bool pf_pending = false;   // a prefetch was enqueued and no run has consumed or dropped it yet
  uint64_t pf_plan = 0, pf_hot = 0;
  cudaEvent_t ev_prefetch = nullptr;
  uint64_t last_use = 0;
  ~WsRecord() {
    for (cudaEvent_t e : {ev_end, ev_ring0, ev_prefetch})
      if (e) cudaEventDestroy(e);
  }
};

std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, std::shared_ptr<WsRecord>> g_ws;
uint64_t g_ws_clock = 0;
constexpr size_t kMaxWsRecords = 256;
std::atomic<uint64_t> g_plan_ids{0};

// The record of `workspace` on `device` (created, with its events, when new). With more than kMaxWsRecords
// workspaces the least recently used record without a pending prefetch is dropped after its events have completed,
// so forgetting it loses nothing: a later run on that workspace restages what it needs.
moe_status ws_record(int device, const void* workspace, std::shared_ptr<WsRecord>* out) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(workspace));
  auto it = g_ws.find(key);
  if (it == g_ws.end()) {
    if (g_ws.size() >= kMaxWsRecords) {
      auto victim = g_ws.end();
      for (auto j = g_ws.begin(); j != g_ws.end(); ++j)
        if (!j->second->pf_pending && (victim == g_ws.end() || j->second->last_use < victim->second->last_use))
          victim = j;
      if (victim != g_ws.end()) {
        for (cudaEvent_t e : {victim->second->ev_end, victim->second->ev_ring0})
          if (e && cudaEventSynchronize(e) != cudaSuccess)
            return fail(MOE_ERR_CUDA, "workspace record eviction: %s", cudaGetErrorString(cudaGetLastError()));
        g_ws.erase(victim);
      }
    }
    auto rec = std::make_shared<WsRecord>();
    for (cudaEvent_t* e : {&rec->ev_end, &rec->ev_ring0, &rec->ev_prefetch}) {
      const cudaError_t ce = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
      if (ce != cudaSuccess) return fail(MOE_ERR_CUDA, "workspace record events: %s", cudaGetErrorString(ce));
    }
    it = g_ws.emplace(key, std::move(rec)).first;
  }
  it->second->last_use = ++g_ws_clock;
  *out = it->second;
  return MOE_OK;
}

}  // namespace

struct moe_plan {
  moe_dims d;
  Shape sh;
  Layout lay;
  int device, num_sms;
  const void *w_router, *w_gu, *w_down, *ws_gu, *ws_down;
  CUtensorMap tm_wr_narrow, tm_wr_wide, tm_wgu, tm_wdown, tm_wsgu, tm_wsdown;
  CUtensorMap tm_wgu3, tm_wsgu3;  // the gate/up weights (or codes) as gate/up halves (one load per tile and K step)
  CUtensorMap tm_sgu, tm_sdown;   // block-scaled weights: their scale planes, one load per tile and K step
  // descriptors of workspace-resident activations, cached per workspace pointer
  const void* ws_cached = nullptr;
  CUtensorMap tm_xp[2], tm_h, tm_hs, tm_ring_gu, tm_ring_down, tm_ring_gu3;
  // The expert GEMMs on CTA pairs (grouped_pair_kernel): bf16 weights whose I, I_s are multiples of 128 and H of
  // 256. pair_ok: the plan's dimensions allow it; pairs: which projections use it (MOE_PAIRS_* bits, set by
  // moe_prefill_set_cta_pairs; the gate/up projection by default). Its descriptors: gate/up weights as gate/up
  // halves, down weights in 128-row boxes, token rows in 128-row and 32-row boxes.
  bool pair_ok = false;
  int32_t pairs = 0;
  CUtensorMap tm_wgu_p, tm_wdown_p, tm_wsgu_p, tm_wsdown_p;
  CUtensorMap tm_xp_p[2], tm_h_p, tm_hs_p, tm_ring_gu_p, tm_ring_down_p;
  CUtensorMap tm_xp_ps[2], tm_h_ps, tm_hs_ps;  // token rows in 32-row boxes (tiles of at most 64 tokens)
  CUtensorMap tm_y, tm_s;  // fp32 outputs of the down projection (routed rows, shared expert rows)
  // offloaded experts: w_gu / w_down are pinned host banks; the copy stream fills the ring (see moe_prefill_run)
  bool offload = false;
  // device-accessible addresses of the pinned banks (null when the device cannot read them directly)
  const void* bank_gu_dev = nullptr;
  const void* bank_down_dev = nullptr;
  int32_t offload_copy = MOE_OFFLOAD_COPY_ALL;
  // resident hot set of offloaded experts: slot of every expert (e % S, or S + its place in the set), and whether
  // the set still has to be staged into the cached workspace
  std::vector<int32_t> slot_map_host;
  uint64_t id = 0;            // unique over the process (a workspace record names the plan that last ran on it)
  uint64_t hot_version = 1;   // changes with every moe_prefill_set_hot_experts (new set, new ring layout)
  // MXFP8 routed experts: w_gu / w_down hold E4M3 codes, these their E8M0 scales ([E][K/32][rows])
  const uint8_t* w_gu_scale = nullptr;
  const uint8_t* w_down_scale = nullptr;
  cudaStream_t own_copy = nullptr;
  cudaEvent_t ev_copy[2] = {}, ev_rel[2] = {};
  // Each chunk's member lists (count, scan, permute) run on a side stream so that they overlap the previous chunk's
  // GEMMs; events order the two streams (see moe_prefill_run).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_span = nullptr, ev_join = nullptr, ev_ready[2] = {}, ev_down = nullptr,
              ev_comb = nullptr;
  // runs from host buffers (moe_prefill_run_host): activations move on their own stream, chunk by chunk
  cudaStream_t host_io = nullptr;
  cudaEvent_t ev_x_head = nullptr, ev_x_rest = nullptr;
  uint64_t timeout_ns = 2000000000ull;
  int32_t combine_mode = MOE_COMBINE_F32;
  int64_t launches = 0;
  bool profiling = false;
  struct Timed {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Timed> pending;
  std::vector<cudaEvent_t> pool;
  double ms[MOE_KERNEL_KINDS] = {};
  int64_t counts[MOE_KERNEL_KINDS] = {};
};

namespace {

moe_status validate_dims(const moe_dims* d) {
  if (!d) return fail(MOE_ERR_INVALID_ARG, "dims is NULL");
  if (d->hidden <= 0 || d->n_experts <= 0 || d->inter <= 0 || d->top_k <= 0 || d->shared_inter < 0 ||
      d->max_chunk <= 0 || d->offload_slots < 0)
    return fail(MOE_ERR_INVALID_ARG, "dims must be positive (shared_inter, offload_slots >= 0)");
  if (d->hidden % 64 || d->inter % 64 || d->shared_inter % 64)
    return fail(MOE_ERR_UNSUPPORTED, "hidden, inter and shared_inter must be multiples of 64");
  if (d->n_experts % 16 || d->n_experts > 1024)
    return fail(MOE_ERR_UNSUPPORTED, "n_experts must be a multiple of 16 and at most 1024 (got %d)", d->n_experts);
  if (d->top_k > d->n_experts || d->top_k > 32)
    return fail(MOE_ERR_UNSUPPORTED, "top_k must be at most min(n_experts, 32) (got %d)", d->top_k);
  if (d->renormalize != 1) return fail(MOE_ERR_UNSUPPORTED, "only renormalize == 1 is implemented");
  if (d->offload_slots != 0) {
    const int S = d->offload_slots;
    if (S < 2 || S % 2 || S > d->n_experts || d->n_experts % (S / 2))
      return fail(MOE_ERR_UNSUPPORTED,
                  "offload_slots must be even, at most n_experts, and half of it must divide n_experts (got %d)", S);
  }
  const int64_t R = static_cast<int64_t>(d->max_chunk) * d->top_k;
  if (R >= (1ll << 30) || static_cast<int64_t>(d->n_experts) * d->hidden >= (1ll << 31) ||
      static_cast<int64_t>(d->n_experts) * 2 * d->inter >= (1ll << 31))
    return fail(MOE_ERR_UNSUPPORTED, "sizes exceed 32-bit row indices");
  return MOE_OK;
}

void record_kernel(moe_plan* p, int kind, cudaStream_t st, bool before) {
  if (!p->profiling) return;
  auto take = [&]() {
    cudaEvent_t e;
    if (!p->pool.empty()) {
      e = p->pool.back();
      p->pool.pop_back();
    } else if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
    }
    return e;
  };
  if (before) {
    moe_plan::Timed t{kind, take(), take()};
    if (t.a) cudaEventRecord(t.a, st);
    p->pending.push_back(t);
  } else if (!p->pending.empty() && p->pending.back().b) {
    cudaEventRecord(p->pending.back().b, st);
  }
}

// Brackets the launches of one kernel kind (timing events when profiling) and counts the kernels launched.
struct LaunchScope {
  moe_plan* p;
  int kind;
  cudaStream_t st;
  int kernels;
  LaunchScope(moe_plan* p_, int kind_, cudaStream_t st_, int kernels_ = 1)
      : p(p_), kind(kind_), st(st_), kernels(kernels_) {
    record_kernel(p, kind, st, true);
  }
  ~LaunchScope() {
    record_kernel(p, kind, st, false);
    p->launches += kernels;
  }
};

moe_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MOE_OK;
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

namespace moe {
// Helpers for noalloc.cu (internal linkage names, not part of the C ABI).
size_t plan_workspace_bytes(moe_plan_t plan) { return plan ? plan->lay.total : 0; }
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace moe

namespace {

moe_status plan_impl(const moe_dims* dims, const void* w_router, const void* w_gu, const void* w_down,
                     const void* ws_gu, const void* ws_down, const void* gu_scale, const void* down_scale, int fmt,
                     size_t* workspace_bytes, moe_plan_t* plan) {
  if (plan) *plan = nullptr;
  moe_status st = validate_dims(dims);
  if (st != MOE_OK) return st;
  const bool mxfp8 = fmt != kFmtBf16;  // any block-scaled format
  if (mxfp8 && (!gu_scale || !down_scale)) return fail(MOE_ERR_INVALID_ARG, "both scale arrays are needed");
  if (mxfp8 && (!aligned16(gu_scale) || !aligned16(down_scale)))
    return fail(MOE_ERR_INVALID_ARG, "scale arrays must be 16-byte aligned");
  if (!workspace_bytes || !plan) return fail(MOE_ERR_INVALID_ARG, "workspace_bytes and plan must not be NULL");
  if (!w_router || !w_gu || !w_down) return fail(MOE_ERR_INVALID_ARG, "weight pointers must not be NULL");
  if (dims->shared_inter > 0 && (!ws_gu || !ws_down))
    return fail(MOE_ERR_INVALID_ARG, "shared_inter > 0 needs ws_gu and ws_down");
  if (dims->shared_inter == 0 && (ws_gu || ws_down))
    return fail(MOE_ERR_INVALID_ARG, "ws_gu / ws_down given but shared_inter == 0");
  for (const void* q : {w_router, w_gu, w_down, ws_gu, ws_down})
    if (q && !aligned16(q)) return fail(MOE_ERR_INVALID_ARG, "weight pointers must be 16-byte aligned");
  int device = 0, num_sms = 0;
  st = check_device(&device, &num_sms);
  if (st != MOE_OK) return st;

  moe_plan* p = new moe_plan();
  p->id = ++g_plan_ids;
  p->d = *dims;
  p->sh = make_shape(*dims);
  p->sh.fmt = fmt;
  p->sh.cb64 = fmt == kFmtNvfp4 ? 32 : (fmt == kFmtMxfp8 ? 64 : 128);
  p->lay = make_layout(p->sh);
  p->device = device;
  p->num_sms = num_sms;
  p->w_router = w_router;
  p->w_gu = w_gu;
  p->w_down = w_down;
  p->ws_gu = ws_gu;
  p->ws_down = ws_down;
  p->w_gu_scale = static_cast<const uint8_t*>(gu_scale);
  p->w_down_scale = static_cast<const uint8_t*>(down_scale);
  const Shape& s = p->sh;
  if (mxfp8) {
    // the GEMM streams the scales with bulk copies: they stay in device memory, also when the codes are offloaded
    for (const void* q : {gu_scale, down_scale}) {
      cudaPointerAttributes a;
      if (cudaPointerGetAttributes(&a, q) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        delete p;
        return fail(MOE_ERR_INVALID_ARG, "MXFP8 scale arrays must be in device memory");
      }
    }
  }
  p->offload = dims->offload_slots > 0;
  if (p->offload) {
    // the expert banks stay in host memory: they must be page-locked so the copy engines can read them
    const void* dev_addr[2] = {nullptr, nullptr};
    int qi = 0;
    for (const void* q : {w_gu, w_down}) {
      cudaPointerAttributes a;
      if (cudaPointerGetAttributes(&a, q) != cudaSuccess || a.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        delete p;
        return fail(MOE_ERR_INVALID_ARG, "offload_slots > 0 needs w_gu and w_down in pinned host memory");
      }
      dev_addr[qi++] = a.devicePointer;
    }
    // kernels can stage only the routed experts when the device reads the banks directly (16-byte aligned)
    if (dev_addr[0] && dev_addr[1] && aligned16(dev_addr[0]) && aligned16(dev_addr[1])) {
      p->bank_gu_dev = dev_addr[0];
      p->bank_down_dev = dev_addr[1];
      p->offload_copy = MOE_OFFLOAD_COPY_ROUTED;
    }
  }
  st = encode_bf16_2d(&p->tm_wr_narrow, w_router, s.E, s.H, s.bn_router_narrow);
  if (st == MOE_OK) st = encode_bf16_2d(&p->tm_wr_wide, w_router, s.E, s.H, s.bn_router_wide);
  if (st == MOE_OK && !p->offload && !mxfp8)
    st = encode_bf16_2d(&p->tm_wgu, w_gu, static_cast<uint64_t>(s.E) * 2 * s.I, s.H, s.gu_half);
  if (st == MOE_OK && !p->offload && !mxfp8)
    st = encode_bf16_2d(&p->tm_wdown, w_down, static_cast<uint64_t>(s.E) * s.H, s.I, s.bn_down);
  if (st == MOE_OK && mxfp8 && !p->offload)
    st = encode_u8_2d(&p->tm_wgu, w_gu, static_cast<uint64_t>(s.E) * 2 * s.I, s.H / 64 * s.cb64, s.gu_half, s.cb64);
  if (st == MOE_OK && mxfp8 && !p->offload)
    st = encode_u8_2d(&p->tm_wdown, w_down, static_cast<uint64_t>(s.E) * s.H, s.I / 64 * s.cb64, s.bn_down, s.cb64);
  if (st == MOE_OK && s.Is > 0) st = encode_bf16_2d(&p->tm_wsgu, ws_gu, 2ull * s.Is, s.H, s.gu_half_s);
  if (st == MOE_OK && s.Is > 0) st = encode_bf16_2d(&p->tm_wsdown, ws_down, s.H, s.Is, s.bn_down);
  if (st == MOE_OK && !p->offload && !mxfp8) st = encode_bf16_halves(&p->tm_wgu3, w_gu, s.E, s.I, s.H, s.gu_half);
  if (st == MOE_OK && !p->offload && mxfp8)
    st = encode_u8_halves(&p->tm_wgu3, w_gu, s.E, s.I, static_cast<uint64_t>(s.H) / 64 * s.cb64, s.gu_half, s.cb64);
  if (mxfp8) {
    // scale planes: one per scale block along K (MXFP8: 32 weights, NVFP4: 16), 64 / block blocks per K step
    const uint32_t blocks = fmt == kFmtNvfp4 ? 4u : 2u;
    if (st == MOE_OK)
      st = encode_u8_scales_gu(&p->tm_sgu, gu_scale, s.E, static_cast<uint64_t>(s.H) / 64 * blocks, s.I, s.gu_half,
                               blocks);
    if (st == MOE_OK)
      st = encode_u8_scales(&p->tm_sdown, down_scale, s.E, static_cast<uint64_t>(s.I) / 64 * blocks, s.H, s.bn_down,
                            blocks);
  }
  if (st == MOE_OK && s.Is > 0) st = encode_bf16_halves(&p->tm_wsgu3, ws_gu, 1, s.Is, s.H, s.gu_half_s);
  p->pair_ok = fmt == kFmtBf16 && s.I % 128 == 0 && s.Is % 128 == 0 && s.H % 256 == 0 && pair_cluster_slots() > 0;
  if (st == MOE_OK && p->pair_ok && !p->offload)
    st = encode_bf16_halves_kb(&p->tm_wgu_p, w_gu, s.E, s.I, s.H, kPairWBoxRows, kPairKB);
  if (st == MOE_OK && p->pair_ok && !p->offload)
    st = encode_bf16_rows_kb(&p->tm_wdown_p, w_down, static_cast<uint64_t>(s.E) * s.H, s.I, kPairDownBoxRows, kPairKB);
  if (st == MOE_OK && p->pair_ok && s.Is > 0)
    st = encode_bf16_halves_kb(&p->tm_wsgu_p, ws_gu, 1, s.Is, s.H, kPairWBoxRows, kPairKB);
  if (st == MOE_OK && p->pair_ok && s.Is > 0)
    st = encode_bf16_rows_kb(&p->tm_wsdown_p, ws_down, s.H, s.Is, kPairDownBoxRows, kPairKB);
  p->pairs = p->pair_ok ? MOE_PAIRS_GATE_UP : 0;
  if (st == MOE_OK) {
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&p->side, cudaStreamNonBlocking, hi);
    if (e == cudaSuccess && p->offload) e = cudaStreamCreateWithFlags(&p->own_copy, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->host_io, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&p->ev_fork,    &p->ev_span,    &p->ev_join,    &p->ev_ready[0], &p->ev_ready[1],
                          &p->ev_down,    &p->ev_comb,    &p->ev_copy[0], &p->ev_copy[1], &p->ev_rel[0],
                          &p->ev_rel[1],  &p->ev_x_head,  &p->ev_x_rest};
    for (cudaEvent_t* ev : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) st = fail(MOE_ERR_CUDA, "stream/event creation: %s", cudaGetErrorString(e));
  }
  if (st != MOE_OK) {
    moe_prefill_destroy(p);
    return st;
  }
  *workspace_bytes = p->lay.total;
  *plan = p;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_prefill_plan(const moe_dims* dims, const void* w_router, const void* w_gu, const void* w_down,
                            const void* ws_gu, const void* ws_down, size_t* workspace_bytes, moe_plan_t* plan) {
  return plan_impl(dims, w_router, w_gu, w_down, ws_gu, ws_down, nullptr, nullptr, kFmtBf16, workspace_bytes, plan);
}

moe_status moe_prefill_plan_mxfp8(const moe_dims* dims, const void* w_router, const uint8_t* w_gu_codes,
                                  const uint8_t* w_gu_scales, const uint8_t* w_down_codes,
                                  const uint8_t* w_down_scales, const void* ws_gu, const void* ws_down,
                                  size_t* workspace_bytes, moe_plan_t* plan) {
  if (plan) *plan = nullptr;
  if (!w_gu_scales || !w_down_scales) return fail(MOE_ERR_INVALID_ARG, "scale arrays must not be NULL");
  return plan_impl(dims, w_router, w_gu_codes, w_down_codes, ws_gu, ws_down, w_gu_scales, w_down_scales, kFmtMxfp8,
                   workspace_bytes, plan);
}

moe_status moe_prefill_plan_nvfp4(const moe_dims* dims, const void* w_router, const uint8_t* w_gu_codes,
                                  const uint8_t* w_gu_scales, const uint8_t* w_down_codes,
                                  const uint8_t* w_down_scales, const void* ws_gu, const void* ws_down,
                                  size_t* workspace_bytes, moe_plan_t* plan) {
  if (plan) *plan = nullptr;
  if (!w_gu_scales || !w_down_scales) return fail(MOE_ERR_INVALID_ARG, "scale arrays must not be NULL");
  return plan_impl(dims, w_router, w_gu_codes, w_down_codes, ws_gu, ws_down, w_gu_scales, w_down_scales, kFmtNvfp4,
                   workspace_bytes, plan);
}

}  // extern "C"

namespace {

// Host buffers of moe_prefill_run_host: X rows are copied into the device staging rows before the routing and the
// member lists that read them, out rows back once their chunk's combine has written them.
struct HostIO {
  const void* x_host;
  void* out_host;
};

moe_status run_impl(moe_plan_t p, const void* x, int64_t T, int32_t chunk, void* workspace, size_t workspace_bytes,
                    void* out, int32_t* topk_id, float* topk_w, int32_t* expert_offsets, int32_t* row_token,
                    moe_stream_t compute_, moe_stream_t copy, const HostIO* hio) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0");
  if (chunk < 1 || chunk > p->d.max_chunk)
    return fail(MOE_ERR_INVALID_ARG, "chunk must be in [1, max_chunk=%d] (got %d)", p->d.max_chunk, chunk);
  if (copy && !p->offload) return fail(MOE_ERR_INVALID_ARG, "copy stream must be NULL for resident weights");
  if (T >= (1ll << 31)) return fail(MOE_ERR_UNSUPPORTED, "T must be below 2^31");
  if (T == 0) return MOE_OK;
  if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x and out must not be NULL");
  if (!workspace || workspace_bytes < p->lay.total)
    return fail(MOE_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", p->lay.total, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  for (const void* q : {x, static_cast<const void*>(out), static_cast<const void*>(topk_id),
                        static_cast<const void*>(topk_w), static_cast<const void*>(expert_offsets),
                        static_cast<const void*>(row_token)})
    if (q && (reinterpret_cast<uintptr_t>(q) & 3u) != 0) return fail(MOE_ERR_INVALID_ARG, "pointers need 4-byte alignment");
  if (!aligned16(x) || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev != p->device) return fail(MOE_ERR_INVALID_ARG, "current device %d differs from the plan's %d", dev, p->device);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(compute_);
  const Shape& s = p->sh;
  const Layout& L = p->lay;
  char* ws = static_cast<char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.hdr);
  float* wnorm = reinterpret_cast<float*>(ws + L.wnorm);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  uint8_t* band = reinterpret_cast<uint8_t*>(ws + L.band);
  cudaStream_t side = p->side;
  cudaStream_t cp = copy ? reinterpret_cast<cudaStream_t>(copy) : p->own_copy;  // offloaded experts only
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
  uint16_t* hs = reinterpret_cast<uint16_t*>(ws + L.hs);
  float* y = reinterpret_cast<float*>(ws + L.y);
  float* sbuf = reinterpret_cast<float*>(ws + L.s);

  // activation descriptors: X per run; workspace-resident ones cached per workspace address
  CUtensorMap tm_x, tm_x_p, tm_x_ps;
  moe_status rc = encode_bf16_2d(&tm_x, x, static_cast<uint64_t>(T), s.H, kABoxRows);
  if (rc == MOE_OK && p->pair_ok)
    rc = encode_bf16_rows_kb(&tm_x_p, x, static_cast<uint64_t>(T), s.H, kPairTBoxRows, kPairKB);
  if (rc == MOE_OK && p->pair_ok)
    rc = encode_bf16_rows_kb(&tm_x_ps, x, static_cast<uint64_t>(T), s.H, kPairTBoxRowsSmall, kPairKB);
  if (rc != MOE_OK) return rc;
  if (p->ws_cached != workspace) {
    const uint64_t R = static_cast<uint64_t>(s.C) * s.k;
    rc = encode_bf16_2d(&p->tm_xp[0], ws + L.xp[0], R, s.H, kABoxRows);
    if (rc == MOE_OK) rc = encode_bf16_2d(&p->tm_xp[1], ws + L.xp[1], R, s.H, kABoxRows);
    if (rc == MOE_OK) rc = encode_bf16_2d(&p->tm_h, h, R, s.I, kABoxRows);
    if (rc == MOE_OK && s.Is > 0) rc = encode_bf16_2d(&p->tm_hs, hs, s.C, s.Is, kABoxRows);
    if (rc == MOE_OK) rc = encode_f32_out(&p->tm_y, y, R, s.H, s.H);
    if (rc == MOE_OK && s.Is > 0) rc = encode_f32_out(&p->tm_s, sbuf, s.C, s.H, s.H);
    // ring slots hold bf16 weights or codes
    const uint64_t ring_slots = static_cast<uint64_t>(s.slots) + static_cast<uint64_t>(s.hot);
    if (rc == MOE_OK && p->offload && s.fmt == kFmtBf16)
      rc = encode_bf16_2d(&p->tm_ring_gu, ws + L.ring_gu, ring_slots * 2 * s.I, s.H, s.gu_half);
    if (rc == MOE_OK && p->offload && s.fmt == kFmtBf16)
      rc = encode_bf16_2d(&p->tm_ring_down, ws + L.ring_down, ring_slots * s.H, s.I, s.bn_down);
    if (rc == MOE_OK && p->offload && s.fmt != kFmtBf16)
      rc = encode_u8_2d(&p->tm_ring_gu, ws + L.ring_gu, ring_slots * 2 * s.I, s.H / 64 * s.cb64, s.gu_half, s.cb64);
    if (rc == MOE_OK && p->offload && s.fmt != kFmtBf16)
      rc = encode_u8_2d(&p->tm_ring_down, ws + L.ring_down, ring_slots * s.H, s.I / 64 * s.cb64, s.bn_down, s.cb64);
    if (rc == MOE_OK && p->offload && s.fmt == kFmtBf16)
      rc = encode_bf16_halves(&p->tm_ring_gu3, ws + L.ring_gu, ring_slots, s.I, s.H, s.gu_half);
    if (rc == MOE_OK && p->offload && s.fmt != kFmtBf16)
      rc = encode_u8_halves(&p->tm_ring_gu3, ws + L.ring_gu, ring_slots, s.I, static_cast<uint64_t>(s.H) / 64 * s.cb64,
                            s.gu_half, s.cb64);
    for (int b = 0; b < 2 && p->pair_ok; ++b) {
      const uint32_t box = b == 0 ? kPairTBoxRows : kPairTBoxRowsSmall;
      CUtensorMap* xp = b == 0 ? p->tm_xp_p : p->tm_xp_ps;
      if (rc == MOE_OK) rc = encode_bf16_rows_kb(&xp[0], ws + L.xp[0], R, s.H, box, kPairKB);
      if (rc == MOE_OK) rc = encode_bf16_rows_kb(&xp[1], ws + L.xp[1], R, s.H, box, kPairKB);
      if (rc == MOE_OK) rc = encode_bf16_rows_kb(b == 0 ? &p->tm_h_p : &p->tm_h_ps, h, R, s.I, box, kPairKB);
      if (rc == MOE_OK && s.Is > 0)
        rc = encode_bf16_rows_kb(b == 0 ? &p->tm_hs_p : &p->tm_hs_ps, hs, s.C, s.Is, box, kPairKB);
    }
    if (rc == MOE_OK && p->pair_ok && p->offload)
      rc = encode_bf16_halves_kb(&p->tm_ring_gu_p, ws + L.ring_gu, ring_slots, s.I, s.H, kPairWBoxRows, kPairKB);
    if (rc == MOE_OK && p->pair_ok && p->offload)
      rc = encode_bf16_rows_kb(&p->tm_ring_down_p, ws + L.ring_down, ring_slots * s.H, s.I, kPairDownBoxRows, kPairKB);
    if (rc != MOE_OK) {
      p->ws_cached = nullptr;
      return rc;
    }
    p->ws_cached = workspace;
  }

  // What this workspace holds from earlier runs (of any plan) and which copies are in flight into it.
  std::shared_ptr<WsRecord> rec;
  rc = ws_record(p->device, workspace, &rec);
  if (rc != MOE_OK) return rc;
  const RingSig my_ring{L.ring_gu, L.ring_down, static_cast<size_t>(2) * s.I * s.H / 64 * s.cb64,
                        static_cast<size_t>(s.H) * s.I / 64 * s.cb64, s.window};
  // The hot set's slots and the slot map are valid only if this plan, with this hot set, was the last to run here.
  const bool stage_hot = p->offload && s.hot > 0 && !(rec->owner == p->id && rec->owner_hot == p->hot_version);
  // A prefetch into this workspace is consumed if this plan, with this hot set, made it: only the first window's
  // GEMMs wait for its copies. Any other run drops it, and all of that run's work waits for its copies.
  const bool pf_waiting = rec->pf_pending;
  const bool prefetched = pf_waiting && p->offload && rec->pf_plan == p->id && rec->pf_hot == p->hot_version;
  rec->pf_pending = false;
  // From here on the run may leave the workspace part-written: until it is fully enqueued, the record names no owner.
  rec->owner = 0;
  rec->ring0_recorded = false;

  // The side stream starts after everything the caller enqueued on `compute` before this call, and every return
  // after this point first makes `compute` wait for all side work (join), so the run is one unit on `compute`.
  if (pf_waiting && !prefetched) rc = cuda_status(cudaStreamWaitEvent(st, rec->ev_prefetch, 0), "prefetch wait");
  if (rc == MOE_OK) rc = cuda_status(cudaEventRecord(p->ev_fork, st), "fork event");
  if (rc == MOE_OK) rc = cuda_status(cudaStreamWaitEvent(side, p->ev_fork, 0), "fork wait");
  if (rc == MOE_OK && p->offload) rc = cuda_status(cudaStreamWaitEvent(cp, p->ev_fork, 0), "fork wait");
  if (rc == MOE_OK && hio) rc = cuda_status(cudaStreamWaitEvent(p->host_io, p->ev_fork, 0), "fork wait");
  if (rc != MOE_OK) return rc;
  auto join = [&](moe_status r) {
    if (cudaEventRecord(p->ev_join, side) == cudaSuccess) cudaStreamWaitEvent(st, p->ev_join, 0);
    if (p->offload && cudaEventRecord(p->ev_join, cp) == cudaSuccess) cudaStreamWaitEvent(st, p->ev_join, 0);
    if (hio && cudaEventRecord(p->ev_join, p->host_io) == cudaSuccess) cudaStreamWaitEvent(st, p->ev_join, 0);
    const bool ended = cudaEventRecord(rec->ev_end, st) == cudaSuccess;
    if (r == MOE_OK && ended) {
      rec->owner = p->id;
      rec->owner_hot = p->hot_version;
      rec->owner_offload = p->offload;
      rec->owner_ring = my_ring;
    }
    return r;
  };
  // The hot set: upload the slot map (read by the GEMMs and the staging kernel) ahead of everything this run
  // enqueues, and stage the hot experts into their slots on the copy stream ahead of the first window's copies
  // (every GEMM waits for a window's copies, so for these too).
  if (stage_hot) {
    rc = cuda_status(cudaMemcpyAsync(ws + L.slot_map, p->slot_map_host.data(), sizeof(int32_t) * s.E,
                                     cudaMemcpyHostToDevice, st),
                     "slot map upload");
    const size_t gu_bytes = my_ring.gu_bytes;
    const size_t dn_bytes = my_ring.dn_bytes;
    for (int e = 0; rc == MOE_OK && e < s.E; ++e) {
      const int32_t slot = p->slot_map_host[e];
      if (slot < s.slots) continue;
      rc = cuda_status(cudaMemcpyAsync(ws + L.ring_gu + static_cast<size_t>(slot) * gu_bytes,
                                       static_cast<const char*>(p->w_gu) + static_cast<size_t>(e) * gu_bytes,
                                       gu_bytes, cudaMemcpyHostToDevice, cp),
                       "hot expert gate/up copy");
      if (rc == MOE_OK)
        rc = cuda_status(cudaMemcpyAsync(ws + L.ring_down + static_cast<size_t>(slot) * dn_bytes,
                                         static_cast<const char*>(p->w_down) + static_cast<size_t>(e) * dn_bytes,
                                         dn_bytes, cudaMemcpyHostToDevice, cp),
                         "hot expert down copy");
    }
    if (rc != MOE_OK) return join(rc);
  }
  // A span is routed in two segments: its first chunk (on `compute`, before anything else) and the rest (on the
  // side stream, beside the first chunk's GEMMs). With host buffers the span's X rows go to the device in the same
  // two copies, each with its event, so each segment starts once its own rows have landed.
  const int64_t span = static_cast<int64_t>(chunk) * std::max(1, s.span_cap / chunk);
  auto segments = [&](int64_t a0, int64_t* n1, int64_t* n2) {
    const int64_t n_span = std::min<int64_t>(span, T - a0);
    *n1 = std::min<int64_t>(chunk, n_span);
    *n2 = n_span - *n1;
  };
  const size_t row_bytes = static_cast<size_t>(s.H) * 2;
  auto copy_x_span = [&](int64_t a0) -> moe_status {
    int64_t n1, n2;
    segments(a0, &n1, &n2);
    const char* src = static_cast<const char*>(hio->x_host) + a0 * row_bytes;
    char* dst = static_cast<char*>(const_cast<void*>(x)) + a0 * row_bytes;
    moe_status r2 = MOE_OK;
    const int64_t lens[2] = {n1, n2};
    cudaEvent_t evs[2] = {p->ev_x_head, p->ev_x_rest};
    for (int i = 0; i < 2 && r2 == MOE_OK; ++i) {
      if (lens[i] > 0)
        r2 = cuda_status(cudaMemcpyAsync(dst, src, lens[i] * row_bytes, cudaMemcpyHostToDevice, p->host_io), "X copy");
      if (r2 == MOE_OK) r2 = cuda_status(cudaEventRecord(evs[i], p->host_io), "X event");
      dst += lens[i] * row_bytes;
      src += lens[i] * row_bytes;
    }
    return r2;
  };
  if (hio) {
    rc = copy_x_span(0);
    if (rc != MOE_OK) return join(rc);
  }

  {
    LaunchScope ls(p, MOE_KERNEL_NORMS, st);
    rc = cuda_status(launch_router_norms(static_cast<const uint16_t*>(p->w_router), s.E, s.H, wnorm, hdr, st),
                     "router norms launch");
  }
  if (rc != MOE_OK) return join(rc);

  // |fp32 tensor-core logit - exact| <= one ulp per 16-wide K step of a partial sum bounded by ||x|| ||w||
  const float tau_coef = static_cast<float>(s.H / 16 + 1) * 0x1p-23f;
  int64_t chunk_idx = 0;
  for (int64_t s0 = 0; s0 < T; s0 += span) {
    // ---------------------------------------------------------------- routing of the span's tokens
    const int ns = static_cast<int>(std::min<int64_t>(span, T - s0));
    int32_t* span_ids = topk_id ? topk_id + s0 * s.k : reinterpret_cast<int32_t*>(ws + L.topk_id);
    float* span_w = topk_w ? topk_w + s0 * s.k : reinterpret_cast<float*>(ws + L.topk_w);

    // Routing of the tokens [g0, g0 + ng) of this span on stream `rs`: router GEMM (logits, fp32), then top-k with
    // weights and the float64 recheck of tokens whose fp32 selection is not certain. Results land at the tokens'
    // offsets in the span buffers.
    auto route = [&](int64_t g0, int ng, cudaStream_t rs) -> moe_status {
      const int64_t off = g0 - s0;
      const bool wide = ng >= 4096;
      const int bn_router = wide ? s.bn_router_wide : s.bn_router_narrow;
      const int nt_router = (s.E + bn_router - 1) / bn_router;
      GemmParams g;
      memset(&g, 0, sizeof g);
      g.tmA[0] = g.tmA[1] = tm_x;
      g.tmB[0] = g.tmB[1] = wide ? p->tm_wr_wide : p->tm_wr_narrow;
      GemmClass rc0{};
      rc0.kblocks = s.H / kBlockK;
      rc0.n_tile = bn_router;
      rc0.b_box_rows = bn_router;
      rc0.out_cols = s.E;
      rc0.out_ld = s.E;
      rc0.out = logits + off * s.E;
      rc0.out_tma = 2;  // the map's rows are the span's ng tokens
      g.cls[0] = g.cls[1] = rc0;
      {
        const moe_status r0 = encode_f32_out(&g.tmOut[0], logits + off * s.E, static_cast<uint64_t>(ng), s.E, s.E);
        if (r0 != MOE_OK) return r0;
        g.tmOut[1] = g.tmOut[0];
      }
      g.tiles = nullptr;
      g.num_tiles = nullptr;
      g.dense_m = ng;
      g.dense_n_tiles = nt_router;
      g.dense_a_row0 = static_cast<int32_t>(g0);
      g.err = &hdr->err;
      g.stall_flag = nullptr;
      g.timeout_ns = p->timeout_ns;
      moe_status r2;
      {
        const int tiles = ((ng + kBlockM - 1) / kBlockM) * nt_router;
        LaunchScope ls(p, MOE_KERNEL_ROUTER, rs);
        r2 = cuda_status(launch_grouped_gemm(g, kEpiF32, std::min(p->num_sms, tiles), rs), "router GEMM launch");
      }
      if (r2 != MOE_OK) return r2;
      RouteParams r;
      r.logits = logits + off * s.E;
      r.x = static_cast<const uint16_t*>(x) + g0 * s.H;
      r.w_router = static_cast<const uint16_t*>(p->w_router);
      r.wnorm = wnorm;
      r.hdr = hdr;
      r.n = ng;
      r.E = s.E;
      r.H = s.H;
      r.k = s.k;
      r.tau_coef = tau_coef;
      r.topk_id = span_ids + off * s.k;
      r.topk_w = span_w + off * s.k;
      r.band_flag = band + off;
      r.band_info = reinterpret_cast<BandInfo*>(ws + L.band_info);
      r.band_grid = p->num_sms;
      LaunchScope ls(p, MOE_KERNEL_TOPK, rs, 2);  // top-k, then the float64 recheck of flagged tokens
      return cuda_status(launch_topk(r, rs), "top-k launch");
    };

    // The span's first chunk is routed on `compute` before anything else; the rest of the span is routed on the
    // side stream after the first chunk's member lists, beside the first chunk's GEMMs, and the member lists of
    // later chunks follow it on that stream. Routing is per token: splitting it changes no result.
    // The previous span's combines and member lists read this span's buffers (logits, top-k): wait for them.
    rc = cuda_status(cudaStreamWaitEvent(st, p->ev_comb, 0), "span start wait");
    if (rc == MOE_OK && hio) rc = cuda_status(cudaStreamWaitEvent(st, p->ev_x_head, 0), "X wait");
    if (rc != MOE_OK) return join(rc);
    int64_t n1, n2;
    segments(s0, &n1, &n2);
    const int head = static_cast<int>(n1);
    rc = route(s0, head, st);
    if (rc == MOE_OK) rc = cuda_status(cudaEventRecord(p->ev_span, st), "span event");
    if (rc != MOE_OK) return join(rc);

    // Per chunk c: member lists L(c) on the side stream, GEMMs G(c) on `compute`, combine C(c) on the side stream.
    // Enqueue order: L(first); then for each chunk G(c), L(c+1), C(c). On the GPU, L(c+1) and C(c) overlap G(c)
    // and G(c+1). Buffer set c%2 (gathered rows, tile lists, token_row) is reused by chunk c+2: L(c+2) follows
    // C(c) on the side stream, and C(c) waits for G(c). The down GEMM of chunk c waits for C(c-1) (y, s reuse).
    auto lists = [&](int64_t c0, int64_t cidx) -> moe_status {
      const int n = static_cast<int>(std::min<int64_t>(chunk, T - c0));
      const int par = static_cast<int>(cidx & 1);
      PermuteParams q;
      q.topk_id = span_ids + (c0 - s0) * s.k;
      q.band_flag = band + (c0 - s0);
      q.x = static_cast<const uint16_t*>(x) + c0 * s.H;
      q.n = n;
      q.E = s.E;
      q.H = s.H;
      q.k = s.k;
      q.nblk = (n + 31) / 32;
      q.token0 = c0;
      q.masks = reinterpret_cast<uint32_t*>(ws + L.masks);
      q.counts = reinterpret_cast<int32_t*>(ws + L.counts);
      q.block_band = reinterpret_cast<int32_t*>(ws + L.block_band);
      q.base = reinterpret_cast<int32_t*>(ws + L.base);
      q.totals = reinterpret_cast<int32_t*>(ws + L.totals);
      q.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
      q.offsets_out = expert_offsets ? expert_offsets + cidx * (s.E + 1) : nullptr;
      q.token_row = reinterpret_cast<int32_t*>(ws + L.token_row[par]);
      q.row_token = row_token ? row_token + c0 * s.k : nullptr;
      q.xp = reinterpret_cast<uint16_t*>(ws + L.xp[par]);
      q.hdr = hdr;
      q.tiles_gu = reinterpret_cast<int4*>(ws + L.tiles_gu[par]);
      q.tiles_down = reinterpret_cast<int4*>(ws + L.tiles_down[par]);
      q.num_tiles = reinterpret_cast<int32_t*>(ws + L.num_tiles[par]);
      q.tile_base = reinterpret_cast<int32_t*>(ws + L.tile_base[par]);
      q.cap_gu = L.cap_gu;
      q.cap_down = L.cap_down;
      q.nt_gu = s.nt_gu;
      q.nt_down = s.nt_down;
      q.nt_gu_shared = s.nt_gu_s;
      q.nt_down_shared = s.Is > 0 ? s.nt_down : 0;
      q.pair_gu = (p->pairs & MOE_PAIRS_GATE_UP) ? 1 : 0;
      q.pair_dn = (p->pairs & MOE_PAIRS_DOWN) ? 1 : 0;
      moe_status r2;
      {
        LaunchScope ls(p, MOE_KERNEL_COUNT, side);
        r2 = cuda_status(launch_count(q, side), "count launch");
      }
      if (r2 != MOE_OK) return r2;
      {
        LaunchScope ls(p, MOE_KERNEL_SCAN, side, 2);
        r2 = cuda_status(launch_block_bases(q, side), "block bases launch");
        if (r2 == MOE_OK) r2 = cuda_status(launch_scan_tiles(q, side), "scan launch");
      }
      if (r2 != MOE_OK) return r2;
      {
        LaunchScope ls(p, MOE_KERNEL_PERMUTE, side);
        r2 = cuda_status(launch_permute(q, side), "permute launch");
      }
      if (r2 != MOE_OK) return r2;
      return cuda_status(cudaEventRecord(p->ev_ready[par], side), "ready event");
    };

    // Offloaded experts: the ring's halves hold windows of W consecutive experts; window [e0, e0 + W) goes to slots
    // e0 % S ... (one copy for its gate/up weights, one for its down weights) once the copy stream has seen the
    // release of the window that last used those slots.
    auto copy_window = [&](int64_t cidx, int e0) -> moe_status {
      const int hb = (e0 / s.window) & 1;
      const size_t slot0 = static_cast<size_t>(e0 % s.slots);
      const size_t gu_bytes = static_cast<size_t>(2) * s.I * s.H / 64 * s.cb64;
      const size_t dn_bytes = static_cast<size_t>(s.H) * s.I / 64 * s.cb64;
      moe_status r2 = cuda_status(cudaStreamWaitEvent(cp, p->ev_rel[hb], 0), "slot release wait");
      if (r2 == MOE_OK && prefetched && cidx == 0 && e0 == 0) {  // every expert of the window is already there
        r2 = cuda_status(cudaStreamWaitEvent(cp, rec->ev_prefetch, 0), "prefetch wait");
        if (r2 == MOE_OK) r2 = cuda_status(cudaEventRecord(p->ev_copy[hb], cp), "copy event");
        return r2;
      }
      if (r2 == MOE_OK && p->offload_copy == MOE_OFFLOAD_COPY_ROUTED) {
        // only the experts this chunk routes rows to, decided on the device once its member lists exist
        const int par = static_cast<int>(cidx & 1);
        r2 = cuda_status(cudaStreamWaitEvent(cp, p->ev_ready[par], 0), "member lists wait");
        RingCopyParams rp;
        rp.bank_gu = static_cast<const uint4*>(p->bank_gu_dev);
        rp.bank_down = static_cast<const uint4*>(p->bank_down_dev);
        rp.ring_gu = reinterpret_cast<uint4*>(ws + L.ring_gu);
        rp.ring_down = reinterpret_cast<uint4*>(ws + L.ring_down);
        rp.tile_base = reinterpret_cast<const int32_t*>(ws + L.tile_base[par]);
        rp.hdr = hdr;
        rp.gu16 = static_cast<int64_t>(gu_bytes / 16);
        rp.dn16 = static_cast<int64_t>(dn_bytes / 16);
        rp.e0 = e0;
        rp.count = s.window;
        rp.slots = s.slots;
        rp.slot_map = s.hot > 0 ? reinterpret_cast<const int32_t*>(ws + L.slot_map) : nullptr;
        if (r2 == MOE_OK) r2 = cuda_status(launch_ring_copy(rp, cp), "expert staging launch");
        if (r2 == MOE_OK) ++p->launches;
        if (r2 == MOE_OK) r2 = cuda_status(cudaEventRecord(p->ev_copy[hb], cp), "copy event");
        return r2;
      }
      if (r2 == MOE_OK)
        r2 = cuda_status(cudaMemcpyAsync(ws + L.ring_gu + slot0 * gu_bytes,
                                         static_cast<const char*>(p->w_gu) + static_cast<size_t>(e0) * gu_bytes,
                                         gu_bytes * s.window, cudaMemcpyHostToDevice, cp),
                         "expert gate/up copy");
      if (r2 == MOE_OK)
        r2 = cuda_status(cudaMemcpyAsync(ws + L.ring_down + slot0 * dn_bytes,
                                         static_cast<const char*>(p->w_down) + static_cast<size_t>(e0) * dn_bytes,
                                         dn_bytes * s.window, cudaMemcpyHostToDevice, cp),
                         "expert down copy");
      if (r2 == MOE_OK) r2 = cuda_status(cudaEventRecord(p->ev_copy[hb], cp), "copy event");
      return r2;
    };

    // The grouped GEMMs of experts [e0, e1) of a chunk (all experts when the weights are resident); the range
    // of the last experts also covers the shared expert's tiles, which follow the routed ones in the lists.
    // One grouped GEMM over the tiles of experts [e0, e1) (and the shared expert's, which follow the routed ones,
    // when the range reaches the last expert). MXFP8 plans run the routed tiles in the decoding kernel and the
    // bf16 shared expert in the plain one, as a second launch on the same stream.
    auto grouped = [&](GemmParams prm, int epi, int cap, const int32_t* tb, const int32_t* n_tiles, int e0, int e1,
                       bool windowed, int kind, const char* what) -> moe_status {
      const bool q = s.fmt != kFmtBf16;
      if (!q) {
        if (windowed) {
          prm.range_lo = tb + e0;
          prm.range_hi = (e1 >= s.E) ? n_tiles : tb + e1;
        }
        LaunchScope ls(p, kind, st);
        return cuda_status(launch_grouped_gemm(prm, epi, std::min(p->num_sms, cap), st), what);
      }
      const bool shared = s.Is > 0 && e1 >= s.E;
      LaunchScope ls(p, kind, st, shared ? 2 : 1);
      prm.range_lo = windowed ? tb + e0 : nullptr;
      prm.range_hi = tb + std::min(e1, s.E);
      moe_status r2 = cuda_status(launch_grouped_gemm(prm, epi, std::min(p->num_sms, cap), st, s.fmt), what);
      if (r2 == MOE_OK && shared) {
        prm.range_lo = tb + s.E;
        prm.range_hi = n_tiles;
        r2 = cuda_status(launch_grouped_gemm(prm, epi, p->num_sms, st, kFmtBf16), what);
      }
      return r2;
    };

    // The same on CTA pairs (bf16 weights only).
    auto pair_grouped = [&](PairParams prm, int epi, int cap, const int32_t* tb, const int32_t* n_tiles, int e0,
                            int e1, bool windowed, int kind, const char* what) -> moe_status {
      if (windowed) {
        prm.range_lo = tb + e0;
        prm.range_hi = (e1 >= s.E) ? n_tiles : tb + e1;
      }
      LaunchScope ls(p, kind, st);
      return cuda_status(launch_grouped_pair(prm, epi, cap, st), what);
    };

    // The grouped GEMMs of one chunk on CTA pairs: weights are the 256-row M operand, the tile's token rows
    // (gathered rows or X; h or the shared h) the N operand. Gate/up + SwiGLU:
    auto pair_gate_up = [&](int par, const int32_t* num_tiles, const int32_t* tbase, int e0, int e1,
                            bool windowed) -> moe_status {
      const int32_t* slot_map = (windowed && s.hot > 0) ? reinterpret_cast<const int32_t*>(ws + L.slot_map) : nullptr;
      PairParams gu;
      memset(&gu, 0, sizeof gu);
      gu.tmW[0] = windowed ? p->tm_ring_gu_p : p->tm_wgu_p;
      gu.tmT[0] = p->tm_xp_p[par];
      gu.tmTs[0] = p->tm_xp_ps[par];
      PairClass c_r{};
      c_r.kblocks = s.H / kBlockK;
      c_r.w_group_rows = 2 * s.I;
      c_r.w_up_offset = s.I;
      c_r.w_stream = 1;
      c_r.w_group_mod = windowed ? s.slots : 0;
      c_r.w_slot_map = slot_map;
      c_r.out = h;
      c_r.out_ld = s.I;
      gu.cls[0] = c_r;
      gu.tmW[1] = gu.tmW[0];
      gu.tmT[1] = gu.tmT[0];
      gu.tmTs[1] = gu.tmTs[0];
      gu.cls[1] = c_r;
      if (s.Is > 0) {
        gu.tmW[1] = p->tm_wsgu_p;
        gu.tmT[1] = tm_x_p;
        gu.tmTs[1] = tm_x_ps;
        PairClass c_s{};
        c_s.kblocks = s.H / kBlockK;
        c_s.w_up_offset = s.Is;
        c_s.out = hs;
        c_s.out_ld = s.Is;
        gu.cls[1] = c_s;
      }
      gu.tiles = reinterpret_cast<const int4*>(ws + L.tiles_gu[par]);
      gu.num_tiles = num_tiles;
      gu.err = &hdr->err;
      gu.timeout_ns = p->timeout_ns;
      return pair_grouped(gu, kEpiSwiGLU, L.cap_gu, tbase, num_tiles, e0, e1, windowed, MOE_KERNEL_GATE_UP,
                          "gate/up launch");
    };

    // down:
    auto pair_down = [&](int par, const int32_t* num_tiles, const int32_t* tbase, int e0, int e1,
                         bool windowed) -> moe_status {
      const int32_t* slot_map = (windowed && s.hot > 0) ? reinterpret_cast<const int32_t*>(ws + L.slot_map) : nullptr;
      PairParams dn;
      memset(&dn, 0, sizeof dn);
      dn.tmW[0] = windowed ? p->tm_ring_down_p : p->tm_wdown_p;
      dn.tmT[0] = p->tm_h_p;
      dn.tmTs[0] = p->tm_h_ps;
      PairClass d_r{};
      d_r.kblocks = s.I / kBlockK;
      d_r.w_group_rows = s.H;
      d_r.w_stream = 1;
      d_r.w_group_mod = windowed ? s.slots : 0;
      d_r.w_slot_map = slot_map;
      d_r.out = y;
      d_r.out_ld = s.H;
      dn.cls[0] = d_r;
      dn.tmW[1] = dn.tmW[0];
      dn.tmT[1] = dn.tmT[0];
      dn.tmTs[1] = dn.tmTs[0];
      dn.cls[1] = d_r;
      if (s.Is > 0) {
        dn.tmW[1] = p->tm_wsdown_p;
        dn.tmT[1] = p->tm_hs_p;
        dn.tmTs[1] = p->tm_hs_ps;
        PairClass d_s{};
        d_s.kblocks = s.Is / kBlockK;
        d_s.out = sbuf;
        d_s.out_ld = s.H;
        dn.cls[1] = d_s;
      }
      dn.tiles = reinterpret_cast<const int4*>(ws + L.tiles_down[par]);
      dn.num_tiles = num_tiles + 1;
      dn.err = &hdr->err;
      dn.timeout_ns = p->timeout_ns;
      return pair_grouped(dn, kEpiF32, L.cap_down, tbase + (s.E + 1), num_tiles + 1, e0, e1, windowed,
                          MOE_KERNEL_DOWN, "down launch");
    };

    // The grouped GEMMs of one chunk on single CTAs: the tile's rows are the 128-row M operand, the weights the N
    // operand. Gate/up + SwiGLU:
    auto single_gate_up = [&](int par, const int32_t* num_tiles, const int32_t* tbase, int e0, int e1,
                              bool windowed) -> moe_status {
      GemmParams gu;
      memset(&gu, 0, sizeof gu);
      gu.tmA[0] = p->tm_xp[par];
      gu.tmB[0] = windowed ? p->tm_ring_gu : p->tm_wgu;
      gu.tmBg[0] = windowed ? p->tm_ring_gu3 : p->tm_wgu3;
      GemmClass c_r{};
      c_r.kblocks = s.H / kBlockK;
      c_r.n_tile = 2 * s.gu_half;
      c_r.b_box_rows = s.gu_half;
      c_r.b_group_rows = 2 * s.I;
      c_r.b_up_offset = s.I;
      c_r.out_cols = s.I;
      c_r.b_stream = 1;
      c_r.b_group_mod = windowed ? s.slots : 0;
      c_r.b_slot_map = (windowed && s.hot > 0) ? reinterpret_cast<const int32_t*>(ws + L.slot_map) : nullptr;
      c_r.out_ld = s.I;
      c_r.out = h;
      c_r.b_scale = p->w_gu_scale;
      gu.tmS[0] = gu.tmS[1] = p->tm_sgu;
      gu.cls[0] = c_r;
      if (s.Is > 0) {
        gu.tmA[1] = tm_x;
        gu.tmB[1] = p->tm_wsgu;
        gu.tmBg[1] = p->tm_wsgu3;
        GemmClass c_s{};
        c_s.kblocks = s.H / kBlockK;
        c_s.n_tile = 2 * s.gu_half_s;
        c_s.b_box_rows = s.gu_half_s;
        c_s.b_group_rows = 0;
        c_s.b_up_offset = s.Is;
        c_s.out_cols = s.Is;
        c_s.b_stream = 0;
        c_s.b_group_mod = 0;
        c_s.out_ld = s.Is;
        c_s.out = hs;
        gu.cls[1] = c_s;
      } else {
        gu.tmA[1] = gu.tmA[0];
        gu.tmB[1] = gu.tmB[0];
        gu.tmBg[1] = gu.tmBg[0];
        gu.cls[1] = c_r;
      }
      gu.tiles = reinterpret_cast<const int4*>(ws + L.tiles_gu[par]);
      gu.num_tiles = num_tiles;
      gu.err = &hdr->err;
      gu.timeout_ns = p->timeout_ns;
      moe_status r2 =
          grouped(gu, kEpiSwiGLU, L.cap_gu, tbase, num_tiles, e0, e1, windowed, MOE_KERNEL_GATE_UP, "gate/up launch");
      return r2;
    };

    // down (class 0 routed h rows -> y, class 1 shared h rows -> s):
    auto single_down = [&](int par, const int32_t* num_tiles, const int32_t* tbase, int e0, int e1,
                           bool windowed) -> moe_status {
      GemmParams dn;
      memset(&dn, 0, sizeof dn);
      dn.tmA[0] = p->tm_h;
      dn.tmB[0] = windowed ? p->tm_ring_down : p->tm_wdown;
      GemmClass d_r{};
      d_r.kblocks = s.I / kBlockK;
      d_r.n_tile = s.bn_down;
      d_r.b_box_rows = s.bn_down;
      d_r.b_group_rows = s.H;
      d_r.b_up_offset = 0;
      d_r.out_cols = s.H;
      d_r.b_stream = 1;
      d_r.b_group_mod = windowed ? s.slots : 0;
      d_r.b_slot_map = (windowed && s.hot > 0) ? reinterpret_cast<const int32_t*>(ws + L.slot_map) : nullptr;
      d_r.out_ld = s.H;
      d_r.out = y;
      d_r.out_tma = 1;
      d_r.b_scale = p->w_down_scale;
      dn.tmS[0] = dn.tmS[1] = p->tm_sdown;
      dn.cls[0] = d_r;
      dn.tmOut[0] = p->tm_y;
      if (s.Is > 0) {
        dn.tmA[1] = p->tm_hs;
        dn.tmB[1] = p->tm_wsdown;
        GemmClass d_s = d_r;
        d_s.b_scale = nullptr;
        d_s.kblocks = s.Is / kBlockK;
        d_s.b_group_rows = 0;
        d_s.b_stream = 0;
        d_s.b_group_mod = 0;
        d_s.b_slot_map = nullptr;
        d_s.out = sbuf;
        dn.cls[1] = d_s;
        dn.tmOut[1] = p->tm_s;
      } else {
        dn.tmA[1] = dn.tmA[0];
        dn.tmB[1] = dn.tmB[0];
        dn.cls[1] = d_r;
        dn.tmOut[1] = dn.tmOut[0];
      }
      dn.tiles = reinterpret_cast<const int4*>(ws + L.tiles_down[par]);
      dn.num_tiles = num_tiles + 1;
      dn.err = &hdr->err;
      dn.timeout_ns = p->timeout_ns;
      return grouped(dn, kEpiF32, L.cap_down, tbase + (s.E + 1), num_tiles + 1, e0, e1, windowed, MOE_KERNEL_DOWN,
                     "down launch");
    };

    auto gemms = [&](int64_t cidx, int e0, int e1, bool last_chunk) -> moe_status {
      const int par = static_cast<int>(cidx & 1);
      const int32_t* num_tiles = reinterpret_cast<const int32_t*>(ws + L.num_tiles[par]);
      const int32_t* tbase = reinterpret_cast<const int32_t*>(ws + L.tile_base[par]);
      const bool windowed = p->offload;
      const int hb = windowed ? (e0 / s.window) & 1 : 0;
      moe_status r2 = cuda_status(cudaStreamWaitEvent(st, p->ev_ready[par], 0), "ready wait");
      if (r2 == MOE_OK && windowed) r2 = cuda_status(cudaStreamWaitEvent(st, p->ev_copy[hb], 0), "copy wait");
      if (r2 != MOE_OK) return r2;
      // 6. grouped gate/up + SwiGLU (class 0 routed on the gathered rows, class 1 shared on the chunk's X rows)
      r2 = (p->pairs & MOE_PAIRS_GATE_UP) ? pair_gate_up(par, num_tiles, tbase, e0, e1, windowed)
                                          : single_gate_up(par, num_tiles, tbase, e0, e1, windowed);
      // 7. grouped down (class 0 routed h rows -> y, class 1 shared h rows -> s), once the previous chunk's combine
      // has read y and s
      if (r2 == MOE_OK) r2 = cuda_status(cudaStreamWaitEvent(st, p->ev_comb, 0), "combine wait");
      if (r2 == MOE_OK)
        r2 = (p->pairs & MOE_PAIRS_DOWN) ? pair_down(par, num_tiles, tbase, e0, e1, windowed)
                                         : single_down(par, num_tiles, tbase, e0, e1, windowed);
      if (r2 != MOE_OK) return r2;
      if (windowed) {
        r2 = cuda_status(cudaEventRecord(p->ev_rel[hb], st), "slot release event");
        // the run's last release of the ring's first half: a prefetch into this workspace may start after it
        if (r2 == MOE_OK && hb == 0 && last_chunk) {
          r2 = cuda_status(cudaEventRecord(rec->ev_ring0, st), "ring release event");
          if (r2 == MOE_OK) rec->ring0_recorded = true;
        }
        if (r2 != MOE_OK) return r2;
      }
      return cuda_status(cudaEventRecord(p->ev_down, st), "down event");
    };

    auto combine = [&](int64_t c0, int64_t cidx) -> moe_status {
      const int n = static_cast<int>(std::min<int64_t>(chunk, T - c0));
      const int par = static_cast<int>(cidx & 1);
      moe_status r2 = cuda_status(cudaStreamWaitEvent(side, p->ev_down, 0), "down wait");
      if (r2 != MOE_OK) return r2;
      // 8. canonical combine (float32, ascending expert id) or the float64 tree over the expert ids
      {
        LaunchScope ls(p, MOE_KERNEL_COMBINE, side);
        if (p->combine_mode == MOE_COMBINE_F64_TREE) {
          CombineTreeParams a;
          memset(&a, 0, sizeof a);
          a.y = y;
          a.w = span_w + (c0 - s0) * s.k;
          a.token_row = reinterpret_cast<const int32_t*>(ws + L.token_row[par]);
          a.topk_id = span_ids + (c0 - s0) * s.k;
          a.s = s.Is > 0 ? sbuf : nullptr;
          a.out = static_cast<uint16_t*>(out) + c0 * s.H;
          a.n = n;
          a.k = s.k;
          a.H = s.H;
          a.lo = 0;
          a.block_log2 = ceil_log2(s.E);
          r2 = cuda_status(launch_combine_tree(a, true, side), "combine launch");
        } else {
          r2 = cuda_status(launch_combine(y, span_w + (c0 - s0) * s.k,
                                          reinterpret_cast<const int32_t*>(ws + L.token_row[par]),
                                          s.Is > 0 ? sbuf : nullptr, n, s.k, s.H,
                                          static_cast<uint16_t*>(out) + c0 * s.H, side),
                           "combine launch");
        }
      }
      if (r2 != MOE_OK) return r2;
      r2 = cuda_status(cudaEventRecord(p->ev_comb, side), "combine event");
      if (r2 == MOE_OK && hio) {
        // the chunk's out rows back to the host once its combine has written them
        r2 = cuda_status(cudaStreamWaitEvent(p->host_io, p->ev_comb, 0), "out wait");
        if (r2 == MOE_OK)
          r2 = cuda_status(cudaMemcpyAsync(static_cast<char*>(hio->out_host) + c0 * row_bytes,
                                           static_cast<const char*>(out) + c0 * row_bytes, n * row_bytes,
                                           cudaMemcpyDeviceToHost, p->host_io),
                           "out copy");
      }
      return r2;
    };

    rc = cuda_status(cudaStreamWaitEvent(side, p->ev_span, 0), "span wait");
    if (rc == MOE_OK) rc = lists(s0, chunk_idx);
    if (rc == MOE_OK && hio) rc = cuda_status(cudaStreamWaitEvent(side, p->ev_x_rest, 0), "X wait");
    if (rc == MOE_OK && n2 > 0) rc = route(s0 + n1, static_cast<int>(n2), side);
    // both waits of this span are enqueued: the next span's X rows may now reuse the events
    if (rc == MOE_OK && hio && s0 + span < T) rc = copy_x_span(s0 + span);
    if (rc != MOE_OK) return join(rc);
    for (int64_t c0 = s0; c0 < s0 + ns; c0 += chunk, ++chunk_idx) {
      const bool last_chunk = c0 + chunk >= T;
      if (!p->offload) {
        rc = gemms(chunk_idx, 0, s.E, last_chunk);
      } else {
        for (int e0 = 0; rc == MOE_OK && e0 < s.E; e0 += s.window) {
          rc = copy_window(chunk_idx, e0);
          if (rc == MOE_OK) rc = gemms(chunk_idx, e0, e0 + s.window, last_chunk);
        }
      }
      if (rc == MOE_OK && c0 + chunk < s0 + ns) rc = lists(c0 + chunk, chunk_idx + 1);
      if (rc == MOE_OK) rc = combine(c0, chunk_idx);
      if (rc != MOE_OK) return join(rc);
    }
  }
  // The side stream's last combine joins `compute` here: the run ends after all of its work.
  return join(MOE_OK);
}

}  // namespace

extern "C" {

moe_status moe_prefill_run(moe_plan_t p, const void* x, int64_t T, int32_t chunk, void* workspace,
                           size_t workspace_bytes, void* out, int32_t* topk_id, float* topk_w,
                           int32_t* expert_offsets, int32_t* row_token, moe_stream_t compute, moe_stream_t copy) {
  return run_impl(p, x, T, chunk, workspace, workspace_bytes, out, topk_id, topk_w, expert_offsets, row_token,
                  compute, copy, nullptr);
}

moe_status moe_prefill_run_host(moe_plan_t p, const void* x_host, int64_t T, int32_t chunk, void* workspace,
                                size_t workspace_bytes, void* x_dev, void* out_dev, void* out_host, int32_t* topk_id,
                                float* topk_w, int32_t* expert_offsets, int32_t* row_token, moe_stream_t compute,
                                moe_stream_t copy) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T > 0) {
    if (!x_host || !out_host || !x_dev || !out_dev)
      return fail(MOE_ERR_INVALID_ARG, "x_host, out_host, x_dev and out_dev must not be NULL");
    for (const void* q : {x_host, static_cast<const void*>(out_host)}) {
      cudaPointerAttributes a;
      if (cudaPointerGetAttributes(&a, q) != cudaSuccess || a.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return fail(MOE_ERR_INVALID_ARG, "x_host and out_host must be pinned host memory");
      }
    }
    if (!aligned16(x_host) || !aligned16(out_host))
      return fail(MOE_ERR_INVALID_ARG, "x_host and out_host must be 16-byte aligned");
  }
  const HostIO hio{x_host, out_host};
  return run_impl(p, x_dev, T, chunk, workspace, workspace_bytes, out_dev, topk_id, topk_w, expert_offsets,
                  row_token, compute, copy, &hio);
}

moe_status moe_prefill_combine(const float* y, const float* w, const int32_t* token_row, const float* s, int64_t n,
                               int32_t k, int32_t H, void* out, moe_stream_t stream) {
  if (n < 0 || k < 1 || k > 32 || H <= 0 || H % 4 != 0)
    return fail(MOE_ERR_INVALID_ARG, "need n >= 0, 1 <= k <= 32, H a positive multiple of 4");
  if (n >= (1ll << 31)) return fail(MOE_ERR_UNSUPPORTED, "n must be below 2^31");
  if (n == 0) return MOE_OK;
  if (!y || !w || !token_row || !out) return fail(MOE_ERR_INVALID_ARG, "y, w, token_row and out must not be NULL");
  if (!aligned16(y) || !aligned16(out) || (s && !aligned16(s)))
    return fail(MOE_ERR_INVALID_ARG, "y, s and out must be 16-byte aligned");
  return cuda_status(launch_combine(y, w, token_row, s, n, k, H, static_cast<uint16_t*>(out),
                                    reinterpret_cast<cudaStream_t>(stream)),
                     "combine launch");
}

static moe_status check_tree_args(const float* y, const float* w, const int32_t* token_row, const int32_t* topk_id,
                                  int64_t n, int32_t k, int32_t H, int32_t n_experts) {
  if (n < 0 || k < 1 || k > 32 || H <= 0 || H % 4 != 0)
    return fail(MOE_ERR_INVALID_ARG, "need n >= 0, 1 <= k <= 32, H a positive multiple of 4");
  if (n_experts < 1 || n_experts > 1024) return fail(MOE_ERR_INVALID_ARG, "need 1 <= n_experts <= 1024");
  if (n >= (1ll << 31)) return fail(MOE_ERR_UNSUPPORTED, "n must be below 2^31");
  if (n > 0 && (!y || !w || !token_row || !topk_id))
    return fail(MOE_ERR_INVALID_ARG, "y, w, token_row and topk_id must not be NULL");
  if (n > 0 && !aligned16(y)) return fail(MOE_ERR_INVALID_ARG, "y must be 16-byte aligned");
  return MOE_OK;
}

moe_status moe_prefill_combine_partial_f64(const float* y, const float* w, const int32_t* token_row,
                                           const int32_t* topk_id, int64_t n, int32_t k, int32_t H,
                                           int32_t n_experts, int32_t n_parts, int32_t part, double* partial,
                                           moe_stream_t stream) {
  moe_status st = check_tree_args(y, w, token_row, topk_id, n, k, H, n_experts);
  if (st != MOE_OK) return st;
  const int lg = ceil_log2(n_experts);
  if (n_parts < 1 || (n_parts & (n_parts - 1)) != 0 || n_parts > (1 << lg) || part < 0 || part >= n_parts)
    return fail(MOE_ERR_INVALID_ARG, "n_parts must be a power of two <= %d and 0 <= part < n_parts", 1 << lg);
  if (n == 0) return MOE_OK;
  if (!partial || !aligned16(partial)) return fail(MOE_ERR_INVALID_ARG, "partial must be a 16-byte aligned pointer");
  CombineTreeParams a;
  memset(&a, 0, sizeof a);
  a.y = y;
  a.w = w;
  a.token_row = token_row;
  a.topk_id = topk_id;
  a.partial = partial;
  a.n = n;
  a.k = k;
  a.H = H;
  a.block_log2 = lg - ceil_log2(n_parts);
  a.lo = part << a.block_log2;
  return cuda_status(launch_combine_tree(a, false, reinterpret_cast<cudaStream_t>(stream)), "combine part launch");
}

moe_status moe_prefill_combine_finish_f64(const double* const* partials, int32_t n_parts, const float* s, int64_t n,
                                          int32_t H, void* out, float* out_f32, moe_stream_t stream) {
  if (n < 0 || H <= 0 || H % 4 != 0) return fail(MOE_ERR_INVALID_ARG, "need n >= 0 and H a positive multiple of 4");
  if (n_parts < 1 || n_parts > kMaxFinishParts || (n_parts & (n_parts - 1)) != 0)
    return fail(MOE_ERR_INVALID_ARG, "n_parts must be a power of two <= %d", kMaxFinishParts);
  if (n == 0) return MOE_OK;
  if (!partials || !out) return fail(MOE_ERR_INVALID_ARG, "partials and out must not be NULL");
  CombineFinishParams a;
  memset(&a, 0, sizeof a);
  for (int i = 0; i < n_parts; ++i) {
    if (!partials[i] || !aligned16(partials[i]))
      return fail(MOE_ERR_INVALID_ARG, "partials[%d] must be a 16-byte aligned device pointer", i);
    a.part[i] = partials[i];
  }
  if (!aligned16(out) || (s && !aligned16(s)) || (out_f32 && !aligned16(out_f32)))
    return fail(MOE_ERR_INVALID_ARG, "s, out and out_f32 must be 16-byte aligned");
  a.s = s;
  a.out = static_cast<uint16_t*>(out);
  a.out_f32 = out_f32;
  a.count = n * H;
  a.n_parts = n_parts;
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  return cuda_status(launch_combine_finish(a, sms, reinterpret_cast<cudaStream_t>(stream)), "combine finish launch");
}

moe_status moe_prefill_combine_f64(const float* y, const float* w, const int32_t* token_row, const int32_t* topk_id,
                                   const float* s, int64_t n, int32_t k, int32_t H, int32_t n_experts, void* out,
                                   float* out_f32, moe_stream_t stream) {
  moe_status st = check_tree_args(y, w, token_row, topk_id, n, k, H, n_experts);
  if (st != MOE_OK) return st;
  if (n == 0) return MOE_OK;
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out must not be NULL");
  if (!aligned16(out) || (s && !aligned16(s)) || (out_f32 && !aligned16(out_f32)))
    return fail(MOE_ERR_INVALID_ARG, "s, out and out_f32 must be 16-byte aligned");
  CombineTreeParams a;
  memset(&a, 0, sizeof a);
  a.y = y;
  a.w = w;
  a.token_row = token_row;
  a.topk_id = topk_id;
  a.s = s;
  a.out = static_cast<uint16_t*>(out);
  a.out_f32 = out_f32;
  a.n = n;
  a.k = k;
  a.H = H;
  a.lo = 0;
  a.block_log2 = ceil_log2(n_experts);
  return cuda_status(launch_combine_tree(a, true, reinterpret_cast<cudaStream_t>(stream)), "combine launch");
}

moe_status moe_prefill_set_offload_copy(moe_plan_t p, int32_t mode) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (!p->offload) return fail(MOE_ERR_INVALID_ARG, "the plan has no offloaded experts");
  if (mode != MOE_OFFLOAD_COPY_ALL && mode != MOE_OFFLOAD_COPY_ROUTED)
    return fail(MOE_ERR_INVALID_ARG, "unknown offload copy mode %d", mode);
  if (mode == MOE_OFFLOAD_COPY_ROUTED && !p->bank_gu_dev)
    return fail(MOE_ERR_UNSUPPORTED, "this device cannot read the pinned banks directly");
  p->offload_copy = mode;
  return MOE_OK;
}

moe_status moe_prefill_set_hot_experts(moe_plan_t p, const int32_t* hot_ids, int32_t n_hot,
                                       size_t* workspace_bytes) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (!p->offload) return fail(MOE_ERR_INVALID_ARG, "the plan has no offloaded experts");
  const int E = p->sh.E;
  if (n_hot < 0 || n_hot > E) return fail(MOE_ERR_INVALID_ARG, "n_hot must be in [0, %d] (got %d)", E, n_hot);
  if (n_hot > 0 && !hot_ids) return fail(MOE_ERR_INVALID_ARG, "hot_ids is NULL");
  std::vector<int32_t> map(static_cast<size_t>(E));
  for (int e = 0; e < E; ++e) map[e] = e % p->sh.slots;
  for (int32_t h = 0; h < n_hot; ++h) {
    const int32_t e = hot_ids[h];
    if (e < 0 || e >= E) return fail(MOE_ERR_INVALID_ARG, "hot expert id %d out of range [0, %d)", e, E);
    if (map[e] >= p->sh.slots) return fail(MOE_ERR_INVALID_ARG, "hot expert id %d given twice", e);
    map[e] = p->sh.slots + h;
  }
  p->slot_map_host.swap(map);
  p->sh.hot = n_hot;
  // a new version: the next run on any workspace stages the set again, and a prefetch made under the old layout
  // (the ring's down slots may move) is dropped by that run
  ++p->hot_version;
  p->lay = make_layout(p->sh);
  p->ws_cached = nullptr;  // new layout: re-encode the workspace maps
  if (workspace_bytes) *workspace_bytes = p->lay.total;
  return MOE_OK;
}

moe_status moe_prefill_prefetch(moe_plan_t p, void* workspace, size_t workspace_bytes, moe_stream_t copy) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (!p->offload) return fail(MOE_ERR_INVALID_ARG, "the plan has no offloaded experts");
  if (!workspace || workspace_bytes < p->lay.total)
    return fail(MOE_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", p->lay.total, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev != p->device) return fail(MOE_ERR_INVALID_ARG, "current device %d differs from the plan's %d", dev, p->device);
  const Shape& s = p->sh;
  const Layout& L = p->lay;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t cp = copy ? reinterpret_cast<cudaStream_t>(copy) : p->own_copy;
  const RingSig my_ring{L.ring_gu, L.ring_down, static_cast<size_t>(2) * s.I * s.H / 64 * s.cb64,
                        static_cast<size_t>(s.H) * s.I / 64 * s.cb64, s.window};
  std::shared_ptr<WsRecord> rec;
  moe_status r = ws_record(p->device, workspace, &rec);
  if (r != MOE_OK) return r;
  // Window 0 = experts [0, W) into slots [0, W), once nothing enqueued earlier reads or writes those bytes: after an
  // earlier prefetch into this workspace, and after the last run on it has read them. When that run's ring lies
  // where this plan's does, its last release of the ring's first half is enough (the copy overlaps its tail);
  // otherwise (another layout: the bytes may hold anything of that run) the copy waits for the end of that run.
  if (rec->pf_pending) r = cuda_status(cudaStreamWaitEvent(cp, rec->ev_prefetch, 0), "prefetch order wait");
  const bool same_ring = rec->owner != 0 && rec->owner_offload && rec->owner_ring == my_ring;
  if (r == MOE_OK && same_ring && rec->ring0_recorded) {
    r = cuda_status(cudaStreamWaitEvent(cp, rec->ev_ring0, 0), "ring release wait");
  } else if (r == MOE_OK) {
    // another layout, a run that failed part-way, or none known: wait for whatever was enqueued last on the workspace
    r = cuda_status(cudaStreamWaitEvent(cp, rec->ev_end, 0), "run end wait");
  }
  // Under another layout these copies can land on what the last run's plan keeps here (its hot slots, its slot
  // map): that plan must stage them again.
  if (r == MOE_OK && rec->owner != p->id && !same_ring) rec->owner = 0;
  bool enqueued = false;  // a copy may be in flight from here on
  if (r == MOE_OK) {
    r = cuda_status(cudaMemcpyAsync(ws + L.ring_gu, p->w_gu, my_ring.gu_bytes * s.window, cudaMemcpyHostToDevice, cp),
                    "prefetch gate/up copy");
    enqueued = true;
  }
  if (r == MOE_OK)
    r = cuda_status(cudaMemcpyAsync(ws + L.ring_down, p->w_down, my_ring.dn_bytes * s.window, cudaMemcpyHostToDevice,
                                    cp),
                    "prefetch down copy");
  if (enqueued) {
    // the record's event covers every copy enqueued so far; a failed prefetch stays pending (later runs on the
    // workspace wait for it) but no run consumes it
    const moe_status re = cuda_status(cudaEventRecord(rec->ev_prefetch, cp), "prefetch event");
    if (r == MOE_OK) r = re;
    rec->pf_pending = rec->pf_pending || re == MOE_OK;
    rec->pf_plan = r == MOE_OK ? p->id : 0;
    rec->pf_hot = p->hot_version;
  }
  return r;
}

moe_status moe_prefill_forget_workspace(void* workspace) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  std::shared_ptr<WsRecord> rec;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    auto it = g_ws.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(workspace)));
    if (it == g_ws.end()) return MOE_OK;
    rec = it->second;
    g_ws.erase(it);
  }
  // the copies and runs the record knows of finish before the caller may reuse the memory
  for (cudaEvent_t e : {rec->ev_end, rec->ev_ring0, rec->ev_prefetch}) CUDA_TRY(cudaEventSynchronize(e));
  return MOE_OK;
}

moe_status moe_prefill_set_combine(moe_plan_t p, int32_t mode) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (mode != MOE_COMBINE_F32 && mode != MOE_COMBINE_F64_TREE)
    return fail(MOE_ERR_INVALID_ARG, "unknown combine mode %d", mode);
  p->combine_mode = mode;
  return MOE_OK;
}

moe_status moe_prefill_set_cta_pairs(moe_plan_t p, int32_t which) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (which & ~(MOE_PAIRS_GATE_UP | MOE_PAIRS_DOWN)) return fail(MOE_ERR_INVALID_ARG, "unknown bits in %d", which);
  if (which && !p->pair_ok)
    return fail(MOE_ERR_UNSUPPORTED, "CTA pairs need bf16 expert weights, inter and shared_inter multiples of 128, "
                                     "hidden a multiple of 256 and room for a cluster of two CTAs");
  p->pairs = which;
  return MOE_OK;
}

int32_t moe_prefill_cta_pairs(moe_plan_t p) { return p ? p->pairs : 0; }

moe_status moe_prefill_check(void* workspace, moe_stream_t stream) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int32_t err = 0;
  CUDA_TRY(cudaMemcpy(&err, workspace, sizeof err, cudaMemcpyDeviceToHost));
  if (err == 0) return MOE_OK;
  const int32_t zero = 0;
  CUDA_TRY(cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice));
  const int kind = err & 0xFF, site = (err >> 8) & 0xFF, block = (err >> 16) & 0xFFFF;
  if (kind == kDevErrTimeout)
    return fail(MOE_ERR_DEVICE_TIMEOUT, "device wait gave up (site %d, block %d, word 0x%08x)", site, block, err);
  return fail(MOE_ERR_DEVICE_BOUNDS, "device bounds check failed (site %d, index %d, word 0x%08x)", site, block, err);
}

moe_status moe_prefill_run_stats(void* workspace, moe_stream_t stream, int32_t* stats, int32_t n_stats) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (n_stats < 0 || (n_stats > 0 && !stats)) return fail(MOE_ERR_INVALID_ARG, "stats array missing");
  CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  WsHeader hdr;
  CUDA_TRY(cudaMemcpy(&hdr, workspace, sizeof hdr, cudaMemcpyDeviceToHost));
  const int32_t all[MOE_STATS_COUNT] = {hdr.chunks_done,       hdr.band_tokens,       hdr.band_levels[0],
                                        hdr.band_levels[1],   hdr.band_levels[2],   hdr.band_levels[3],
                                        hdr.experts_copied, hdr.experts_skipped, hdr.experts_hot};
  for (int32_t i = 0; i < n_stats; ++i) stats[i] = i < MOE_STATS_COUNT ? all[i] : 0;
  return MOE_OK;
}

void moe_prefill_destroy(moe_plan_t p) {
  if (!p) return;
  if (p->host_io) cudaStreamDestroy(p->host_io);
  for (cudaEvent_t e : {p->ev_x_head, p->ev_x_rest}) if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : {p->ev_fork, p->ev_span, p->ev_join, p->ev_ready[0], p->ev_ready[1], p->ev_down, p->ev_comb,
                        p->ev_copy[0], p->ev_copy[1], p->ev_rel[0], p->ev_rel[1]})
    if (e) cudaEventDestroy(e);
  if (p->side) cudaStreamDestroy(p->side);
  if (p->own_copy) cudaStreamDestroy(p->own_copy);
  for (auto& t : p->pending) {
    if (t.a) cudaEventDestroy(t.a);
    if (t.b) cudaEventDestroy(t.b);
  }
  for (cudaEvent_t e : p->pool) cudaEventDestroy(e);
  delete p;
}

const char* moe_prefill_last_error(void) { return g_last_error.c_str(); }

moe_status moe_prefill_set_profiling(moe_plan_t p, int32_t enable) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  p->profiling = enable != 0;
  return MOE_OK;
}

moe_status moe_prefill_kernel_times(moe_plan_t p, double* ms, int64_t* launches) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  moe_status st = MOE_OK;
  for (auto& t : p->pending) {
    if (t.a && t.b) {
      cudaError_t e = cudaEventSynchronize(t.b);
      float el = 0.0f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&el, t.a, t.b);
      if (e != cudaSuccess && st == MOE_OK) st = fail(MOE_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
      p->ms[t.kind] += el;
      p->counts[t.kind] += 1;
    }
    if (t.a) p->pool.push_back(t.a);
    if (t.b) p->pool.push_back(t.b);
  }
  p->pending.clear();
  for (int i = 0; i < MOE_KERNEL_KINDS; ++i) {
    if (ms) ms[i] = p->ms[i];
    if (launches) launches[i] = p->counts[i];
    p->ms[i] = 0.0;
    p->counts[i] = 0;
  }
  return st;
}

moe_status moe_prefill_kernel_trace(moe_plan_t p, int32_t* kinds, float* start_ms, float* end_ms, int32_t capacity,
                                    int32_t* count) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (capacity < 0 || (capacity > 0 && (!kinds || !start_ms || !end_ms)) || !count)
    return fail(MOE_ERR_INVALID_ARG, "output arrays missing");
  moe_status st = MOE_OK;
  int32_t n = 0;
  cudaEvent_t origin = nullptr;
  for (auto& t : p->pending) {
    if (t.a && t.b) {
      cudaError_t e = cudaEventSynchronize(t.b);
      if (!origin) origin = t.a;
      float t0 = 0.0f, t1 = 0.0f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&t0, origin, t.a);
      if (e == cudaSuccess) e = cudaEventElapsedTime(&t1, origin, t.b);
      if (e != cudaSuccess && st == MOE_OK) st = fail(MOE_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
      if (n < capacity) {
        kinds[n] = t.kind;
        start_ms[n] = t0;
        end_ms[n] = t1;
      }
      ++n;
    }
  }
  for (auto& t : p->pending) {
    if (t.a) p->pool.push_back(t.a);
    if (t.b) p->pool.push_back(t.b);
  }
  p->pending.clear();
  *count = n;
  return st;
}

int64_t moe_prefill_launch_count(moe_plan_t p) { return p ? p->launches : 0; }

moe_status moe_prefill_set_wait_timeout(moe_plan_t p, uint64_t timeout_ns) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (timeout_ns == 0) return fail(MOE_ERR_INVALID_ARG, "timeout must be positive");
  p->timeout_ns = timeout_ns;
  return MOE_OK;
}

moe_status moe_prefill_debug_gemm(const void* a, const void* b, void* c, int32_t m, int32_t n, int32_t k_dim,
                                  int32_t epilogue, int32_t* err_word, const int32_t* stall_flag,
                                  uint64_t timeout_ns, moe_stream_t stream) {
  if (!a || !b || !c || !err_word) return fail(MOE_ERR_INVALID_ARG, "a, b, c and err_word must not be NULL");
  if (m < 1 || n < 1 || k_dim < 64 || k_dim % 64) return fail(MOE_ERR_INVALID_ARG, "need m, n >= 1, k_dim % 64 == 0");
  if (epilogue != kEpiF32 && epilogue != kEpiSwiGLU) return fail(MOE_ERR_INVALID_ARG, "epilogue must be 0 or 1");
  if (epilogue == kEpiF32 && n % 16) return fail(MOE_ERR_UNSUPPORTED, "epilogue 0 needs n % 16 == 0");
  if (epilogue == kEpiSwiGLU && n % 64) return fail(MOE_ERR_UNSUPPORTED, "epilogue 1 needs n % 64 == 0");
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return fail(MOE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  int device = 0, num_sms = 0;
  moe_status st = check_device(&device, &num_sms);
  if (st != MOE_OK) return st;
  GemmParams g;
  memset(&g, 0, sizeof g);
  GemmClass cl{};
  cl.kblocks = k_dim / kBlockK;
  cl.b_group_rows = 0;
  cl.out_cols = n;
  cl.b_stream = 0;
  cl.b_group_mod = 0;
  cl.out_ld = n;
  cl.out = c;
  int n_tiles;
  if (epilogue == kEpiF32) {
    cl.n_tile = std::min(256, n);
    cl.b_box_rows = cl.n_tile;
    cl.b_up_offset = 0;
    n_tiles = (n + cl.n_tile - 1) / cl.n_tile;
    st = encode_bf16_2d(&g.tmB[0], b, n, k_dim, cl.b_box_rows);
    cl.out_tma = 2;  // TMA stores, clipped at the map's m rows and n columns
    if (st == MOE_OK) st = encode_f32_out(&g.tmOut[0], c, m, n, n);
    g.tmOut[1] = g.tmOut[0];
  } else {
    const int half = (n % 128 == 0) ? 128 : 64;
    cl.n_tile = 2 * half;
    cl.b_box_rows = half;
    cl.b_up_offset = n;
    n_tiles = n / half;
    st = encode_bf16_2d(&g.tmB[0], b, 2ull * n, k_dim, half);
    if (st == MOE_OK) st = encode_bf16_halves(&g.tmBg[0], b, 1, n, k_dim, half);
    g.tmBg[1] = g.tmBg[0];
  }
  if (st == MOE_OK) st = encode_bf16_2d(&g.tmA[0], a, m, k_dim, kABoxRows);
  if (st != MOE_OK) return st;
  g.tmA[1] = g.tmA[0];
  g.tmB[1] = g.tmB[0];
  g.cls[0] = g.cls[1] = cl;
  g.tiles = nullptr;
  g.dense_m = m;
  g.dense_n_tiles = n_tiles;
  g.dense_a_row0 = 0;
  g.err = err_word;
  g.stall_flag = stall_flag;
  g.timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
  const int tiles = ((m + kBlockM - 1) / kBlockM) * n_tiles;
  return cuda_status(launch_grouped_gemm(g, epilogue, std::min(num_sms, tiles), reinterpret_cast<cudaStream_t>(stream)),
                     "debug GEMM launch");
}

// Tiles of the pair kernel for one dense GEMM: m token rows as one group (pair_tile_count(m) tiles of
// pair_tile_width(m) rows) times the weight blocks (F32: n / 256; SwiGLU: n / 128).
size_t moe_prefill_debug_gemm_pairs_scratch(int32_t m, int32_t n, int32_t epilogue) {
  if (m < 1 || n < 1 || (epilogue != kEpiF32 && epilogue != kEpiSwiGLU)) return 0;
  const size_t tiles = static_cast<size_t>(pair_tile_count(m)) * (epilogue == kEpiF32 ? n / 256 : n / 128);
  return 16 * (tiles + 1);
}

moe_status moe_prefill_debug_gemm_pairs(const void* a, const void* b, void* c, int32_t m, int32_t n, int32_t k_dim,
                                        int32_t epilogue, void* scratch, size_t scratch_bytes, int32_t* err_word,
                                        const int32_t* stall_flag, uint64_t timeout_ns, moe_stream_t stream) {
  if (!a || !b || !c || !err_word || !scratch)
    return fail(MOE_ERR_INVALID_ARG, "a, b, c, scratch and err_word must not be NULL");
  if (epilogue != kEpiF32 && epilogue != kEpiSwiGLU) return fail(MOE_ERR_INVALID_ARG, "epilogue must be 0 or 1");
  if (m < 1 || k_dim < 128 || k_dim % 128) return fail(MOE_ERR_INVALID_ARG, "need m >= 1, k_dim % 128 == 0");
  if ((epilogue == kEpiF32 && (n < 256 || n % 256)) || (epilogue == kEpiSwiGLU && (n < 128 || n % 128)))
    return fail(MOE_ERR_UNSUPPORTED, "the pair kernel needs n % 256 == 0 (epilogue 0) or n % 128 == 0 (epilogue 1)");
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(scratch))
    return fail(MOE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const size_t need = moe_prefill_debug_gemm_pairs_scratch(m, n, epilogue);
  if (scratch_bytes < need) return fail(MOE_ERR_WORKSPACE, "scratch needs %zu bytes", need);
  int device = 0, num_sms = 0;
  moe_status st = check_device(&device, &num_sms);
  if (st != MOE_OK) return st;
  if (pair_cluster_slots() <= 0) return fail(MOE_ERR_UNSUPPORTED, "no room for a cluster of two CTAs");
  const int width = pair_tile_width(m), mt = pair_tile_count(m);
  const int nblocks = epilogue == kEpiF32 ? n / 256 : n / 128;
  const int ntiles = mt * nblocks;
  std::vector<int4> host(static_cast<size_t>(ntiles) + 1);
  host[0] = make_int4(ntiles, 0, 0, 0);
  for (int wb = 0; wb < nblocks; ++wb)
    for (int i = 0; i < mt; ++i)
      host[1 + static_cast<size_t>(wb) * mt + i] =
          make_int4(wb << 16, i * width, std::min(width, m - i * width), i * width);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  st = cuda_status(cudaMemcpyAsync(scratch, host.data(), host.size() * sizeof(int4), cudaMemcpyHostToDevice, cs),
                   "tile list copy");
  if (st != MOE_OK) return st;
  PairParams prm;
  memset(&prm, 0, sizeof prm);
  if (epilogue == kEpiF32)
    st = encode_bf16_rows_kb(&prm.tmW[0], b, n, k_dim, kPairDownBoxRows, kPairKB);
  else
    st = encode_bf16_halves_kb(&prm.tmW[0], b, 1, n, k_dim, kPairWBoxRows, kPairKB);
  if (st == MOE_OK) st = encode_bf16_rows_kb(&prm.tmT[0], a, m, k_dim, kPairTBoxRows, kPairKB);
  if (st == MOE_OK) st = encode_bf16_rows_kb(&prm.tmTs[0], a, m, k_dim, kPairTBoxRowsSmall, kPairKB);
  if (st != MOE_OK) return st;
  prm.tmW[1] = prm.tmW[0];
  prm.tmT[1] = prm.tmT[0];
  prm.tmTs[1] = prm.tmTs[0];
  PairClass cl{};
  cl.kblocks = k_dim / kBlockK;
  cl.w_up_offset = n;
  cl.out = c;
  cl.out_ld = n;
  prm.cls[0] = prm.cls[1] = cl;
  prm.tiles = reinterpret_cast<const int4*>(static_cast<char*>(scratch) + 16);
  prm.num_tiles = static_cast<const int32_t*>(scratch);
  prm.err = err_word;
  prm.stall_flag = stall_flag;
  prm.timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
  return cuda_status(launch_grouped_pair(prm, epilogue, ntiles, cs), "debug pair GEMM launch");
}

}  // extern "C"
