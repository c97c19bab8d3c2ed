// Internal declarations shared by the kernels (gemm.cu, route.cu, combine.cu) and the C-ABI (moe_prefill.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// ------------------------------------------------------------------ device error word (workspace header)
// Low byte: kind; bits 8..15: role/site; bits 16..31: block index (saturated).
enum DeviceErrorKind : int32_t {
  kDevErrNone = 0,
  kDevErrTimeout = 1,   // a bounded wait on an mbarrier gave up
  kDevErrBounds = 2,    // a device-side bounds check failed (access skipped)
};
enum DeviceErrorSite : int32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpilogueFull = 4,
  kSiteStallFlag = 5,
  kSiteDrain = 6,
  kSiteRouting = 7,
  kSiteDecodeFull = 8,  // an MXFP8 decoder warp waiting for its stage
};
__host__ __device__ inline int32_t dev_error_code(int32_t kind, int32_t site, int32_t block) {
  return kind | (site << 8) | ((block > 0xFFFF ? 0xFFFF : block) << 16);
}

// Workspace header (first 256 bytes of the workspace).
struct WsHeader {
  int32_t err;                 // device error word for the most recent run
  int32_t band_tokens;         // tokens whose top-k needed the float64 recheck (this run)
  int32_t chunks_done;         // chunks processed (this run)
  int32_t pad0;
  float wnorm_max;             // max_e ||w_router[e]||_2 (upper bound)
  int32_t band_levels[4];      // flagged tokens decided by: float sums, double sums, sequential sums, many-candidate path
  int32_t experts_copied;      // offloaded experts staged into the ring (this run)
  int32_t experts_skipped;     // offloaded experts not staged: no row of their chunk was routed to them (this run)
  int32_t experts_hot;         // offloaded experts with rows in a chunk served from the resident hot set (this run)
  int32_t pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ------------------------------------------------------------------ grouped GEMM
constexpr int kBlockM = 128;        // UMMA M (rows of a tile)
constexpr int kBlockK = 64;         // bf16 elements per 128-byte swizzle row
constexpr int kStages = 4;          // smem pipeline depth
constexpr int kMaxN = 256;          // widest UMMA N (TMEM columns per accumulator)
// A rows per TMA box: a tile's rows in one box (rows past the tile are loaded and not used). A stage costs about the
// same per TMA operation whatever the box size, so fewer, larger boxes make a stage shorter.
constexpr int kABoxRows = 128;
constexpr int kGemmThreads = 192;   // warp 0 TMA, warp 1 MMA + TMEM alloc, warps 2..5 epilogue
constexpr int kStageABytes = kBlockM * kBlockK * 2;   // 16 KB
constexpr int kStageBBytes = kMaxN * kBlockK * 2;     // 32 KB
constexpr int kEpiBufBytes = 32 * 128;   // epilogue staging buffer: 32 rows x 128 B (a 32 x 32 fp32 block)
// One staging buffer per epilogue warp: a second one (overlapping a block's TMA store with the next block) measured
// no faster, and the CTA's shared memory stays at 210 KB, which leaves room on each SM for the routing and combine
// kernels that run beside the GEMMs on the other stream (at 226 KB they could not, and the gate/up launches started
// late on the SMs they held: +13% gate/up time).
constexpr int kEpiBufs = 1;
constexpr int kBarRegionBytes = 1024;    // mbarriers and slots; keeps the staging buffers 1024-byte aligned
constexpr int kGemmSmemBytes = 1024 /*align slack*/ + kStages * (kStageABytes + kStageBBytes) + kBarRegionBytes +
                               4 * kEpiBufs * kEpiBufBytes;
// Block-scaled FP8 weights (MXFP8), grouped_gemm_q_kernel: rings of activation rows (A), E4M3 codes with their
// E8M0 scales (C) and decoded bf16 B tiles (D, one per decoder group). Warps: 0 codes TMA, 1 UMMA, 2..5 epilogue,
// 6..13 two decoder groups of 4, 14 activation TMA.
constexpr int kQStagesA = 3;
constexpr int kQStagesC = 5;
constexpr int kQStagesD = 2;
constexpr int kQStageCodeBytes = kMaxN * kBlockK;  // 16 KB: up to 256 rows x 64 codes
constexpr int kQStageScaleBytes = 4 * kMaxN;       // up to four scale blocks (NVFP4: 16-wide) x 256 rows
constexpr int kGemmThreadsQ = 15 * 32;
constexpr int kGemmSmemBytesQ = 1024 /*align slack*/ + kQStagesA * kStageABytes + kQStagesD * kStageBBytes +
                                kQStagesC * (kQStageCodeBytes + kQStageScaleBytes) + kBarRegionBytes +
                                4 * kEpiBufs * kEpiBufBytes;

enum Epilogue : int { kEpiF32 = 0, kEpiSwiGLU = 1 };

static_assert(kGemmSmemBytes <= 215040 && kGemmSmemBytesQ <= 232448, "shared memory per CTA");

// One operand class of a grouped GEMM launch (class 0: routed experts, class 1: shared expert).
struct GemmClass {
  int32_t kblocks;        // K / 64
  int32_t n_tile;         // UMMA N = TMEM columns used by a tile
  int32_t b_box_rows;     // rows per B TMA box (SwiGLU: gate half = up half = n_tile/2; F32: n_tile)
  int32_t b_group_rows;   // B rows per group (expert): row base of group e is e * b_group_rows
  int32_t b_up_offset;    // SwiGLU: row offset of the up half inside a group (= I), else 0
  int32_t out_cols;       // valid output columns (masks a ragged last N tile)
  int32_t b_stream;       // 1: honour the tile's stream bit (expert weights); 0: never use the evict-first policy
  int32_t b_group_mod;    // > 0: B holds a ring of b_group_mod groups and group e lives in slot e % b_group_mod
  int64_t out_ld;         // output row stride in elements
  void* out;              // F32: float*, SwiGLU: bf16*
  int32_t out_tma;        // F32: 0 plain stores; 1 full 32-row slabs through GemmParams::tmOut[cls] (partial slabs
                          // stored directly: rows past a tile belong to other tiles); 2 every slab through the map
                          // (its row bound is the valid rows, so TMA clips the rest)
  int32_t pad_;
  const uint8_t* b_scale; // quantised B: scales [G][K/block][b_group_rows] (one plane per scale block);
                          // nullptr: B is bf16
  const int32_t* b_slot_map;  // b_group_mod > 0 with a hot set: slot of each group [G] (a ring slot e % b_group_mod
                              // or a hot slot >= b_group_mod); nullptr: slot e % b_group_mod
};

// Tile record: x = group | (cls << 15) | (n_idx << 16) | (stream << 31); y = first A row; z = valid rows (1..128);
// w = first out row. stream = 1 marks a tile whose B tile no other tile of the launch reads (its expert has one M
// tile): the B loads then use an evict-first L2 policy.
struct GemmParams {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  CUtensorMap tmBg[2];        // SwiGLU: the fused gate/up weights (bf16, or the codes of block-scaled weights) as
                              // (K, I, 2 x groups), box 64 (or a code row's step bytes) x b_box_rows x 2: a tile's
                              // gate rows and up rows in one load
  CUtensorMap tmS[2];         // block-scaled weights: the scale planes, uint8. SwiGLU: (row in half I, half 2,
                              // plane, expert), box b_box_rows x 2 x blocks per step x 1; F32: (row, plane, expert),
                              // box b_box_rows x blocks per step x 1
  CUtensorMap tmOut[2];       // F32 outputs with out_tma != 0: fp32 [rows][out_ld] map, box 32 x 32, 128B swizzle
  GemmClass cls[2];
  const int4* tiles;          // device tile list (nullptr: dense mode)
  const int32_t* num_tiles;   // device tile count (used when tiles != nullptr)
  const int32_t* range_lo;    // optional device bounds: only tiles [*range_lo, *range_hi) of the list run
  const int32_t* range_hi;
  int32_t dense_m;            // dense mode: M rows, tiles = ceil(M/128) x n_tiles, A rows start at dense_a_row0
  int32_t dense_n_tiles;
  int32_t dense_a_row0;
  int32_t pad_;
  int32_t* err;               // device error word
  const int32_t* stall_flag;  // test hook: producer waits for *stall_flag != 0 before any load (nullptr: none)
  uint64_t timeout_ns;        // bound on every mbarrier wait
};

// CTA-pair grouped GEMM (grouped_pair_kernel, gemm_pair.cu): a cluster of two CTAs computes one tile with
// tcgen05.mma.cta_group::2, M = 256 rows of weights (128 in each CTA's shared memory and TMEM lanes) times N tokens
// (N = the tile's token count rounded up to 32, at most 256; each CTA loads N/2 of the token rows). The output is
// the transpose of the single-CTA kernel's tile: TMEM lane = weight row (an output column), TMEM column = token.
constexpr int kPairKB = 2;                // 64-wide K blocks per stage: one box per operand carries both
constexpr int kPairStages = 3;
constexpr int kPairWBoxRows = 64;         // gate/up: 64 gate and 64 up rows per CTA in one 3-D box
constexpr int kPairDownBoxRows = 128;     // down: 128 weight rows per CTA in one box
constexpr int kPairTBoxRows = 128;        // token rows per box (one box: a CTA's N/2 <= 128 rows, and the rest unused)
constexpr int kPairTBoxRowsSmall = 32;    // token rows per box for tiles with N/2 <= 32
constexpr int kPairMaxTokens = 256;       // UMMA N limit
constexpr int kPairStageWBytes = kPairKB * 128 * kBlockK * 2;                  // 32 KB: 128 weight rows
constexpr int kPairStageTBytes = kPairKB * (kPairMaxTokens / 2) * kBlockK * 2; // 32 KB: up to 128 token rows
constexpr int kPairThreads = 320;          // warp 0 TMA, warp 1 MMA (+ TMEM alloc), warps 2..9 epilogue (two groups)
constexpr int kPairXchgBytes = 2 * 8192;   // per epilogue group: a 16-column slice staged in shared memory
constexpr int kPairSmemBytes = 1024 /*align slack*/ + kPairStages * (kPairStageWBytes + kPairStageTBytes) +
                               kBarRegionBytes + kPairXchgBytes;
static_assert(kPairSmemBytes <= 215040, "shared memory per CTA");

// Token tiles of an expert with `rows` member rows: ceil(rows / 256) tiles of equal width rounded up to 32.
__host__ __device__ inline int pair_tile_width(int rows) {
  if (rows <= 0) return 0;
  const int nt = (rows + kPairMaxTokens - 1) / kPairMaxTokens;
  return ((rows + nt - 1) / nt + 31) / 32 * 32;
}
__host__ __device__ inline int pair_tile_count(int rows) {
  const int w = pair_tile_width(rows);
  return w > 0 ? (rows + w - 1) / w : 0;
}

struct PairClass {
  int32_t kblocks;        // K / 64
  int32_t w_group_rows;   // weight rows per group (expert): 2I (gate/up) or H (down)
  int32_t w_up_offset;    // SwiGLU: row offset of the up rows inside a group (= I)
  int32_t w_stream;       // 1: honour the tile's stream bit (expert weights)
  int32_t w_group_mod;    // > 0: the weights are a ring of w_group_mod slots (offloaded experts)
  int32_t pad_;
  const int32_t* w_slot_map;  // ring with a hot set: slot of each group [G]; nullptr: slot e % w_group_mod
  void* out;              // SwiGLU: bf16 [rows][out_ld]; F32: float [rows][out_ld]
  int64_t out_ld;
};

// Pair tile record: x = group | (cls << 15) | (weight block << 16) | (stream << 31); y = first token row of the
// operand; z = tokens (1..256); w = first output row. A weight block is 128 values of j (gate/up: 64 gate and 64 up
// rows per CTA) or 256 output columns (down: 128 per CTA).
struct PairParams {
  // Every map has the 64-wide K block as its outermost dimension (stride 128 B), so that one box holds kPairKB
  // consecutive K blocks of its rows, one after the other.
  CUtensorMap tmW[2];         // weights, bf16: gate/up as (64, I, 2 x groups, K/64), box 64 x 64 x 2 x kPairKB;
                              // down as (64, rows, K/64), box 64 x 128 x kPairKB
  CUtensorMap tmT[2];         // token rows (gathered rows or X; h or shared h), (64, rows, K/64), box 64 x 128 x kPairKB
  CUtensorMap tmTs[2];        // the same, box 64 x 32 x kPairKB
  PairClass cls[2];
  const int4* tiles;
  const int32_t* num_tiles;
  const int32_t* range_lo;
  const int32_t* range_hi;
  int32_t* err;
  const int32_t* stall_flag;  // test hook, as GemmParams::stall_flag
  uint64_t timeout_ns;
};
cudaError_t launch_grouped_pair(const PairParams& p, int epilogue, int max_tiles, cudaStream_t stream);
cudaError_t prepare_pair_kernels();  // shared memory attribute and the co-resident clusters (once per device)
int pair_cluster_slots();     // co-resident clusters of two of grouped_pair_kernel (0 before prepare_pair_kernels)

// Routed expert weight formats. kFmtMxfp8: E4M3 codes, one E8M0 scale per 32 along K; kFmtNvfp4: E2M1 codes (two
// per byte), one E4M3 scale per 16 along K. A quantised launch runs grouped_gemm_q_kernel on the tiles of classes
// with b_scale (their tmB is a uint8 map of the codes).
enum WeightFormat : int { kFmtBf16 = 0, kFmtMxfp8 = 1, kFmtNvfp4 = 2 };
cudaError_t launch_grouped_gemm(const GemmParams& p, int epilogue, int grid, cudaStream_t stream,
                                int fmt = kFmtBf16);
cudaError_t prepare_gemm_kernels();   // sets the dynamic shared memory attribute (once per device)

// ------------------------------------------------------------------ routing
// Left for band_kernel by topk_kernel for a token it could not decide: the bound and the k-th / (k+1)-th logits.
struct BandInfo {
  double tau, vk, vk1, pad;
};

struct RouteParams {
  const float* logits;        // [n][E] fp32 (chunk-local)
  const uint16_t* x;          // chunk rows of X, bf16 [n][H]
  const uint16_t* w_router;   // bf16 [E][H]
  const float* wnorm;         // [E] ||w_e||_2
  WsHeader* hdr;
  int32_t n, E, H, k;
  float tau_coef;             // tau = tau_coef * ||x_t|| * max_e ||w_e||
  int32_t* topk_id;           // [n][k]
  float* topk_w;              // [n][k]
  uint8_t* band_flag;         // [n] 1 when the float64 recheck ran
  BandInfo* band_info;        // [n] of tokens left to band_kernel
  int32_t band_grid;          // CTAs of band_kernel (one per SM)
};
cudaError_t launch_router_norms(const uint16_t* w_router, int E, int H, float* wnorm, WsHeader* hdr,
                                cudaStream_t stream);
cudaError_t launch_topk(const RouteParams& p, cudaStream_t stream);  // top-k kernel + band kernel (2 launches)

struct PermuteParams {
  const int32_t* topk_id;     // [n][k]
  const uint8_t* band_flag;   // [n]
  const uint16_t* x;          // chunk rows of X [n][H]
  int32_t n, E, H, k, nblk;
  int64_t token0;             // global id of the chunk's first token
  uint32_t* masks;            // [nblk][E]
  int32_t* counts;            // [nblk][E]
  int32_t* block_band;        // [nblk]
  int32_t* base;              // [nblk][E]: rows of expert e in the blocks before block b (relative to the expert's
                              // first row, which is offsets[e])
  int32_t* totals;            // [E]: rows of expert e in the chunk
  int32_t* offsets;           // [E+1] (workspace)
  int32_t* offsets_out;       // user [E+1] for this chunk, or nullptr
  int32_t* token_row;         // [n][k]
  int32_t* row_token;         // [n*k] (global token ids)
  uint16_t* xp;               // gathered rows [n*k][H]
  WsHeader* hdr;
  // tile lists for the two grouped GEMMs
  int4* tiles_gu;             // capacity cap_gu
  int4* tiles_down;           // capacity cap_down
  int32_t* num_tiles;         // [2]: gu, down
  int32_t* tile_base;         // [2][E+1]: first gate/up and first down tile of each expert ([E] = routed total)
  int32_t cap_gu, cap_down;
  int32_t nt_gu, nt_down;     // N tiles per routed expert (GU: I / half, down: H / bn_down)
  int32_t nt_gu_shared, nt_down_shared;  // N tiles of the shared expert (0 = no shared expert)
  int32_t pair_gu, pair_dn;   // 1: that GEMM's tile list is for grouped_pair_kernel (its nt_* count weight blocks)
};
cudaError_t launch_count(const PermuteParams& p, cudaStream_t stream);
cudaError_t launch_block_bases(const PermuteParams& p, cudaStream_t stream);
cudaError_t launch_scan_tiles(const PermuteParams& p, cudaStream_t stream);
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ combine
cudaError_t launch_combine(const float* y, const float* w, const int32_t* token_row, const float* s, int64_t n,
                           int k, int H, uint16_t* out, cudaStream_t stream);

// ------------------------------------------------------------------ float64 tree combine (expert-parallel parts)
struct CombineTreeParams {
  const float* y;            // [R][H]
  const float* w;            // [n][k]
  const int32_t* token_row;  // [n][k]
  const int32_t* topk_id;    // [n][k]
  const float* s;            // [n][H] or null (finish only)
  double* partial;           // [n][H] (part only)
  uint16_t* out;             // bf16 [n][H] (finish only)
  float* out_f32;            // [n][H] or null (finish only)
  int64_t n;
  int32_t k, H;
  int32_t lo, block_log2;    // the part's experts: [lo, lo + 2^block_log2)
};
constexpr int kMaxFinishParts = 16;
struct CombineFinishParams {
  const double* part[kMaxFinishParts];  // n_parts arrays of count values
  const float* s;
  uint16_t* out;
  float* out_f32;
  int64_t count;  // n * H (even)
  int32_t n_parts;
};
size_t combine_tree_smem_bytes(int k);
// finish = false: write the part's float64 values to a.partial; true: the unsplit combine (one part covering all
// experts), + s, float32, bf16 in the same kernel.
cudaError_t launch_combine_tree(const CombineTreeParams& a, bool finish, cudaStream_t stream);
cudaError_t launch_combine_finish(const CombineFinishParams& a, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------------ ring of offloaded experts
struct RingCopyParams {
  const uint4* bank_gu;      // device-accessible address of the pinned host bank [E][2I][H] bf16
  const uint4* bank_down;    // [E][H][I]
  uint4* ring_gu;            // [S][2I][H]
  uint4* ring_down;          // [S][H][I]
  const int32_t* tile_base;  // the chunk's gate/up tile base per expert [E+1]: expert e is routed to iff it has tiles
  WsHeader* hdr;
  int64_t gu16, dn16;        // one expert's gate/up and down bytes / 16
  int32_t e0, count, slots;  // experts [e0, e0 + count) into slots e % slots
  const int32_t* slot_map;   // nullptr, or [E]: experts with slot_map[e] >= slots are resident (hot) and not staged
};
cudaError_t launch_ring_copy(const RingCopyParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ host helpers shared with noalloc.cu
void set_last_error(const char* msg);

}  // namespace moe
