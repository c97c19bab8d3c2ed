// Grouped GEMM on the 5th-generation tensor cores: TMA -> shared memory (128B swizzle) -> tcgen05.mma (TMEM
// accumulators) -> epilogue from TMEM. One persistent CTA per SM walks a tile list with a static stride.
//
// This is the expert-major projection step of the layer: "Flash Next EXL3: exact deep prefill" (introduction) runs
// each chunk expert by expert, and the maintainer review of the deep-prefill draft names the two expert kernels, a
// gate/up projection and a down projection, on tiles of expert members. Here a tile is 128 member rows of one expert
// (or of the shared expert) times up to 256 output columns; the K loop is fixed (64 per stage, 16 per instruction),
// so every output element is computed with the same accumulation order whatever the tile's row position or the
// number of members of its expert. That makes each row independent of the chunk size.
//
// bf16 weights, grouped_gemm_kernel (192 threads): warp 0 lane 0 issues TMA loads, two per stage (the tile's rows in
// one 128-row box, and its weight rows in one box: for gate/up a 3-D box of the tile's gate rows then its up rows);
// warp 1 owns the TMEM allocation and lane 0 issues the UMMAs; warps 2..5 read the accumulator back (warp w reads
// TMEM lanes 32*(w%4)..+31) and store the outputs. Two TMEM accumulators of 256 columns let the epilogue of one tile
// overlap the main loop of the next. The layer runs its gate/up projection on CTA pairs by default
// (grouped_pair_kernel, gemm_pair.cu), with the same bytes; this kernel serves the down projection, the router GEMM,
// the shared expert of block-scaled plans, and layers whose dimensions the pair kernel does not take.
//
// Block-scaled FP8 weights (MXFP8: E4M3 codes, one E8M0 power-of-two scale per 32 weights along K),
// grouped_gemm_q_kernel (480 threads): the weight codes stream through their own ring of 5 stages, which carries
// twice (four times for NVFP4: E2M1 codes, one E4M3 scale per 16) the weights per byte of shared memory that a
// bf16 stage does, and the activation rows through a ring of 3.
// Two groups of four warps take alternate steps: each decodes a stage's codes to bf16 into its own buffer, in the
// 128B-swizzled layout the UMMA descriptor reads (the layout TMA writes for bf16), and hands it to the UMMA issuer.
// A code times its scale is exactly a bf16 value, so the tensor core sees exactly the decoded weights and the
// accumulation order is that of the bf16 path. Warp 14 issues the activation loads.
#include "internal.h"
#include "ptx.cuh"
#include "swiglu.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace moe {
namespace {

struct TileInfo {
  int cls, group, n_idx, a_row0, rows, out_row0, stream;
};

// Tile t of a launch's walk over [lo, ntiles), its range of the list. The CTAs walk the range from its end: the
// shared expert's tiles (after the routed ones in the list, and the longest ones when I_s > I) start first and the
// last wave is made of the shortest tiles. Every tile is computed whole by one CTA, so the order changes no result.
// The tile read is ntiles - 1 - (t - lo), in the same range.
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t, int ntiles, int lo) {
  TileInfo ti;
  if (p.tiles != nullptr) {
    const int4 r = __ldg(p.tiles + (ntiles - 1 - (t - lo)));
    const uint32_t x = static_cast<uint32_t>(r.x);
    ti.group = static_cast<int>(x & 0x7FFFu);
    ti.cls = static_cast<int>((x >> 15) & 1u);
    ti.n_idx = static_cast<int>((x >> 16) & 0x7FFFu);
    ti.stream = static_cast<int>(x >> 31);
    ti.a_row0 = r.y;
    ti.rows = r.z;
    ti.out_row0 = r.w;
  } else {
    const int mt = (p.dense_m + kBlockM - 1) / kBlockM;
    const int m = t % mt;
    ti.cls = 0;
    ti.group = 0;
    ti.n_idx = t / mt;
    ti.stream = 0;
    ti.a_row0 = p.dense_a_row0 + m * kBlockM;
    ti.rows = min(kBlockM, p.dense_m - m * kBlockM);
    ti.out_row0 = m * kBlockM;
  }
  return ti;
}

__device__ __forceinline__ int total_tiles(const GemmParams& p) {
  if (p.tiles != nullptr) return *reinterpret_cast<const volatile int32_t*>(p.num_tiles);
  return ((p.dense_m + kBlockM - 1) / kBlockM) * p.dense_n_tiles;
}

// First tile of this launch and the end of its range: the whole list, or the part [*range_lo, *range_hi) of it
// (either bound may be absent).
__device__ __forceinline__ int2 tile_range(const GemmParams& p) {
  int lo = 0, hi = total_tiles(p);
  if (p.range_lo != nullptr) lo = max(0, *reinterpret_cast<const volatile int32_t*>(p.range_lo));
  if (p.range_hi != nullptr) hi = min(hi, *reinterpret_cast<const volatile int32_t*>(p.range_hi));
  return make_int2(lo, hi);
}

__device__ __forceinline__ void raise_error(const GemmParams& p, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, site, static_cast<int>(blockIdx.x)));
}

// Where a group's B rows live: the group itself (resident weights), its ring slot e % b_group_mod (offloaded
// experts), or the slot the map gives (offloaded experts with a resident hot set).
__device__ __forceinline__ int b_slot(const GemmClass& C, int group) {
  if (C.b_group_mod <= 0) return group;
  return C.b_slot_map != nullptr ? __ldg(C.b_slot_map + group) : group % C.b_group_mod;
}

// First B row of a tile's (first) box: the group's (or ring slot's) row base plus the N tile's offset.
template <int EPI>
__device__ __forceinline__ int tile_b_row(const GemmClass& C, int slot, int n_idx) {
  return slot * C.b_group_rows + n_idx * (EPI == kEpiSwiGLU ? C.b_box_rows : C.n_tile);
}

// Reads one tile's accumulator (columns [0, n_tile) at tbase) back from TMEM and stores the tile's outputs. Each of
// the four epilogue warps owns a 32-row slab; a 32-column block of the accumulator arrives one row per lane.
// SwiGLU: the bf16 results are staged in shared memory (odd row stride: no bank conflicts) and written back
// row-contiguously, so every store instruction covers whole 128-byte lines.
// F32: a block whose 32 rows all belong to the tile (or whose map clips the rest) is written into one of the warp's
// NBUF staging buffers in the 128B-swizzled layout (16-byte chunk j of row r at chunk j ^ (r % 8): conflict-free)
// and stored by a single TMA tensor store; the buffer is reused once that store has read it. Rows of a partial slab
// are stored directly, one row per lane, since the rows after them belong to other tiles.
template <int EPI, int NBUF>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const GemmClass& C, const TileInfo& ti,
                                              uint32_t tbase, uint8_t* bufs, int lane, int q, uint32_t& blk) {
  const int slab_rows = ti.rows - q * 32;
  const int64_t slab_row0 = static_cast<int64_t>(ti.out_row0) + q * 32;
  if (EPI == kEpiSwiGLU) {
    uint32_t* stage = reinterpret_cast<uint32_t*>(bufs);
    const int half = C.b_box_rows;
    const int64_t ldw = C.out_ld / 2;  // row stride in 32-bit words (two bf16 each)
    uint32_t* outw = reinterpret_cast<uint32_t*>(C.out) + (static_cast<int64_t>(ti.n_idx) * half) / 2;
    for (int c = 0; c < half; c += 32) {
      uint32_t g[32], u[32];
      ptx::tmem_ld32(tbase + c, g);
      ptx::tmem_ld32(tbase + half + c, u);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        stage[lane * 17 + i] = pack_bf16(swiglu(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                         swiglu(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
      __syncwarp();
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = m * 8 + (lane >> 2), w0 = (lane & 3) * 4;
        if (r < slab_rows) {
          const uint32_t* sr = stage + r * 17 + w0;
          *reinterpret_cast<uint4*>(outw + (slab_row0 + r) * ldw + c / 2 + w0) = make_uint4(sr[0], sr[1], sr[2], sr[3]);
        }
      }
      __syncwarp();
    }
  } else {
    if (slab_rows <= 0) return;
    const int col0 = ti.n_idx * C.n_tile;
    const bool tma = C.out_tma == 2 || (C.out_tma == 1 && slab_rows >= 32);
    float* outb = static_cast<float*>(C.out) + col0;
    const bool vec = (C.out_ld % 4) == 0;
    for (int c = 0; c < C.n_tile; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c, v);
      ptx::tmem_ld_wait();
      if (tma) {
        uint8_t* buf = bufs + (blk % NBUF) * kEpiBufBytes;
        if (lane == 0) ptx::bulk_wait_group_read<NBUF - 1>();  // the store that last read this buffer is done
        __syncwarp();
        uint8_t* rowp = buf + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
              make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&p.tmOut[ti.cls], ptx::smem_u32(buf), col0 + c, static_cast<int32_t>(slab_row0));
          ptx::bulk_commit_group();
        }
        ++blk;
      } else if (lane < slab_rows) {
        float* dst = outb + (slab_row0 + lane) * C.out_ld + c;
        const int gc0 = col0 + c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gc = gc0 + 4 * j;
          if (vec && gc + 4 <= C.out_cols) {
            *reinterpret_cast<float4*>(dst + 4 * j) =
                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                            __uint_as_float(v[4 * j + 3]));
          } else {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              if (gc + jj < C.out_cols) dst[4 * j + jj] = __uint_as_float(v[4 * j + jj]);
          }
        }
      }
    }
  }
}

// The epilogue role (warps 2..5) of both kernels: waits for each tile's accumulator, stores it, frees it. Before
// the role ends, lane 0 waits for its TMA stores to complete (their shared-memory sources stay live until then).
template <int EPI, int NBUF>
__device__ __forceinline__ void epilogue_role(const GemmParams& p, int tfirst, int ntiles, uint32_t tmem_base,
                                              uint32_t tfull0, uint32_t tempty0, uint8_t* bufs, int warp, int lane,
                                              volatile int* abort_flag) {
  const int q = warp & 3;
  int local = 0;
  uint32_t blk = 0;
  const int lo = tfirst - static_cast<int>(blockIdx.x);
  for (int t = tfirst; t < ntiles; t += gridDim.x, ++local) {
    const TileInfo ti = decode_tile(p, t, ntiles, lo);
    const int acc = local & 1;
    const uint32_t use = static_cast<uint32_t>(local >> 1);
    bool ok = ptx::wait_bounded(tfull0 + 8u * acc, use & 1u, p.timeout_ns, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) raise_error(p, abort_flag, kSiteEpilogueFull);
      break;
    }
    ptx::tc_fence_after();
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kMaxN);
    epilogue_tile<EPI, NBUF>(p, p.cls[ti.cls], ti, tbase, bufs, lane, q, blk);
    ptx::tc_fence_before();
    ptx::mbar_arrive(tempty0 + 8u * acc);
  }
  if (lane == 0) ptx::bulk_wait_group_all();
  __syncwarp();
}

// An exact f16x2 value whose significands need at most 7 fraction bits, as the bf16x2 bits of the same values times
// 2^-112: f16 and bf16 share the sign bit and the leading fraction bits, and the 5-bit f16 exponent (bias 15) read
// as a bf16 exponent (bias 127) scales by 2^-112. Zeros stay (signed) zeros; no f16 subnormal reaches here (E4M3
// and E2M1 values are f16 normals).
__device__ __forceinline__ uint32_t f16x2_as_bf16x2_m112(uint32_t h2) {
  return ((h2 & 0x7FFF7FFFu) >> 3) | (h2 & 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16x2 with both halves 2^e (e + 127 in 1..254).
__device__ __forceinline__ uint32_t bf16x2_pow2(int e) {
  return static_cast<uint32_t>(e + 127) * 0x00800080u;
}

// Two E4M3 codes times 2^(s - 127) as two bf16 values: E4M3 -> f16 (one conversion, exact), the bits read as bf16
// times 2^-112, then two exact multiplies by 2^ea and 2^eb (ea + eb = s - 15; each factor and every intermediate
// stays a bf16 normal for s in [10, 246], where the products are bf16 values).
__device__ __forceinline__ uint32_t decode_pair(uint32_t codes16, uint32_t fa, uint32_t fb) {
  const uint32_t h2 = ptx::e4m3x2_to_f16x2(static_cast<uint16_t>(codes16));
  return bf16x2_mul(bf16x2_mul(f16x2_as_bf16x2_m112(h2), fa), fb);
}

// Decodes one stage of MXFP8 weights: `rows` rows of 64 E4M3 codes (row-major, as TMA landed them) with scales
// sc[2][rows] (K blocks 0..31 and 32..63 of the stage), by the 128 threads of a decoder group (ct = 0..127), into
// bf16 rows of 128 B in the 128B-swizzled K-major layout (8-row atoms of 1024 B, 16-byte chunk c of row r at chunk
// c ^ (r % 8)).
__device__ __forceinline__ void decode_stage(const uint8_t* codes, const uint8_t* sc, uint8_t* dst, int rows,
                                             int ct) {
  const int items = rows * 4;  // 16-code chunks, chunk i = row i / 4, K elements 16 * (i % 4) ..
  uint4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = ct + 128 * j;
    if (i < items) v[j] = *reinterpret_cast<const uint4*>(codes + i * 16);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = ct + 128 * j;
    if (i < items) {
      const int r = i >> 2, c = i & 3;
      const int e = static_cast<int>(sc[(c >> 1) * rows + r]) - 15;  // 2^(s - 127) = 2^-112 * 2^e
      const int ea = e >> 1;
      const uint32_t fa = bf16x2_pow2(ea), fb = bf16x2_pow2(e - ea);
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t o[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        o[2 * q] = decode_pair(w[q], fa, fb);
        o[2 * q + 1] = decode_pair(w[q] >> 16, fa, fb);
      }
      uint8_t* rowp = dst + (r >> 3) * 1024 + (r & 7) * 128;
      *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// Two E2M1 codes (one byte) times the block scale as two bf16 values: E2M1 -> f16 (one conversion, exact), read as
// bf16 times 2^-112, times f2 = the scale times 2^112 (a bf16 normal for every E4M3 scale but zero). Exact: a code
// times an E4M3 value has at most 2 x 4 significant bits and magnitude 2^-10 .. 2688.
__device__ __forceinline__ uint32_t decode_pair_fp4(uint32_t byte, uint32_t f2) {
  return bf16x2_mul(f16x2_as_bf16x2_m112(ptx::e2m1x2_to_f16x2(byte & 0xFFu)), f2);
}

// Decodes one stage of NVFP4 weights: `rows` rows of 32 bytes (64 E2M1 codes, element 2j in the low nibble of byte
// j) with E4M3 scales sc[4][rows] (16-wide K blocks of the stage), into the same bf16 layout as decode_stage.
__device__ __forceinline__ void decode_stage_fp4(const uint8_t* codes, const uint8_t* sc, uint8_t* dst, int rows,
                                                 int ct) {
  const int items = rows * 4;  // 16-code (8-byte) chunks, chunk i = row i / 4, K block i % 4
  uint2 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = ct + 128 * j;
    if (i < items) v[j] = *reinterpret_cast<const uint2*>(codes + i * 8);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = ct + 128 * j;
    if (i < items) {
      const int r = i >> 2, c = i & 3;
      const uint32_t sh = ptx::e4m3x2_to_f16x2(static_cast<uint16_t>(sc[c * rows + r]));
      const float f = __half2float(*reinterpret_cast<const __half*>(&sh)) * 0x1p112f;  // the E4M3 scale x 2^112
      const uint32_t f2 = pack_bf16(f, f);
      const uint32_t w[2] = {v[j].x, v[j].y};
      uint32_t o[8];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int b = 0; b < 4; ++b) o[4 * q + b] = decode_pair_fp4(w[q] >> (8 * b), f2);
      uint8_t* rowp = dst + (r >> 3) * 1024 + (r & 7) * 128;
      *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// ============================================================================================ bf16 weights
template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + kStages * kStageABytes;
  const uint32_t bars = sB + kStages * kStageBBytes;
  uint8_t* bars_ptr = base_ptr + kStages * (kStageABytes + kStageBBytes);
  // barrier slots: full[kStages], empty[kStages], tmem_full[2], tmem_empty[2], drain
  const uint32_t full0 = bars, empty0 = bars + 8u * kStages, tfull0 = bars + 16u * kStages;
  const uint32_t tempty0 = tfull0 + 16u, drain_bar = tempty0 + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 16 * kStages + 40);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 16 * kStages + 44);

  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull0 + 8u * a, 1);
      ptx::mbar_init(tempty0 + 8u * a, 4 * 32);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&p.tmA[0]);
    ptx::tma_prefetch_desc(&p.tmA[1]);
    ptx::tma_prefetch_desc(EPI == kEpiSwiGLU ? &p.tmBg[0] : &p.tmB[0]);
    ptx::tma_prefetch_desc(EPI == kEpiSwiGLU ? &p.tmBg[1] : &p.tmB[1]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 2 * kMaxN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int2 trange = tile_range(p);
  const int tfirst = trange.x + static_cast<int>(blockIdx.x);
  const int ntiles = trange.y;
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool failed = false;
      const uint64_t pol_stream = ptx::make_policy_evict_first();
      if (p.stall_flag != nullptr) {
        // Test hook: wait (bounded) for a flag in global memory before loading anything.
        const uint64_t t0 = ptx::globaltimer();
        while (*reinterpret_cast<const volatile int32_t*>(p.stall_flag) == 0) {
          if (ptx::globaltimer() - t0 > tmo || *abort_flag) {
            raise_error(p, abort_flag, kSiteStallFlag);
            failed = true;
            break;
          }
        }
      }
      for (int t = tfirst; !failed && t < ntiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
        const GemmClass& C = p.cls[ti.cls];
        const void* tA = &p.tmA[ti.cls];
        const void* tB = &p.tmB[ti.cls];
        const int nA = (ti.rows + kABoxRows - 1) / kABoxRows;
        const uint32_t b_loads = (EPI == kEpiSwiGLU) ? 2u : 1u;
        const uint32_t bytes = static_cast<uint32_t>(nA * kABoxRows * 128) + b_loads * C.b_box_rows * 128u;
        const int slot = b_slot(C, ti.group);
        const int b_row0 = tile_b_row<EPI>(C, slot, ti.n_idx);
        for (int kb = 0; kb < C.kblocks; ++kb) {
          if (!ptx::wait_bounded(empty0 + 8u * stage, phase ^ 1u, tmo, abort_flag)) {
            raise_error(p, abort_flag, kSiteProducerEmpty);
            failed = true;
            break;
          }
          const uint32_t fb = full0 + 8u * stage;
          ptx::mbar_arrive_expect_tx(fb, bytes);
          const uint32_t a_dst = sA + stage * kStageABytes;
          const uint32_t b_dst = sB + stage * kStageBBytes;
          const int kc = kb * kBlockK;
          for (int j = 0; j < nA; ++j)
            ptx::tma_load_2d(a_dst + j * (kABoxRows * 128), tA, kc, ti.a_row0 + j * kABoxRows, fb);
          const bool stream = C.b_stream && ti.stream;
          if (EPI == kEpiSwiGLU) {
            // the tile's gate rows and up rows in one box of the (K, j, 2 x slot + half) view, gate rows first
            const void* tBg = &p.tmBg[ti.cls];
            const int j0 = ti.n_idx * C.b_box_rows;
            if (stream)
              ptx::tma_load_3d_hint(b_dst, tBg, kc, j0, 2 * slot, fb, pol_stream);
            else
              ptx::tma_load_3d(b_dst, tBg, kc, j0, 2 * slot, fb);
          } else if (stream) {
            ptx::tma_load_2d_hint(b_dst, tB, kc, b_row0, fb, pol_stream);
          } else {
            ptx::tma_load_2d(b_dst, tB, kc, b_row0, fb);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        // Wait (bounded) until every load already issued has landed, so no copy targets a CTA that has exited.
        int no_abort = 0;
        for (int s = 0; s < kStages; ++s) {
          const uint32_t cnt = issued / kStages + (static_cast<uint32_t>(s) < issued % kStages ? 1u : 0u);
          if (cnt == 0) continue;
          if (!ptx::wait_bounded(full0 + 8u * s, (cnt - 1u) & 1u, tmo, &no_abort))
            atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      int stage = 0, local = 0;
      uint32_t phase = 0;
      bool failed = false, issued_any = false;
      for (int t = tfirst; t < ntiles; t += gridDim.x, ++local) {
        const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
        const GemmClass& C = p.cls[ti.cls];
        const int acc = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!ptx::wait_bounded(tempty0 + 8u * acc, (use & 1u) ^ 1u, tmo, abort_flag)) {
          raise_error(p, abort_flag, kSiteMmaTmemEmpty);
          failed = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kMaxN);
        const uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, static_cast<uint32_t>(C.n_tile));
        for (int kb = 0; kb < C.kblocks; ++kb) {
          if (!ptx::wait_bounded(full0 + 8u * stage, phase, tmo, abort_flag)) {
            raise_error(p, abort_flag, kSiteMmaFull);
            failed = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t a_desc = ptx::sw128_kmajor_desc(sA + stage * kStageABytes);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sB + stage * kStageBBytes);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk) {
            // advancing K by 16 bf16 = 32 bytes = 2 units of the descriptor's start address
            ptx::umma_bf16(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit(empty0 + 8u * stage);  // frees the smem stage once these UMMAs have read it
          issued_any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (failed) break;
        ptx::umma_commit(tfull0 + 8u * acc);  // accumulator ready for the epilogue
      }
      if (failed && issued_any) {
        int no_abort = 0;
        ptx::umma_commit(drain_bar);
        if (!ptx::wait_bounded(drain_bar, 0u, tmo, &no_abort))
          atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    uint8_t* bufs = bars_ptr + kBarRegionBytes + (warp - 2) * kEpiBufs * kEpiBufBytes;
    epilogue_role<EPI, kEpiBufs>(p, tfirst, ntiles, tmem_base, tfull0, tempty0, bufs, warp, lane, abort_flag);
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 2 * kMaxN);
  }
}

// ============================================================================================ MXFP8 weights
// Rings: A (activation rows, kQStagesA x 16 KB), C (E4M3 codes, kQStagesC x 16 KB, with 2 x rows scale bytes
// each), D (decoded bf16 B tiles, one 32 KB buffer per decoder group). Step i of the CTA's (tile, K block) sequence
// uses A slot i % kQStagesA, C slot i % kQStagesC and D buffer i % 2, decoded by group i % 2. Only tiles whose
// class has scales run here (the routed experts); the bf16 shared expert takes grouped_gemm_kernel.
template <int EPI, int FMT>
__global__ void __launch_bounds__(kGemmThreadsQ, 1) grouped_gemm_q_kernel(const __grid_constant__ GemmParams p) {
  // per row and 64-wide K step: code bytes and scale blocks (MXFP8: 64 codes, 2 blocks of 32; NVFP4: 32 bytes of
  // two codes each, 4 blocks of 16)
  constexpr uint32_t kCodeBytes = FMT == kFmtNvfp4 ? 32u : 64u;
  constexpr int kScaleBlocks = FMT == kFmtNvfp4 ? 4 : 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sD = sA + kQStagesA * kStageABytes;
  const uint32_t sC = sD + kQStagesD * kStageBBytes;
  const uint32_t sS = sC + kQStagesC * kQStageCodeBytes;
  const uint32_t bars = sS + kQStagesC * kQStageScaleBytes;
  uint8_t* sD_ptr = base_ptr + (sD - base);
  const uint8_t* sC_ptr = base_ptr + (sC - base);
  const uint8_t* sS_ptr = base_ptr + (sS - base);
  uint8_t* bars_ptr = base_ptr + (bars - base);
  const uint32_t a_full0 = bars, a_empty0 = a_full0 + 8u * kQStagesA;
  const uint32_t c_full0 = a_empty0 + 8u * kQStagesA, c_empty0 = c_full0 + 8u * kQStagesC;
  const uint32_t d_full0 = c_empty0 + 8u * kQStagesC, d_empty0 = d_full0 + 8u * kQStagesD;
  const uint32_t tfull0 = d_empty0 + 8u * kQStagesD, tempty0 = tfull0 + 16u, drain_bar = tempty0 + 16u;
  static_assert(8 * (2 * kQStagesA + 2 * kQStagesC + 2 * kQStagesD + 5) + 8 <= 256, "barrier region");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + (drain_bar + 8u - bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + (drain_bar + 12u - bars));

  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStagesA; ++s) {
      ptx::mbar_init(a_full0 + 8u * s, 1);
      ptx::mbar_init(a_empty0 + 8u * s, 1);
    }
    for (int s = 0; s < kQStagesC; ++s) {
      ptx::mbar_init(c_full0 + 8u * s, 1);
      ptx::mbar_init(c_empty0 + 8u * s, 4);  // one arrival per warp of the decoder group
    }
    for (int s = 0; s < kQStagesD; ++s) {
      ptx::mbar_init(d_full0 + 8u * s, 4);
      ptx::mbar_init(d_empty0 + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull0 + 8u * a, 1);
      ptx::mbar_init(tempty0 + 8u * a, 4 * 32);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&p.tmA[0]);
    ptx::tma_prefetch_desc(EPI == kEpiSwiGLU ? &p.tmBg[0] : &p.tmB[0]);
    ptx::tma_prefetch_desc(&p.tmS[0]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 2 * kMaxN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int2 trange = tile_range(p);
  const int tfirst = trange.x + static_cast<int>(blockIdx.x);
  const int ntiles = trange.y;
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA: E4M3 codes and their scales
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0, issued = 0;
      bool failed = false;
      const uint64_t pol_stream = ptx::make_policy_evict_first();
      for (int t = tfirst; !failed && t < ntiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
        const GemmClass& C = p.cls[ti.cls];
        const void* tB = &p.tmB[ti.cls];
        const uint32_t b_loads = (EPI == kEpiSwiGLU) ? 2u : 1u;
        const uint32_t bytes = b_loads * C.b_box_rows * (kCodeBytes + kScaleBlocks);
        const int gslot = b_slot(C, ti.group);
        const int b_row0 = tile_b_row<EPI>(C, gslot, ti.n_idx);
        const int r0 = b_row0 - gslot * C.b_group_rows;  // first row inside the group
        const bool hint = C.b_stream && ti.stream;
        for (int kb = 0; kb < C.kblocks; ++kb) {
          if (!ptx::wait_bounded(c_empty0 + 8u * slot, phase ^ 1u, tmo, abort_flag)) {
            raise_error(p, abort_flag, kSiteProducerEmpty);
            failed = true;
            break;
          }
          const uint32_t fb = c_full0 + 8u * slot;
          ptx::mbar_arrive_expect_tx(fb, bytes);
          const uint32_t c_dst = sC + slot * kQStageCodeBytes;
          const uint32_t s_dst = sS + slot * kQStageScaleBytes;
          const int kx = kb * static_cast<int>(kCodeBytes);  // inner coordinate of the code map, in bytes
          if (EPI == kEpiSwiGLU) {
            // the tile's gate and up code rows in one box of the (bytes, j, 2 x slot + half) view
            const void* tBg = &p.tmBg[ti.cls];
            if (hint)
              ptx::tma_load_3d_hint(c_dst, tBg, kx, r0, 2 * gslot, fb, pol_stream);
            else
              ptx::tma_load_3d(c_dst, tBg, kx, r0, 2 * gslot, fb);
            // the step's scale blocks of those rows in one box of the (row in half, half, plane, expert) view:
            // block h of the gate rows, then of the up rows, for each h in turn
            ptx::tma_load_4d(s_dst, &p.tmS[ti.cls], r0, 0, kScaleBlocks * kb, ti.group, fb);
          } else {
            if (hint)
              ptx::tma_load_2d_hint(c_dst, tB, kx, b_row0, fb, pol_stream);
            else
              ptx::tma_load_2d(c_dst, tB, kx, b_row0, fb);
            // the step's scale blocks of the tile's rows in one box of the (row, plane, expert) view
            ptx::tma_load_3d(s_dst, &p.tmS[ti.cls], r0, kScaleBlocks * kb, ti.group, fb);
          }
          ++issued;
          if (++slot == kQStagesC) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        int no_abort = 0;
        for (int s = 0; s < kQStagesC; ++s) {
          const uint32_t cnt = issued / kQStagesC + (static_cast<uint32_t>(s) < issued % kQStagesC ? 1u : 0u);
          if (cnt == 0) continue;
          if (!ptx::wait_bounded(c_full0 + 8u * s, (cnt - 1u) & 1u, tmo, &no_abort))
            atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
        }
      }
    }
    __syncwarp();
  } else if (warp == kGemmThreadsQ / 32 - 1) {
    // ------------------------------------------------------------ TMA: activation rows
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0, issued = 0;
      bool failed = false;
      for (int t = tfirst; !failed && t < ntiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
        const GemmClass& C = p.cls[ti.cls];
        const void* tA = &p.tmA[ti.cls];
        const int nA = (ti.rows + kABoxRows - 1) / kABoxRows;
        const uint32_t bytes = static_cast<uint32_t>(nA * kABoxRows * 128);
        for (int kb = 0; kb < C.kblocks; ++kb) {
          if (!ptx::wait_bounded(a_empty0 + 8u * slot, phase ^ 1u, tmo, abort_flag)) {
            raise_error(p, abort_flag, kSiteProducerEmpty);
            failed = true;
            break;
          }
          const uint32_t fb = a_full0 + 8u * slot;
          ptx::mbar_arrive_expect_tx(fb, bytes);
          const uint32_t a_dst = sA + slot * kStageABytes;
          for (int j = 0; j < nA; ++j)
            ptx::tma_load_2d(a_dst + j * (kABoxRows * 128), tA, kb * kBlockK, ti.a_row0 + j * kABoxRows, fb);
          ++issued;
          if (++slot == kQStagesA) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        int no_abort = 0;
        for (int s = 0; s < kQStagesA; ++s) {
          const uint32_t cnt = issued / kQStagesA + (static_cast<uint32_t>(s) < issued % kQStagesA ? 1u : 0u);
          if (cnt == 0) continue;
          if (!ptx::wait_bounded(a_full0 + 8u * s, (cnt - 1u) & 1u, tmo, &no_abort))
            atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      int local = 0;
      uint32_t i = 0;
      bool failed = false, issued_any = false;
      for (int t = tfirst; t < ntiles; t += gridDim.x, ++local) {
        const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
        const GemmClass& C = p.cls[ti.cls];
        const int acc = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!ptx::wait_bounded(tempty0 + 8u * acc, (use & 1u) ^ 1u, tmo, abort_flag)) {
          raise_error(p, abort_flag, kSiteMmaTmemEmpty);
          failed = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kMaxN);
        const uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, static_cast<uint32_t>(C.n_tile));
        for (int kb = 0; kb < C.kblocks; ++kb, ++i) {
          const uint32_t as = i % kQStagesA, aph = (i / kQStagesA) & 1u;
          const uint32_t ds = i % kQStagesD, dph = (i / kQStagesD) & 1u;
          if (!ptx::wait_bounded(a_full0 + 8u * as, aph, tmo, abort_flag) ||
              !ptx::wait_bounded(d_full0 + 8u * ds, dph, tmo, abort_flag)) {
            raise_error(p, abort_flag, kSiteMmaFull);
            failed = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t a_desc = ptx::sw128_kmajor_desc(sA + as * kStageABytes);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(sD + ds * kStageBBytes);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)
            ptx::umma_bf16(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          ptx::umma_commit(a_empty0 + 8u * as);  // both buffers are free once these UMMAs have read them
          ptx::umma_commit(d_empty0 + 8u * ds);
          issued_any = true;
        }
        if (failed) break;
        ptx::umma_commit(tfull0 + 8u * acc);
      }
      if (failed && issued_any) {
        int no_abort = 0;
        ptx::umma_commit(drain_bar);
        if (!ptx::wait_bounded(drain_bar, 0u, tmo, &no_abort))
          atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    uint8_t* bufs = bars_ptr + kBarRegionBytes + (warp - 2) * kEpiBufs * kEpiBufBytes;
    epilogue_role<EPI, kEpiBufs>(p, tfirst, ntiles, tmem_base, tfull0, tempty0, bufs, warp, lane, abort_flag);
  } else {
    // ------------------------------------------------------------ decoders (warps 6..13: groups 0 and 1)
    const int dt = static_cast<int>(threadIdx.x) - 6 * 32;
    const int group = dt / 128, ct = dt % 128;
    uint32_t i = 0;
    bool failed = false;
    for (int t = tfirst; t < ntiles; t += gridDim.x) {
      const TileInfo ti = decode_tile(p, t, ntiles, trange.x);
      const GemmClass& C = p.cls[ti.cls];
      for (int kb = 0; kb < C.kblocks; ++kb, ++i) {
        if (static_cast<int>(i % kQStagesD) != group) continue;
        const uint32_t cs = i % kQStagesC, cph = (i / kQStagesC) & 1u;
        const uint32_t dph = (i / kQStagesD) & 1u;
        // one lane per warp waits for the codes and for the group's buffer; the warp shares the outcome
        int ok = 1;
        if (lane == 0 && !failed)
          ok = (ptx::wait_bounded(c_full0 + 8u * cs, cph, tmo, abort_flag) &&
                ptx::wait_bounded(d_empty0 + 8u * group, dph ^ 1u, tmo, abort_flag)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok && !failed) {
          if (lane == 0) raise_error(p, abort_flag, kSiteDecodeFull);
          failed = true;
        }
        if (failed) break;
        if (FMT == kFmtNvfp4)
          decode_stage_fp4(sC_ptr + cs * kQStageCodeBytes, sS_ptr + cs * kQStageScaleBytes,
                           sD_ptr + group * kStageBBytes, C.n_tile, ct);
        else
          decode_stage(sC_ptr + cs * kQStageCodeBytes, sS_ptr + cs * kQStageScaleBytes,
                       sD_ptr + group * kStageBBytes, C.n_tile, ct);
        // the decoded tile to the async proxy; the codes have been consumed
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(c_empty0 + 8u * cs);
          ptx::mbar_arrive(d_full0 + 8u * group);
        }
      }
      if (failed) break;
    }
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 2 * kMaxN);
  }
}

}  // namespace

cudaError_t prepare_gemm_kernels() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kEpiF32>, attr, kGemmSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_kernel<kEpiSwiGLU>, attr, kGemmSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_q_kernel<kEpiF32, kFmtMxfp8>, attr, kGemmSmemBytesQ);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_q_kernel<kEpiSwiGLU, kFmtMxfp8>, attr, kGemmSmemBytesQ);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_q_kernel<kEpiF32, kFmtNvfp4>, attr, kGemmSmemBytesQ);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_q_kernel<kEpiSwiGLU, kFmtNvfp4>, attr, kGemmSmemBytesQ);
  return e;
}

cudaError_t launch_grouped_gemm(const GemmParams& p, int epilogue, int grid, cudaStream_t stream, int fmt) {
  if (grid <= 0) return cudaSuccess;
  const bool glu = epilogue == kEpiSwiGLU;
  if (fmt == kFmtMxfp8) {
    if (glu)
      grouped_gemm_q_kernel<kEpiSwiGLU, kFmtMxfp8><<<grid, kGemmThreadsQ, kGemmSmemBytesQ, stream>>>(p);
    else
      grouped_gemm_q_kernel<kEpiF32, kFmtMxfp8><<<grid, kGemmThreadsQ, kGemmSmemBytesQ, stream>>>(p);
  } else if (fmt == kFmtNvfp4) {
    if (glu)
      grouped_gemm_q_kernel<kEpiSwiGLU, kFmtNvfp4><<<grid, kGemmThreadsQ, kGemmSmemBytesQ, stream>>>(p);
    else
      grouped_gemm_q_kernel<kEpiF32, kFmtNvfp4><<<grid, kGemmThreadsQ, kGemmSmemBytesQ, stream>>>(p);
  } else if (glu) {
    grouped_gemm_kernel<kEpiSwiGLU><<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(p);
  } else {
    grouped_gemm_kernel<kEpiF32><<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace moe
