// Grouped GEMM on CTA pairs: a cluster of two CTAs computes each tile with tcgen05.mma.cta_group::2.
//
// Same step of the layer as grouped_gemm_kernel (the expert-major gate/up and down projections, "Flash Next EXL3:
// exact deep prefill", introduction) on the same tile lists' experts and rows, with the operands the other way
// round: M = 256 rows of an expert's weights (each CTA holds 128 of them in shared memory, and their accumulators
// in its 128 TMEM lanes), N = the tile's tokens rounded up to 32 (at most 256; each CTA loads half of the token
// rows, and the tensor cores of the pair read both halves). Per SM and 64-wide K block that is 16 KB of weights and
// N/2 x 128 B of tokens for 128 x N x 64 multiply-adds, against 48 KB for 128 x 256 x 64 in the single-CTA kernel;
// and an expert's rows are covered in steps of 32 tokens instead of 128 rows. The K order is the same (64-wide K
// blocks, 16 per instruction, in order), so each output element is accumulated in the same order as there.
//
// A stage is two K blocks. A stage costs about the same per TMA operation whatever the box size, so each CTA loads a
// stage with two: its weight rows of both K blocks in one box, its token rows of both K blocks in another (the maps
// have the K block as their outermost dimension).
//
// Roles (320 threads per CTA, both CTAs): warp 0 lane 0 loads the CTA's weight and token boxes; their completion is
// counted on the even CTA's full barrier. Warp 1 of the even CTA issues the UMMAs and commits each stage to the
// empty barriers of both CTAs, and each accumulator to both CTAs' TMEM-full barriers. Warps 2..9 of each CTA, two
// groups of four, read that CTA's accumulator lanes (an output column each) in alternate 16-token slices, stage
// each slice as token rows in shared memory and store whole rows with 16-byte stores; they release the accumulator
// on the even CTA's TMEM-empty barrier. Gate/up: lanes 0..63 hold gate rows j and lanes 64..127 the up rows of the
// same j; gate and up threads exchange half of their values through shared memory and each forms half of h.
#include "internal.h"
#include "ptx.cuh"
#include "swiglu.cuh"

#include <cuda_bf16.h>
#include <algorithm>

namespace moe {
namespace {

struct PairTile {
  int cls, group, wb, stream, t_row0, n, out_row0;
};

// Tile t of the walk over [lo, hi), read from the end of the range (as grouped_gemm_kernel's walk).
__device__ __forceinline__ PairTile decode_pair_tile(const PairParams& p, int t, int hi, int lo) {
  const int4 r = __ldg(p.tiles + (hi - 1 - (t - lo)));
  const uint32_t x = static_cast<uint32_t>(r.x);
  PairTile ti;
  ti.group = static_cast<int>(x & 0x7FFFu);
  ti.cls = static_cast<int>((x >> 15) & 1u);
  ti.wb = static_cast<int>((x >> 16) & 0x7FFFu);
  ti.stream = static_cast<int>(x >> 31);
  ti.t_row0 = r.y;
  ti.n = r.z;
  ti.out_row0 = r.w;
  return ti;
}

__device__ __forceinline__ void pair_raise(const PairParams& p, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, site, static_cast<int>(blockIdx.x)));
}

__device__ __forceinline__ int pair_width(int n) { return (n + 31) & ~31; }

// One tile's accumulator (this CTA's 128 lanes, columns [0, N)) to the outputs, by one group of four epilogue
// warps (warp q = warp % 4 reads TMEM lanes 32q..32q+31; gt = the thread's index in the group, 0..127). The group
// takes the 16-column slices s = group, group + 2, ... of the tile's token columns; a slice arrives one lane (an
// output column) per thread and 16 tokens per thread, is staged in shared memory (8 KB per group) as 16 token rows,
// and leaves as 16-byte vector stores of whole rows. Slices past the tile's tokens are skipped.
// SwiGLU: lanes 0..63 hold gate rows j and lanes 64..127 up rows of the same j. Gate threads stage their g of
// tokens 8..15, up threads their u of tokens 0..7; then gate threads form h for tokens 0..7 and up threads for
// tokens 8..15.
template <int EPI>
__device__ __forceinline__ void pair_epilogue_tile(const PairClass& C, const PairTile& ti, uint32_t tbase,
                                                   float* stg, int lane, int q, int group, int gt, uint32_t rank) {
  const uint32_t bar_id = 1u + static_cast<uint32_t>(group);
  const int nslices = (ti.n + 15) / 16;
  if (EPI == kEpiSwiGLU) {
    const int jl = 32 * (q & 1) + lane;        // j within this CTA's 64
    const bool gate = q < 2;
    float* xg = stg;                           // [8][64] g of tokens 8..15
    float* xu = stg + 8 * 64;                  // [8][64] u of tokens 0..7
    __nv_bfloat16* hst = reinterpret_cast<__nv_bfloat16*>(stg + 16 * 64);  // [16][64] h
    const int64_t jbase = static_cast<int64_t>(ti.wb) * 128 + 64 * static_cast<int>(rank);
    for (int sl = group; sl < nslices; sl += 2) {
      uint32_t v[16];
      ptx::tmem_ld16(tbase + 16 * sl, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (gate)
          xg[c * 64 + jl] = __uint_as_float(v[8 + c]);
        else
          xu[c * 64 + jl] = __uint_as_float(v[c]);
      }
      ptx::named_barrier(bar_id, 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float g = gate ? __uint_as_float(v[c]) : xg[c * 64 + jl];
        const float u = gate ? xu[c * 64 + jl] : __uint_as_float(v[8 + c]);
        hst[(gate ? c : 8 + c) * 64 + jl] = __float2bfloat16_rn(swiglu(g, u));
      }
      ptx::named_barrier(bar_id, 128);
      {
        const int r = gt >> 3, k = gt & 7;  // row r of the slice, 16-byte chunk k (8 values of j)
        const int tok = 16 * sl + r;
        if (tok < ti.n) {
          const uint4 val = *reinterpret_cast<const uint4*>(hst + r * 64 + 8 * k);
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(C.out) +
                                    static_cast<int64_t>(ti.out_row0 + tok) * C.out_ld + jbase + 8 * k) = val;
        }
      }
      // no third barrier: the next slice rewrites hst only after its first barrier, which every thread reaches
      // after its read of hst above
    }
  } else {
    const int ol = 32 * q + lane;              // output column within this CTA's 128
    const int64_t obase = static_cast<int64_t>(ti.wb) * 256 + 128 * static_cast<int>(rank);
    for (int sl = group; sl < nslices; sl += 2) {
      uint32_t v[16];
      ptx::tmem_ld16(tbase + 16 * sl, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 16; ++c) stg[c * 128 + ol] = __uint_as_float(v[c]);
      ptx::named_barrier(bar_id, 128);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int i = gt + 128 * m;
        const int r = i >> 5, k = i & 31;  // row r of the slice, 16-byte chunk k (4 columns)
        const int tok = 16 * sl + r;
        if (tok < ti.n)
          *reinterpret_cast<float4*>(static_cast<float*>(C.out) + static_cast<int64_t>(ti.out_row0 + tok) * C.out_ld +
                                     obase + 4 * k) = *reinterpret_cast<const float4*>(stg + r * 128 + 4 * k);
      }
      ptx::named_barrier(bar_id, 128);
    }
  }
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    grouped_pair_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sW = base;
  const uint32_t sT = base + kPairStages * kPairStageWBytes;
  const uint32_t bars = sT + kPairStages * kPairStageTBytes;
  uint8_t* bars_ptr = base_ptr + kPairStages * (kPairStageWBytes + kPairStageTBytes);
  // barrier slots: full[kPairStages], empty[kPairStages], tmem_full[2], tmem_empty[2], drain
  const uint32_t full0 = bars, empty0 = bars + 8u * kPairStages, tfull0 = bars + 16u * kPairStages;
  const uint32_t tempty0 = tfull0 + 16u, drain_bar = tempty0 + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 16 * kPairStages + 40);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 16 * kPairStages + 44);

  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const uint32_t rank = ptx::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);   // used in the even CTA: its producer's arrival + both CTAs' bytes
      ptx::mbar_init(empty0 + 8u * s, 1);  // one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull0 + 8u * a, 1);
      ptx::mbar_init(tempty0 + 8u * a, 16);  // used in the even CTA: one arrival per epilogue warp of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int c = 0; c < 2; ++c) {
      ptx::tma_prefetch_desc(&p.tmW[c]);
      ptx::tma_prefetch_desc(&p.tmT[c]);
      ptx::tma_prefetch_desc(&p.tmTs[c]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 2 * kMaxN);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int lo = 0, hi = *reinterpret_cast<const volatile int32_t*>(p.num_tiles);
  if (p.range_lo != nullptr) lo = max(0, *reinterpret_cast<const volatile int32_t*>(p.range_lo));
  if (p.range_hi != nullptr) hi = min(hi, *reinterpret_cast<const volatile int32_t*>(p.range_hi));
  const int ncl = static_cast<int>(ptx::num_clusters_x());
  const int tfirst = lo + static_cast<int>(ptx::cluster_id_x());
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool failed = false, issued_any = false;
      const uint64_t pol_stream = ptx::make_policy_evict_first();
      const uint32_t full_even = ptx::map_to_rank(full0, 0);
      if (p.stall_flag != nullptr) {
        const uint64_t t0 = ptx::globaltimer();
        while (*reinterpret_cast<const volatile int32_t*>(p.stall_flag) == 0) {
          if (ptx::globaltimer() - t0 > tmo || *abort_flag) {
            pair_raise(p, abort_flag, kSiteStallFlag);
            failed = true;
            break;
          }
        }
      }
      for (int t = tfirst; !failed && t < hi; t += ncl) {
        const PairTile ti = decode_pair_tile(p, t, hi, lo);
        const PairClass& C = p.cls[ti.cls];
        const void* tW = &p.tmW[ti.cls];
        const int N = pair_width(ti.n);
        // this CTA's N/2 token rows in one box (the rows after them land in the slot and are not read)
        const bool small = N / 2 <= kPairTBoxRowsSmall;
        const void* tTok = small ? &p.tmTs[ti.cls] : &p.tmT[ti.cls];
        const uint32_t t_bytes = kPairKB * (small ? kPairTBoxRowsSmall : kPairTBoxRows) * 128u;
        const uint32_t bytes = 2u * (kPairStageWBytes + t_bytes);
        const int slot = C.w_group_mod <= 0
                             ? ti.group
                             : (C.w_slot_map != nullptr ? __ldg(C.w_slot_map + ti.group) : ti.group % C.w_group_mod);
        // gate/up: 64 gate rows and the same 64 up rows in one box at (0, j, 2 x slot, k block); down: 128 rows
        const int w_c1 = EPI == kEpiSwiGLU ? ti.wb * 128 + 64 * static_cast<int>(rank)
                                           : slot * C.w_group_rows + ti.wb * 256 + 128 * static_cast<int>(rank);
        const int t_row = ti.t_row0 + static_cast<int>(rank) * (N / 2);
        const bool stream = C.w_stream && ti.stream;
        for (int kb = 0; kb < C.kblocks; kb += kPairKB) {
          if (!ptx::wait_bounded(empty0 + 8u * stage, phase ^ 1u, tmo, abort_flag)) {
            pair_raise(p, abort_flag, kSiteProducerEmpty);
            failed = true;
            break;
          }
          if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8u * stage, bytes);
          const uint32_t fb = full_even + 8u * stage;
          const uint32_t w_dst = sW + stage * kPairStageWBytes;
          const uint32_t t_dst = sT + stage * kPairStageTBytes;
          if (EPI == kEpiSwiGLU) {
            if (stream)
              ptx::tma_load_4d_pair_hint(w_dst, tW, 0, w_c1, 2 * slot, kb, fb, pol_stream);
            else
              ptx::tma_load_4d_pair(w_dst, tW, 0, w_c1, 2 * slot, kb, fb);
          } else if (stream) {
            ptx::tma_load_3d_pair_hint(w_dst, tW, 0, w_c1, kb, fb, pol_stream);
          } else {
            ptx::tma_load_3d_pair(w_dst, tW, 0, w_c1, kb, fb);
          }
          ptx::tma_load_3d_pair(t_dst, tTok, 0, t_row, kb, fb);
          issued_any = true;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed && issued_any) {
        // The loads already issued complete on the even CTA's barrier, which this CTA cannot wait on: give them
        // time to land (bounded) before the CTA can exit.
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000u) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      int stage = 0, local = 0;
      uint32_t phase = 0;
      bool failed = false, issued_any = false;
      for (int t = tfirst; t < hi; t += ncl, ++local) {
        const PairTile ti = decode_pair_tile(p, t, hi, lo);
        const PairClass& C = p.cls[ti.cls];
        const int acc = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!ptx::wait_bounded(tempty0 + 8u * acc, (use & 1u) ^ 1u, tmo, abort_flag)) {
          pair_raise(p, abort_flag, kSiteMmaTmemEmpty);
          failed = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kMaxN);
        const int N = pair_width(ti.n);
        const uint32_t idesc = ptx::idesc_bf16_f32(256u, static_cast<uint32_t>(N));
        const uint32_t t_kb_bytes = (N / 2 <= kPairTBoxRowsSmall ? kPairTBoxRowsSmall : kPairTBoxRows) * 128u;
        for (int kb = 0; kb < C.kblocks; kb += kPairKB) {
          if (!ptx::wait_bounded(full0 + 8u * stage, phase, tmo, abort_flag)) {
            pair_raise(p, abort_flag, kSiteMmaFull);
            failed = true;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int j = 0; j < kPairKB; ++j) {
            // K block kb + j: its weight rows (16 KB) and token rows follow those of block kb + j - 1 in the slot
            const uint64_t a_desc = ptx::sw128_kmajor_desc(sW + stage * kPairStageWBytes + j * 16384u);
            const uint64_t b_desc = ptx::sw128_kmajor_desc(sT + stage * kPairStageTBytes + j * t_kb_bytes);
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk)
              ptx::umma_bf16_pair(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc, (kb | j | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(empty0 + 8u * stage, 0x3);  // frees the stage in both CTAs
          issued_any = true;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (failed) break;
        ptx::umma_commit_pair(tfull0 + 8u * acc, 0x3);  // accumulator ready in both CTAs
      }
      if (failed && issued_any) {
        int no_abort = 0;
        ptx::umma_commit_pair(drain_bar, 0x1);
        if (!ptx::wait_bounded(drain_bar, 0u, tmo, &no_abort))
          atomicCAS(p.err, 0, dev_error_code(kDevErrTimeout, kSiteDrain, static_cast<int>(blockIdx.x)));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9 of both CTAs)
    const int q = warp & 3;
    const int group = (warp - 2) / 4;
    const int gt = (warp - 2 - 4 * group) * 32 + lane;
    float* stg = reinterpret_cast<float*>(bars_ptr + kBarRegionBytes) + group * (8192 / 4);
    const uint32_t tempty_even = ptx::map_to_rank(tempty0, 0);
    int local = 0;
    for (int t = tfirst; t < hi; t += ncl, ++local) {
      const PairTile ti = decode_pair_tile(p, t, hi, lo);
      const int acc = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      bool ok = ptx::wait_bounded(tfull0 + 8u * acc, use & 1u, tmo, abort_flag);
      // all eight warps take the same decision (each group meets at named barriers in the epilogue)
      ok = ptx::named_barrier_and(3, 256, ok);
      if (!ok) {
        if (warp == 2 && lane == 0) pair_raise(p, abort_flag, kSiteEpilogueFull);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kMaxN);
      pair_epilogue_tile<EPI>(p.cls[ti.cls], ti, tbase, stg, lane, q, group, gt, rank);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(tempty_even + 8u * acc);
    }
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while the other may still signal its barriers or read its shared memory
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, 2 * kMaxN);
  }
}

int g_pair_clusters = 0;

}  // namespace

cudaError_t prepare_pair_kernels() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(grouped_pair_kernel<kEpiF32>, attr, kPairSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_pair_kernel<kEpiSwiGLU>, attr, kPairSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int n[2] = {0, 0};
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 2;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    e = i == 0 ? cudaOccupancyMaxActiveClusters(&n[i], grouped_pair_kernel<kEpiF32>, &cfg)
               : cudaOccupancyMaxActiveClusters(&n[i], grouped_pair_kernel<kEpiSwiGLU>, &cfg);
  }
  if (e != cudaSuccess) return e;
  g_pair_clusters = std::min(n[0], n[1]);
  return g_pair_clusters > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

int pair_cluster_slots() { return g_pair_clusters; }

cudaError_t launch_grouped_pair(const PairParams& p, int epilogue, int max_tiles, cudaStream_t stream) {
  if (max_tiles <= 0) return cudaSuccess;
  if (g_pair_clusters <= 0) return cudaErrorInvalidConfiguration;
  const int grid = 2 * std::min(g_pair_clusters, max_tiles);
  if (epilogue == kEpiSwiGLU)
    grouped_pair_kernel<kEpiSwiGLU><<<grid, kPairThreads, kPairSmemBytes, stream>>>(p);
  else
    grouped_pair_kernel<kEpiF32><<<grid, kPairThreads, kPairSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
