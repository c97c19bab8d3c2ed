/*
 * moe_prefill.h — C ABI of the expert-major chunked MoE prefill layer for NVIDIA GB300 (sm_103a), one GPU.
 *
 * What it computes. The routed-expert (MoE) layer of long-prompt prefill, run expert-major in chunks, as described by
 * the pull-request pages "EXL3 Flash Next: deep prefill" (draft slice 3 of 7, sections "What" and "Exactness", and
 * the maintainer review "To land"), "EXL3 Flash Next: deep prefill (3/8)" (sections "What this changes", "Device
 * results"), "Flash Next EXL3: exact deep prefill" (introduction; "Completed final functional audit") and the
 * umbrella draft PR #1113 ("What it adds", "Memory and execution split", "Latest prefill efficiency candidate").
 * For every chunk of consecutive tokens:
 *   1. router logits l = x . W_router^T (bf16 inputs, fp32 tensor-core accumulation);
 *   2. top-k experts per token by logit, an exact tie going to the lower expert id; the selection equals the one
 *      made on the plain float64 logits (ambiguous cases are recomputed in float64); weights = softmax over the k
 *      selected logits (renormalised);
 *   3. per-chunk member lists: histogram, exclusive scan and a stable permutation of the (token, slot) pairs into
 *      expert-major order (no atomics);
 *   4. grouped gate/up GEMM per touched expert with fused SwiGLU: h = bf16(silu(x.Wg^T) * (x.Wu^T));
 *   5. grouped down GEMM: y = h . W_down^T (fp32);
 *   6. the shared expert on every token (same FFN, weight 1);
 *   7. the canonical combine: out = bf16( (sum over slots in ascending expert id of w*y, in float32, from +0.0f,
 *      each product and sum rounded separately) + shared ).
 * The output is bit-identical for every chunk size (including one pass over all tokens) and from run to run.
 *
 * Conventions.
 *   - Every tensor is row-major and dense; bf16 tensors are passed as raw 16-bit patterns (void pointers).
 *   - Weights are "K-major": W_router [E][H]; W_gu [E][2I][H] with rows 0..I-1 the gate and rows I..2I-1 the up
 *     projection of each expert; W_down [E][H][I]; shared Ws_gu [2I_s][H]; Ws_down [H][I_s].
 *   - Pointers marked "device" must point to memory of the current CUDA device, 16-byte aligned.
 *   - The caller owns every buffer, including the workspace. The library allocates no device memory. A plan holds
 *     host state only (sizes, TMA descriptors, pointers, optional timing events) and must not outlive the weights.
 *   - Calls enqueue work on the given stream and return; a status of MOE_OK means "enqueued". Errors found on the
 *     host are returned at once and leave the stream untouched. Errors found on the device (a bounded wait that
 *     gave up, a failed bounds check) are written to the workspace error word, which moe_prefill_check() reports.
 *   - No call throws, exits, aborts or traps. Messages for the last non-OK status of the calling thread come from
 *     moe_prefill_last_error().
 *   - Streams are cudaStream_t values; 0 is the legacy default stream.
 */
#ifndef MOE_PREFILL_H
#define MOE_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,    /* null / misaligned pointer, negative size, chunk < 1, ... */
  MOE_ERR_UNSUPPORTED = -2,    /* dims outside what the kernels handle (see moe_prefill_plan) */
  MOE_ERR_WORKSPACE = -3,      /* workspace missing or smaller than moe_prefill_plan reported */
  MOE_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed (message has the CUDA error) */
  MOE_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up a bounded wait (reported by moe_prefill_check) */
  MOE_ERR_ARCH = -6,           /* the current device is not sm_103 or the kernels do not load on it */
  MOE_ERR_DEVICE_BOUNDS = -7   /* a device-side bounds check failed (reported by moe_prefill_check) */
} moe_status;

typedef struct {
  int32_t hidden;        /* H: multiple of 64 */
  int32_t n_experts;     /* E: routed experts, multiple of 16, 16..1024 */
  int32_t inter;         /* I: routed expert intermediate size, multiple of 64 */
  int32_t top_k;         /* k: 1..min(E, 32) */
  int32_t shared_inter;  /* I_s: 0 = no shared expert, else a multiple of 64 */
  int32_t renormalize;   /* must be 1: weights are the softmax over the selected logits */
  int32_t max_chunk;     /* largest chunk size (tokens) a run may use; sizes the workspace */
  int32_t offload_slots; /* 0: expert weights resident in device memory. S > 0: w_gu / w_down are pinned host
                            banks, streamed through a ring of S expert slots in the workspace (S even, S <= E,
                            S/2 divides E) */
} moe_dims;

typedef struct moe_plan* moe_plan_t;

/*
 * moe_prefill_plan — validate the layer's sizes, bind its weights and build the TMA descriptors.
 *   dims            in: sizes (see moe_dims for the accepted ranges).
 *   w_router        device bf16 [E][H].
 *   w_gu            device bf16 [E][2I][H] (gate rows, then up rows, per expert).
 *   w_down          device bf16 [E][H][I].
 *   ws_gu, ws_down  device bf16 [2I_s][H] and [H][I_s]; both NULL when shared_inter == 0.
 *   With offload_slots = S > 0, w_gu and w_down are page-locked HOST memory (cudaHostAlloc / cudaHostRegister)
 *   in the same layouts; the router and shared-expert weights stay in device memory. (Offloaded experts follow
 *   the umbrella PR #1113, "What it adds" / "Memory and execution split": pinned host banks, device expert
 *   lines, asynchronous host-to-device staging; and the deep-prefill draft, "What": a ring of staged expert
 *   lines overlapped with compute.)
 *   workspace_bytes out: bytes of device workspace moe_prefill_run needs for chunks up to max_chunk.
 *   plan            out: the plan; free it with moe_prefill_destroy.
 * Requires the current device to be sm_103 (else MOE_ERR_ARCH). Allocates no device memory. Thread-compatible:
 * one plan must not be used by two threads at once.
 */
moe_status moe_prefill_plan(const moe_dims* dims, const void* w_router, const void* w_gu, const void* w_down,
                            const void* ws_gu, const void* ws_down, size_t* workspace_bytes, moe_plan_t* plan);

/*
 * moe_prefill_plan_mxfp8 — moe_prefill_plan for routed experts stored as block-scaled FP8 (MXFP8).
 * The deep-prefill draft's review ("To land") quantises the weights of prompt tiles (NVFP4) and asks for the same
 * bytes as decode; this is the 8-bit block-scaled member of that family (OCP Microscaling Formats v1.0, MXFP8
 * E4M3), for the bytes that bound the layer: the routed experts' weights are read at half the bf16 size.
 *   w_gu_codes    device uint8 [E][2I][H]: E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 fraction bits;
 *                 exponent field 0 = subnormals m/8 * 2^-6), same row order as w_gu.
 *   w_gu_scales   device uint8 [E][H/32][2I]: E8M0 scale s of each 32-wide K block (value 2^(s-127)), one plane
 *                 of 2I bytes per K block.
 *   w_down_codes  device uint8 [E][H][I];  w_down_scales: device uint8 [E][I/32][H].
 *   Other arguments as for moe_prefill_plan (router and shared expert stay bf16). With offload_slots > 0 the two
 *   code arrays are pinned host memory staged through the ring like bf16 banks (half the bytes over the host
 *   link); the scale arrays stay in device memory in every case. All pointers 16-byte aligned.
 * A weight is code * 2^(s-127). The kernels decode each tile to bf16 in shared memory and run the bf16 tensor-core
 * path on it; the results equal, byte for byte, moe_prefill_plan on the decoded bf16 weights, provided every
 * decoded weight is exactly a bf16 value: no NaN code (0x7F, 0xFF), scales in [10, 246] (then every code times
 * its scale is a normal bf16 number). These are not checked on the device.
 */
moe_status moe_prefill_plan_mxfp8(const moe_dims* dims, const void* w_router, const uint8_t* w_gu_codes,
                                  const uint8_t* w_gu_scales, const uint8_t* w_down_codes,
                                  const uint8_t* w_down_scales, const void* ws_gu, const void* ws_down,
                                  size_t* workspace_bytes, moe_plan_t* plan);

/*
 * moe_prefill_plan_nvfp4 — moe_prefill_plan for routed experts stored as block-scaled FP4 (NVFP4), the format the
 * deep-prefill draft's review ("To land") names for prompt tiles: a quarter of the bf16 bytes.
 *   w_gu_codes    device (or, with offload_slots > 0, pinned host) uint8 [E][2I][H/2]: E2M1 codes (1 sign, 2 exponent
 *                 bits with bias 1, 1 fraction bit; values 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte, element 2j in
 *                 the low nibble of byte j.
 *   w_gu_scales   device uint8 [E][H/16][2I]: the E4M3 scale of each 16-wide K block (not NaN), one plane per block.
 *   w_down_codes  uint8 [E][H][I/2];  w_down_scales: device uint8 [E][I/16][H].
 *   Other arguments and behaviour as for moe_prefill_plan_mxfp8. No tensor-wide scale (it is 1). A code times its
 *   scale (at most 2 x 4 significant bits, magnitude 2^-10 .. 2688) is always exactly a bf16 value, so the results
 *   equal, byte for byte, moe_prefill_plan on the decoded bf16 weights.
 */
moe_status moe_prefill_plan_nvfp4(const moe_dims* dims, const void* w_router, const uint8_t* w_gu_codes,
                                  const uint8_t* w_gu_scales, const uint8_t* w_down_codes,
                                  const uint8_t* w_down_scales, const void* ws_gu, const void* ws_down,
                                  size_t* workspace_bytes, moe_plan_t* plan);

/*
 * moe_prefill_run — the layer over T tokens, in chunks of `chunk` tokens (the last chunk may be shorter).
 * "Flash Next EXL3: exact deep prefill" (introduction): prompt rows are run expert-major in chunks of consecutive
 * tokens; "Completed final functional audit": the output bytes are the same at chunks 256/1,024/2,048 and equal to
 * one batched pass. Steps 1-7 of the file comment, per chunk.
 *   x               device bf16 [T][H].
 *   T               tokens (T == 0: no-op, MOE_OK).
 *   chunk           1..max_chunk tokens per chunk; chunk >= T is one single pass.
 *   workspace       device buffer of at least workspace_bytes (moe_prefill_plan), 256-byte aligned. It holds the
 *                   device error word of the most recent run. Several plans (the layers of a model) may share one
 *                   workspace if their runs on it are ordered on the GPU (for example all on one stream); runs
 *                   that overlap on the GPU race on it. What a run leaves in it for later runs (an offloaded
 *                   plan's hot set and slot map, a prefetched first window) is recorded per workspace address and
 *                   device: a run uses it only if that plan, with that hot set, put it there, and stages it again
 *                   otherwise. The library keeps these records for the 256 most recently used workspaces; a run on
 *                   a workspace whose record was dropped stages what it needs again. Before freeing a workspace or
 *                   reusing its memory, call moe_prefill_forget_workspace.
 *   out             device bf16 [T][H] (may not alias x).
 *   topk_id         device int32 [T][k] or NULL: selected expert ids per token, ascending.
 *   topk_w          device float [T][k] or NULL: their weights (same order).
 *   expert_offsets  device int32 [n_chunks][E+1] or NULL: per-chunk exclusive offsets of each expert's rows.
 *   row_token       device int32 [T*k] or NULL: row j of chunk c (chunk-local index) at c*chunk*k + j holds the
 *                   global id of the token placed in that row (rows ordered by expert, then token).
 *   compute         stream for all kernels.
 *   copy            resident weights: must be NULL. Offloaded experts: the stream for the host-to-device expert
 *                   copies, or NULL for one owned by the plan. For every chunk the experts are staged in windows of
 *                   S/2 consecutive experts into alternate halves of the ring; a window's GEMMs wait for its copies
 *                   and a copy waits until the GEMMs of the window that last used its half have finished. Which
 *                   experts of a window are staged depends on the staging mode (moe_prefill_set_offload_copy): by
 *                   default only those the chunk routes rows to; with MOE_OFFLOAD_COPY_ALL every expert.
 * Returns after enqueueing; call moe_prefill_check(workspace, compute) for device-side errors.
 */
moe_status moe_prefill_run(moe_plan_t plan, const void* x, int64_t T, int32_t chunk, void* workspace,
                           size_t workspace_bytes, void* out, int32_t* topk_id, float* topk_w,
                           int32_t* expert_offsets, int32_t* row_token, moe_stream_t compute, moe_stream_t copy);

/*
 * moe_prefill_run_host — moe_prefill_run for activations in host memory, with the copies overlapped.
 *   x_host     pinned host bf16 [T][H] (cudaHostAlloc / cudaHostRegister), read.
 *   out_host   pinned host bf16 [T][H], written.
 *   x_dev, out_dev   device bf16 [T][H] staging buffers owned by the caller (16-byte aligned).
 *   Other arguments as for moe_prefill_run.
 * The X rows of each routing span are copied to x_dev on a stream of the plan in two parts, the span's first
 * chunk and the rest: the first chunk's routing and expert GEMMs start once its rows have landed while the rest is
 * in flight (routing of the rest waits for them). Each chunk's out rows are copied back as soon as its combine has
 * written them, beside the next chunks' GEMMs. The results (out_host, and the optional device outputs) are those of
 * moe_prefill_run on x_dev; every copy is ordered after the work enqueued on `compute` before the call, and all of
 * them have finished when `compute` reaches the end of the run.
 */
moe_status moe_prefill_run_host(moe_plan_t plan, const void* x_host, int64_t T, int32_t chunk, void* workspace,
                                size_t workspace_bytes, void* x_dev, void* out_dev, void* out_host, int32_t* topk_id,
                                float* topk_w, int32_t* expert_offsets, int32_t* row_token, moe_stream_t compute,
                                moe_stream_t copy);

/*
 * moe_prefill_combine — the canonical combine alone (the same kernel run uses). "Flash Next EXL3: exact deep
 * prefill" (introduction): each token's expert contributions are reduced in one canonical, fixed order, which is
 * what makes the output independent of the chunk size; here: ascending expert id, float32, shared expert last.
 *   y          device float [R][H]: per-row expert outputs.
 *   w          device float [n][k]: weights, slot order = ascending expert id.
 *   token_row  device int32 [n][k]: row of y for each (token, slot); every value in [0, R).
 *   s          device float [n][H] or NULL: shared-expert output added last.
 *   out        device bf16 [n][H].
 * n >= 0, 1 <= k <= 32, H a positive multiple of 4. Row indices are not range-checked on the device.
 */
moe_status moe_prefill_combine(const float* y, const float* w, const int32_t* token_row, const float* s, int64_t n,
                               int32_t k, int32_t H, void* out, moe_stream_t stream);

/*
 * Float64 combine for an expert-parallel split ("EXL3 Flash Next: deep prefill (3/8)", "What this changes": the
 * tensor-parallel prefill partials are float64; "Checklist": they are summed in float64 and rounded once, to float32,
 * at the finish, so a split over two GPUs reproduces one GPU bit for bit). The pages leave the order inside a partial
 * open; this library fixes it as a complete binary tree over the expert ids 0 .. Ep-1, Ep = the least power of two
 * >= n_experts: leaf e = w*y of the token's slot routed to expert e (the product of two floats, exact in float64),
 * +0.0 for an expert the token did not choose; each inner node = left + right in float64 (round to nearest).
 * A part of a split is one of n_parts aligned blocks of Ep/n_parts ids, i.e. a subtree; the finish sums the parts
 * pairwise in the same tree, adds the shared expert's output (float64), rounds once to float32 and then to bf16
 * (ties to even). Splitting therefore changes no operation: partial + finish over any n_parts equals
 * moe_prefill_combine_f64 bit for bit.
 *
 * moe_prefill_combine_partial_f64 — one part's float64 value.
 *   y, w, token_row   as for moe_prefill_combine; token_row is read only for slots whose expert is in the part
 *                     (an expert-parallel rank needs y rows for its own experts only).
 *   topk_id   device int32 [n][k]: each slot's expert id in [0, n_experts), distinct within a token, any slot order
 *             (an id outside the part is skipped; a repeated id counts once, in its first slot).
 *   n_experts 1..1024.  n_parts: a power of two <= Ep.  part: 0 <= part < n_parts, experts
 *             [part*Ep/n_parts, (part+1)*Ep/n_parts).
 *   partial   device double [n][H], 16-byte aligned.
 * n >= 0, 1 <= k <= 32, H a positive multiple of 4, y 16-byte aligned. Row indices are not range-checked on the
 * device.
 */
moe_status moe_prefill_combine_partial_f64(const float* y, const float* w, const int32_t* token_row,
                                           const int32_t* topk_id, int64_t n, int32_t k, int32_t H,
                                           int32_t n_experts, int32_t n_parts, int32_t part, double* partial,
                                           moe_stream_t stream);

/*
 * moe_prefill_combine_finish_f64 — sum the parts, add the shared expert, round.
 *   partials  HOST array of n_parts DEVICE pointers, part 0 first, each double [n][H] (16-byte aligned).
 *   n_parts   a power of two, 1..16.
 *   s         device float [n][H] or NULL.
 *   out       device bf16 [n][H];  out_f32: device float [n][H] or NULL (the float32 value before the bf16
 *             rounding). All 16-byte aligned; H a positive multiple of 4.
 */
moe_status moe_prefill_combine_finish_f64(const double* const* partials, int32_t n_parts, const float* s, int64_t n,
                                          int32_t H, void* out, float* out_f32, moe_stream_t stream);

/*
 * moe_prefill_combine_f64 — the unsplit float64 combine in one kernel (one part covering every expert, then the
 * finish); the kernel the layer runs under MOE_COMBINE_F64_TREE. Arguments as above.
 */
moe_status moe_prefill_combine_f64(const float* y, const float* w, const int32_t* token_row, const int32_t* topk_id,
                                   const float* s, int64_t n, int32_t k, int32_t H, int32_t n_experts, void* out,
                                   float* out_f32, moe_stream_t stream);

/*
 * How offloaded experts reach the ring (plans with offload_slots > 0).
 *   MOE_OFFLOAD_COPY_ROUTED  (default where the device can read the pinned banks directly) a small kernel on the
 *     copy stream stages, per chunk and window, only the experts that the chunk's member lists route rows to,
 *     reading the banks through their device-accessible addresses; the decision is made on the device (umbrella
 *     PR #1113, "Memory and execution split": device-planned paths fill expert lines from mapped host banks;
 *     "Latest measured follow-up": transfer volume is the cost). Counts in MOE_STATS_EXPERTS_COPIED / _SKIPPED.
 *   MOE_OFFLOAD_COPY_ALL  the copy engines stage every expert of every window (two cudaMemcpyAsync per window).
 * Both give the same output bytes. moe_prefill_set_offload_copy fails with MOE_ERR_UNSUPPORTED for ROUTED when
 * the device cannot read the banks directly, and with MOE_ERR_INVALID_ARG for a plan without offloaded experts.
 */
enum { MOE_OFFLOAD_COPY_ALL = 0, MOE_OFFLOAD_COPY_ROUTED = 1 };
moe_status moe_prefill_set_offload_copy(moe_plan_t plan, int32_t mode);

/*
 * moe_prefill_set_hot_experts — keep n_hot offloaded experts resident ("hot set") in extra slots after the ring,
 * for plans with offload_slots > 0. Umbrella PR #1113: "Persistent expert-profile checkpoint" keeps per-expert use
 * counts as placement priors that warm resident expert lines at startup, and "Latest measured follow-up" accounts
 * the copied bytes by category (demand, initial prefetch, cross-layer prefetch); the plain reading here: the caller
 * names the most used experts (e.g. by the expert_offsets of an earlier run), they are staged into a workspace by
 * the first run of this plan there, and no chunk stages them again.
 *   hot_ids          host int32 [n_hot], distinct expert ids in [0, E); copied, the caller keeps ownership.
 *   n_hot            0 .. E; 0 removes the set.
 *   workspace_bytes  out (may be NULL): the workspace size later runs need (the set's slots are part of it:
 *                    n_hot x one expert's gate/up + down bytes more than without a set).
 * The hot experts are copied from the pinned banks on the copy stream at the start of the next run on a workspace,
 * and again at the start of a later run there whenever another plan (or this plan with another set) ran on that
 * workspace in between; the routed staging kernel skips them (counted in MOE_STATS_EXPERTS_HOT) and the
 * GEMMs read them from their slots. With MOE_OFFLOAD_COPY_ALL every window is still copied whole. Output bytes are
 * the same with and without a set. Errors: MOE_ERR_INVALID_ARG for a NULL plan, a plan without offloaded experts,
 * n_hot out of range, hot_ids NULL with n_hot > 0, an id out of range or given twice (the plan is then unchanged).
 */
moe_status moe_prefill_set_hot_experts(moe_plan_t plan, const int32_t* hot_ids, int32_t n_hot,
                                       size_t* workspace_bytes);

/*
 * moe_prefill_prefetch — cross-layer prefetch for plans with offload_slots > 0: stages, on `copy`, the first window
 * of experts (ids 0 .. offload_slots/2 − 1, every one of them: the next run's routing is not known yet) into the
 * ring of `workspace`, so that the next moe_prefill_run on that workspace starts its first chunk's GEMMs without
 * waiting for that window's copy. Umbrella PR #1113, "Latest measured follow-up": copies are accounted as demand,
 * initial prefetch and cross-layer prefetch; the plain reading: while one layer computes, the next layer's first
 * experts move. Call it once the previous layer's run (or this plan's own last run) is enqueued.
 *   workspace, workspace_bytes  the workspace the next run of this plan will use (at least the plan's size).
 *   copy                        stream for the copies (NULL: the plan's own copy stream).
 * The copy waits for an earlier prefetch into the same workspace and for the last run enqueued on it (of any plan):
 * if that run's ring lies at the same place as this plan's (same sizes, slots and hot-set size), for its last
 * release of the ring's first half, so the copy overlaps that run's tail; otherwise for its end. The next run of
 * this plan on that workspace consumes the prefetch (its first window's GEMMs wait for these copies) unless
 * moe_prefill_set_hot_experts was called in between; a run of any other plan there drops it, and all of that run's
 * work waits for these copies first. The prefetched window is not counted in the staging statistics. Output bytes
 * do not change. Not available for moe_prefill_run_noalloc (its array has no address the caller can pass). Errors: MOE_ERR_INVALID_ARG (NULL plan, plan without offloaded experts, misaligned workspace, wrong
 * device), MOE_ERR_WORKSPACE (workspace too small), MOE_ERR_CUDA.
 */
moe_status moe_prefill_prefetch(moe_plan_t plan, void* workspace, size_t workspace_bytes, moe_stream_t copy);

/*
 * moe_prefill_forget_workspace — drop what the library remembers about `workspace` on the current device (the
 * plan that ran there last, its hot set, a pending prefetch: see moe_prefill_run). Call it before the workspace's
 * memory is freed or used for anything else: the records are keyed by address, so memory reused at the same address
 * would otherwise be trusted to hold what a plan staged there. Waits (host-side) until the runs and copies the record
 * knows of have finished. A workspace the library does not know is ignored (MOE_OK). Errors: MOE_ERR_INVALID_ARG
 * (NULL), MOE_ERR_CUDA. No counterpart in the pages: a convenience of this library's workspace records.
 */
moe_status moe_prefill_forget_workspace(void* workspace);

/* Combine of the layer: the float32 canonical reduction (default) or the float64 tree above. */
enum { MOE_COMBINE_F32 = 0, MOE_COMBINE_F64_TREE = 1 };
/* moe_prefill_set_combine — select the combine of later runs of this plan. */
moe_status moe_prefill_set_combine(moe_plan_t plan, int32_t mode);

/*
 * moe_prefill_set_cta_pairs — which expert projections of later runs of this plan run on CTA pairs: a mask of
 * MOE_PAIRS_GATE_UP and MOE_PAIRS_DOWN (default MOE_PAIRS_GATE_UP where the plan allows it; 0: both on single CTAs).
 * The pair kernel takes an expert's weights as the 256-row operand of tcgen05.mma.cta_group::2 (two SMs share one
 * tile) and its member rows in steps of 32; the single-CTA kernel takes 128 member rows against 256 weight rows.
 * Both accumulate every output element over K in the same order, so the choice changes no output byte. Needs bf16
 * expert weights, inter and shared_inter multiples of 128 and hidden a multiple of 256: MOE_ERR_UNSUPPORTED for a
 * non-zero mask otherwise. MOE_ERR_INVALID_ARG: NULL plan or unknown bits.
 * moe_prefill_cta_pairs — the plan's current mask (0 for NULL).
 * The expert-major projections they compute: "Flash Next EXL3: exact deep prefill", introduction.
 */
enum { MOE_PAIRS_GATE_UP = 1, MOE_PAIRS_DOWN = 2 };
moe_status moe_prefill_set_cta_pairs(moe_plan_t plan, int32_t which);
int32_t moe_prefill_cta_pairs(moe_plan_t plan);

/*
 * moe_prefill_check — wait for `stream`, then read and clear the device error word in the workspace header.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BOUNDS or MOE_ERR_CUDA (a failed synchronisation).
 */
moe_status moe_prefill_check(void* workspace, moe_stream_t stream);

/* moe_prefill_destroy — free a plan (host memory and its timing events). NULL is ignored. */
void moe_prefill_destroy(moe_plan_t plan);

/* moe_prefill_last_error — message for the last non-OK status returned on this thread ("" if none). */
const char* moe_prefill_last_error(void);

/*
 * moe_prefill_run_noalloc — moe_prefill_run for callers that cannot allocate device memory.
 * No counterpart in the pages this layer follows: it is a convenience of this library.
 *
 * Who needs it: callers that must not call cudaMalloc where they run the layer — code whose device memory belongs
 * to another allocator or pool (an allocation behind its back breaks its accounting and can fail once the pool has
 * reserved the GPU), serving loops that forbid allocation after start-up (cudaMalloc/cudaFree synchronise the
 * device), and plug-ins that are only handed input and output pointers. It computes exactly what moe_prefill_run
 * computes (same kernels, same bytes out) but keeps its scratch in a fixed array of MOE_NOALLOC_WORKSPACE_BYTES
 * inside the library, so it allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   plan, x, T, chunk, out, topk_id, topk_w, expert_offsets, row_token, stream: as for moe_prefill_run.
 *   device_status   device int32 or NULL: receives the run's device error word once the run's work has finished on
 *                   `stream` (0 = no device-side error; otherwise the code moe_prefill_check would decode).
 * Limits and behaviour:
 *   - The plan's workspace_bytes must be at most MOE_NOALLOC_WORKSPACE_BYTES; larger plans get MOE_ERR_WORKSPACE
 *     with a message (use a smaller max_chunk, or moe_prefill_run).
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - The array is shared by all calls on a device and keeps the last call's contents. Each run first clears the
 *     part that must start at zero (error word, counters) and writes the per-run bytes whose values reach an
 *     output before reading them. What an offloaded plan keeps between runs (its hot set's slots and slot map) is
 *     recorded as for any shared workspace: a plan whose last run here was not the last run on the array stages
 *     them again. Calls whose work overlaps on the GPU (e.g. on different streams) race on the array: serialise
 *     them.
 *   - moe_prefill_prefetch and moe_prefill_check take a workspace address and so do not apply to these runs;
 *     device_status takes the place of moe_prefill_check.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture.
 */
#define MOE_NOALLOC_WORKSPACE_BYTES ((size_t)64 << 20)
moe_status moe_prefill_run_noalloc(moe_plan_t plan, const void* x, int64_t T, int32_t chunk, void* out,
                                   int32_t* topk_id, float* topk_w, int32_t* expert_offsets, int32_t* row_token,
                                   int32_t* device_status, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------------------------
 * Diagnostics. These are part of the ABI for measurement and tests; the layer needs none of them.
 * ------------------------------------------------------------------------------------------------------------ */

/* Kernel kinds for moe_prefill_kernel_times, in launch order within a chunk. */
enum {
  MOE_KERNEL_NORMS = 0,  /* router row norms + header reset (once per run) */
  MOE_KERNEL_ROUTER = 1, /* router GEMM */
  MOE_KERNEL_TOPK = 2,    /* top-k selection + float64 recheck of ambiguous tokens (2 kernels) */
  MOE_KERNEL_COUNT = 3,
  MOE_KERNEL_SCAN = 4,
  MOE_KERNEL_PERMUTE = 5,
  MOE_KERNEL_GATE_UP = 6, /* grouped gate/up GEMM + SwiGLU (routed + shared) */
  MOE_KERNEL_DOWN = 7,    /* grouped down GEMM (routed + shared) */
  MOE_KERNEL_COMBINE = 8,
  MOE_KERNEL_KINDS = 9
};

/* Enable (1) or disable (0) per-kernel CUDA-event timing of later runs of this plan. */
moe_status moe_prefill_set_profiling(moe_plan_t plan, int32_t enable);

/* Synchronise on the recorded events and return, per kernel kind, the summed device milliseconds and the number
   of launches timed since the last call (arrays of MOE_KERNEL_KINDS entries; either may be NULL). Clears them. */
moe_status moe_prefill_kernel_times(moe_plan_t plan, double* ms, int64_t* launches);

/* The launches timed since the last call (profiling enabled), in the order they were enqueued: kind, start and end
   in milliseconds from the start of the first one (CUDA events on each launch's stream). Writes min(count,
   capacity) entries, sets *count to the number of timed launches, synchronises on the events and clears them (as
   moe_prefill_kernel_times does). */
moe_status moe_prefill_kernel_trace(moe_plan_t plan, int32_t* kinds, float* start_ms, float* end_ms, int32_t capacity,
                                    int32_t* count);

/* Total kernels launched by this plan since it was created. */
int64_t moe_prefill_launch_count(moe_plan_t plan);

/* Bound, in nanoseconds, on every device-side wait of later runs of this plan (default 2e9). */
moe_status moe_prefill_set_wait_timeout(moe_plan_t plan, uint64_t timeout_ns);

/* Statistics of the most recent run on `workspace` (synchronises `stream`), in this order: */
enum {
  MOE_STATS_CHUNKS = 0,       /* chunks processed */
  MOE_STATS_FLAGGED = 1,      /* tokens whose fp32 top-k was not certain and went to the float64 recheck */
  MOE_STATS_BY_FLOAT = 2,     /* ... decided by float sums of the exact products */
  MOE_STATS_BY_DOUBLE = 3,    /* ... decided by double sums */
  MOE_STATS_BY_SEQUENTIAL = 4,/* ... decided by the sequential float64 sums */
  MOE_STATS_BY_MANY = 5,      /* ... with more candidates than the recheck list holds (sequential sums) */
  MOE_STATS_EXPERTS_COPIED = 6,  /* offloaded experts staged into the ring, summed over chunks (routed mode) */
  MOE_STATS_EXPERTS_SKIPPED = 7, /* offloaded experts left out: their chunk routed no row to them (routed mode) */
  MOE_STATS_EXPERTS_HOT = 8,     /* offloaded experts with rows in a chunk, read from the hot set (routed mode) */
  MOE_STATS_COUNT = 9
};
/* Writes min(n_stats, ...) entries of the list above to stats (entries past MOE_STATS_COUNT are 0). */
moe_status moe_prefill_run_stats(void* workspace, moe_stream_t stream, int32_t* stats, int32_t n_stats);

/*
 * moe_prefill_debug_gemm — one dense GEMM through the same tcgen05 kernel the layer uses.
 *   epilogue 0:  c = float [m][n] = a . b^T with a bf16 [m][k_dim], b bf16 [n][k_dim]; n a multiple of 16.
 *   epilogue 1:  c = bf16 [m][n] = bf16(silu(a . bg^T) * (a . bu^T)) with b bf16 [2n][k_dim] holding the gate rows
 *                (0..n-1) then the up rows (n..2n-1); n a multiple of 64.
 *   k_dim a multiple of 64, m >= 1.
 *   err_word     device int32, must be 0 on entry; set to a non-zero code when a wait gives up.
 *   stall_flag   device int32 or NULL: when given, the load warp first waits for it to become non-zero (a test of
 *                the bounded-wait path: pass a zero flag and a short timeout_ns).
 *   timeout_ns   bound on every device-side wait (0 = default 2e9).
 */
moe_status moe_prefill_debug_gemm(const void* a, const void* b, void* c, int32_t m, int32_t n, int32_t k_dim,
                                  int32_t epilogue, int32_t* err_word, const int32_t* stall_flag,
                                  uint64_t timeout_ns, moe_stream_t stream);

/*
 * moe_prefill_debug_gemm_pairs — the same dense GEMM through the CTA-pair kernel the layer uses for its expert
 * projections (b as the 256-row weight operand, the rows of a in token tiles of at most 256).
 *   epilogue 0:  c = float [m][n] = a . b^T; n a multiple of 256.
 *   epilogue 1:  c = bf16 [m][n] = bf16(silu(a . bg^T) * (a . bu^T)), b = gate rows then up rows; n a multiple of 128.
 *   k_dim a multiple of 128, m >= 1.
 *   scratch      device memory of at least moe_prefill_debug_gemm_pairs_scratch(m, n, epilogue) bytes (16-byte
 *                aligned) for the tile list, which is copied there on `stream` from pageable host memory.
 *   err_word, stall_flag, timeout_ns: as for moe_prefill_debug_gemm.
 * MOE_ERR_UNSUPPORTED for other n or when no cluster of two CTAs fits; MOE_ERR_WORKSPACE for a short scratch.
 * moe_prefill_debug_gemm_pairs_scratch returns 0 for invalid arguments.
 */
size_t moe_prefill_debug_gemm_pairs_scratch(int32_t m, int32_t n, int32_t epilogue);
moe_status moe_prefill_debug_gemm_pairs(const void* a, const void* b, void* c, int32_t m, int32_t n, int32_t k_dim,
                                        int32_t epilogue, void* scratch, size_t scratch_bytes, int32_t* err_word,
                                        const int32_t* stall_flag, uint64_t timeout_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_PREFILL_H */
