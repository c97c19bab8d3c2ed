"""Benchmark of the expert-major chunked MoE prefill layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME] [--chunk C]

One step = one call of the layer (moe_prefill_run) over all tokens of the workload: per chunk the router GEMM,
top-k, histogram/scan/permute, grouped gate/up + SwiGLU, grouped down, shared expert and the canonical combine.
`value` is tokens/s over all ranks with inputs resident in device memory; `e2e` repeats the measurement through
the same call with the activations in pinned host memory, the host->device copy of x and the device->host copy of
the output inside the timed region. Prints one JSON line (rank 0).

--impl reference times the float64 CPU oracle (oracle/) on the host cores on a bounded sample of the same
workload: the reference arm of this layer is that plain CPU implementation.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer prefill tokens/s (1×GB300); grouped-GEMM tensor-pipe % of peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "e512_t16022"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--chunk", type=int, default=0, help="chunk size (default: the workload's first chunk size)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-single-pass", dest="single_pass", action="store_false",
                    help="skip the chunk = T (one pass over all tokens) figures, where the grouped GEMMs have enough "
                         "rows per expert to be tensor-bound")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count (profiling runs)")
    ap.add_argument("--combine", choices=["f32", "f64"], default="f32",
                    help="layer combine: canonical float32 (default) or the float64 tree over expert ids")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-size (1 and 8 token) latency lines")
    ap.add_argument("--weights", choices=["bf16", "mxfp8", "nvfp4"], default="bf16",
                    help="routed expert weights: bf16, MXFP8 (E4M3 codes + E8M0 scale per 32 along K) or NVFP4 "
                         "(E2M1 codes + E4M3 scale per 16 along K)")
    ap.add_argument("--hot-experts", type=int, default=0,
                    help="offloaded experts: keep the N experts routed in the most chunks of the warm-up run resident")
    ap.add_argument("--prefetch", action="store_true",
                    help="offloaded experts: after each run, stage the next run's first window (cross-layer prefetch)")
    ap.add_argument("--offload-copy", choices=["routed", "all"], default="routed",
                    help="offloaded experts: stage only the routed experts (kernel) or every expert (copy engines)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate_rate(units_per_rank: list, seconds_per_rank: list) -> float:
    """Whole-job throughput of weakly scaled replicas: all units processed over the slowest rank's time."""
    return sum(units_per_rank) / max(seconds_per_rank)


# ------------------------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, log_path: str | None = None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.log_path = log_path

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-lms", "200", "-i", self.gpu_id], stdout=subprocess.PIPE,
                                     stderr=subprocess.DEVNULL, text=True)
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=5)
        if self.log_path:
            with open(self.log_path, "w") as f:
                f.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_selector(torch, device_index: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


# ------------------------------------------------------------------------------------------------ helpers

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("expert_major_chunked_gb300/csrc/gemm.cu", "expert_major_chunked_gb300/csrc/gemm_pair.cu",
                "expert_major_chunked_gb300/csrc/swiglu.cuh", "expert_major_chunked_gb300/csrc/ptx.cuh",
                "expert_major_chunked_gb300/csrc/internal.h", "expert_major_chunked_gb300/csrc/route.cu"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, chunk: int):
    """DRAM bytes per gate/up launch from the committed ncu summary, if it was taken on the current kernel."""
    import re
    path = os.path.join(ROOT, "profiles", f"gate_up_{workload}_c{chunk}.md")
    if not os.path.exists(path):
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+kernel_source_hash:\s*([0-9a-f]+)", open(path).read())
    if not m or m.group(2) != kernel_source_hash():
        return None
    return int(m.group(1))


# ------------------------------------------------------------------------------------------------ reference arm

def run_reference(args, dist: Dist):
    if dist.rank != 0:
        dist.close()
        return
    import numpy as np
    import torch
    import oracle
    from expert_major_chunked_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    chunk = args.chunk or wl.chunks[0]
    inp = workloads.generate(wl)
    if args.weights != "bf16":  # the oracle runs on the decoded block-scaled weights
        inp = decoded_weights(inp, quantized_weights(inp, args.weights), args.weights)
    cores = oracle.num_threads()
    # calibrate, then size each step so that warm-up + timed steps fit in about two minutes
    t0 = time.perf_counter()
    oracle.moe_forward(inp, wl.top_k, token_idx=np.arange(min(32, wl.tokens)))
    rate = min(32, wl.tokens) / (time.perf_counter() - t0)
    per_step = int(max(1, min(wl.tokens, rate * 120.0 / (args.steps + args.warmup))))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.moe_forward(inp, wl.top_k, token_idx=rng.choice(wl.tokens, per_step, replace=False))
    secs = 0.0
    for _ in range(args.steps):
        idx = rng.choice(wl.tokens, per_step, replace=False)
        t0 = time.perf_counter()
        oracle.moe_forward(inp, wl.top_k, token_idx=idx)
        secs += time.perf_counter() - t0
    value = per_step * args.steps / secs
    sample = f"{per_step} random tokens per step of the {wl.tokens}-token workload, float64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, chunk, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    dist.close()


def workload_config(wl, chunk: int, n_gpus: int) -> dict:
    return {"workload": wl.name, "tokens": wl.tokens, "hidden": wl.hidden, "experts": wl.n_experts,
            "inter": wl.inter, "top_k": wl.top_k, "shared_inter": wl.shared_inter, "chunk": chunk,
            "router": "zipf(1.1) prior" if wl.zipf_prior else "uniform N(0,1) logits",
            "l2": "inputs larger than L2: every chunk streams all touched expert weights (GBs) from HBM",
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "1 GPU"}


# ------------------------------------------------------------------------------------------------ our arm

def cpu_baseline(inp, wl, budget_s: float = 10.0) -> dict:
    import numpy as np
    import oracle
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    probe = min(64, wl.tokens)
    oracle.moe_forward(inp, wl.top_k, token_idx=np.arange(probe))
    rate = probe / (time.perf_counter() - t0)
    n = int(min(wl.tokens, max(probe, rate * budget_s)))
    t0 = time.perf_counter()
    oracle.moe_forward(inp, wl.top_k, token_idx=np.arange(n))
    secs = time.perf_counter() - t0
    return {"value": n / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {wl.tokens} tokens, full layer in float64 ({secs:.1f} s)"}


WEIGHT_BYTES = {"bf16": 2.0, "mxfp8": 1.0 + 1.0 / 32.0, "nvfp4": 0.5 + 1.0 / 16.0}  # per routed weight, with scales
WEIGHT_DESC = {"bf16": "bf16",
               "mxfp8": "mxfp8 (E4M3 codes + E8M0 scale per 32 along K; bf16 tensor-core math)",
               "nvfp4": "nvfp4 (E2M1 codes + E4M3 scale per 16 along K; bf16 tensor-core math)"}


def quantized_weights(inp, fmt):
    from expert_major_chunked_gb300 import workloads
    return workloads.mxfp8_weights(inp) if fmt == "mxfp8" else workloads.nvfp4_weights(inp)


def decoded_weights(inp, q, fmt):
    """The inputs with the routed expert weights replaced by the oracle's decoding of their block-scaled form."""
    import numpy as np
    import torch
    import oracle
    deq = oracle.dequant_mxfp8 if fmt == "mxfp8" else oracle.dequant_nvfp4
    dec = lambda c, sc: torch.from_numpy(deq(c.numpy(), sc.numpy()).view(np.int16)).view(torch.bfloat16)
    return dict(inp, w_gu=dec(q["w_gu_q"], q["w_gu_s"]), w_down=dec(q["w_down_q"], q["w_down_s"]))


def popular_experts(expert_offsets, n):
    """The n experts to keep resident, from a run's per-chunk expert offsets [chunks][E+1]: most chunks with rows
    first (each such chunk would stage the expert once), then most rows, then the lower id."""
    import numpy as np
    rows = np.diff(np.asarray(expert_offsets, dtype=np.int64), axis=1)
    order = np.lexsort((np.arange(rows.shape[1]), -rows.sum(0), -(rows > 0).sum(0)))
    return [int(e) for e in order[:n]]


def gate_up_bytes_and_flops(wl, offs_per_chunk, chunk_sizes, wb=2.0, staged_rows=False):
    """Algorithmic DRAM bytes and useful FLOPs of one gate/up launch (per chunk, averaged over the chunks): weights
    of the touched experts (wb bytes per routed weight, WEIGHT_BYTES: codes and scales) + shared expert, the chunk's
    x rows read once, h written once. staged_rows: count the gathered copy of the x rows (one per routed row) that
    the kernel reads instead of x, i.e. the design's bytes rather than the method's minimum."""
    H, I, Is, k = wl.hidden, wl.inter, wl.shared_inter, wl.top_k
    tot_b = tot_f = 0.0
    for offs, n in zip(offs_per_chunk, chunk_sizes):
        counts = offs[1:] - offs[:-1]
        touched = int((counts > 0).sum())
        R = n * k
        rows_read = (R + (n if Is else 0)) if staged_rows else n
        b = touched * 2 * I * H * wb + (2 * Is * H * 2 if Is else 0) + rows_read * H * 2 + (R * I + n * Is) * 2
        f = 2.0 * R * H * 2 * I + 2.0 * n * H * 2 * Is
        tot_b += b
        tot_f += f
    m = len(chunk_sizes)
    return tot_b / m, tot_f / m


def layer_weight_bytes(wl, offs_per_chunk, wb=2.0):
    """Weight bytes one step must stream (the method's bound at this chunk size): per chunk the touched routed
    experts' gate/up and down weights plus the shared expert's, and the router's weights once per chunk."""
    H, I, Is, E = wl.hidden, wl.inter, wl.shared_inter, wl.n_experts
    tot = 0.0
    for offs in offs_per_chunk:
        touched = int(((offs[1:] - offs[:-1]) > 0).sum())
        tot += touched * 3 * I * H * wb + 3 * Is * H * 2 + E * H * 2
    return tot


def tree_fp64_ops(ids_row, n_experts: int) -> int:
    """float64 additions per output column of the tree combine for one token: one per merge of two nodes (the leaf
    products w*y are formed exactly on the integer pipe)."""
    return max(0, len(set(int(v) for v in ids_row)) - 1)


def down_bytes_and_flops(wl, offs_per_chunk, chunk_sizes, wb=2.0):
    H, I, Is, k = wl.hidden, wl.inter, wl.shared_inter, wl.top_k
    tot_b = tot_f = 0.0
    for offs, n in zip(offs_per_chunk, chunk_sizes):
        counts = offs[1:] - offs[:-1]
        touched = int((counts > 0).sum())
        R = n * k
        b = touched * H * I * wb + (H * Is * 2 if Is else 0) + (R * I + n * Is) * 2 + (R + (n if Is else 0)) * H * 4
        f = 2.0 * R * I * H + 2.0 * n * Is * H
        tot_b += b
        tot_f += f
    m = len(chunk_sizes)
    return tot_b / m, tot_f / m


def run_ours(args, dist: Dist):
    import numpy as np
    import torch
    from expert_major_chunked_gb300 import binding, workloads

    assert torch.cuda.is_available(), "the benchmark needs a CUDA device"
    torch.cuda.set_device(dist.local_rank)
    wl = workloads.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_(tokens=args.tokens)
    chunk = args.chunk or wl.chunks[0]
    T = wl.tokens
    inp = workloads.generate(wl)
    wb = WEIGHT_BYTES[args.weights]
    quant = args.weights != "bf16"
    if quant:
        q = quantized_weights(inp, args.weights)
    if wl.offload_slots and quant:
        # code banks in pinned host memory, scales, router and shared expert in device memory
        dev = {k: v.cuda() for k, v in inp.items() if k not in ("x", "w_gu", "w_down")}
        dev.update({"w_gu_q": q["w_gu_q"].pin_memory(), "w_down_q": q["w_down_q"].pin_memory(),
                    "w_gu_s": q["w_gu_s"].cuda(), "w_down_s": q["w_down_s"].cuda()})
        args.single_pass = False
    elif wl.offload_slots:
        # expert banks stay in pinned host memory; router and shared expert in device memory
        dev = {k: (v.pin_memory() if k in ("w_gu", "w_down") else v.cuda()) for k, v in inp.items() if k != "x"}
        args.single_pass = False
    elif quant:
        dev = {k: v.cuda() for k, v in inp.items() if k not in ("x", "w_gu", "w_down")}
        dev.update({k: v.cuda() for k, v in q.items()})
    else:
        dev = {k: v.cuda() for k, v in inp.items() if k != "x"}
    layer = binding.MoePrefill(dev, top_k=wl.top_k, max_chunk=max(chunk, T if args.single_pass else chunk),
                               offload_slots=wl.offload_slots, weight_format=args.weights if quant else None)
    if args.combine == "f64":
        layer.set_combine(binding.COMBINE_F64_TREE)
    if wl.offload_slots:
        layer.set_offload_copy(binding.OFFLOAD_COPY_ROUTED if args.offload_copy == "routed"
                               else binding.OFFLOAD_COPY_ALL)
    stream = torch.cuda.current_stream()
    x = inp["x"].cuda()
    out = torch.empty_like(x)
    n_chunks = (T + chunk - 1) // chunk
    offs = torch.empty((n_chunks, wl.n_experts + 1), dtype=torch.int32, device="cuda")

    prefetch = bool(wl.offload_slots) and args.prefetch

    def step(xd, od, ch=chunk, offs_buf=None):
        layer.run(xd, ch, out=od, expert_offsets=offs_buf)
        if prefetch:  # the same layer stands in for the next one: its first window moves during this run's tail
            layer.prefetch()

    # warm-up (also records the per-chunk expert offsets for the byte/FLOP accounting)
    step(x, out, offs_buf=offs)
    layer.raise_on_device_error()
    for _ in range(max(0, args.warmup - 1)):
        step(x, out)
    layer.raise_on_device_error()
    offs_host = offs.cpu().numpy()
    chunk_sizes = [min(chunk, T - c0) for c0 in range(0, T, chunk)]
    hot = []
    if wl.offload_slots and args.hot_experts > 0:
        hot = popular_experts(offs_host, args.hot_experts)
        layer.set_hot_experts(hot)
        step(x, out)  # stages the set once
        layer.raise_on_device_error()

    # ---------------------------------------------------------------- timed region (device-resident inputs)
    clocks = ClockSampler(gpu_selector(torch, dist.local_rank))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = binding.moe_prefill_launch_count(layer.plan)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0.record(stream)
    for _ in range(args.steps):
        step(x, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks_info = clocks.stop()
    dist.barrier()
    gpu_launches = binding.moe_prefill_launch_count(layer.plan) - launches0
    st = layer.check()
    if st != 0:
        raise binding.MoeError(st, binding.moe_prefill_last_error())
    secs = ev0.elapsed_time(ev1) / 1e3
    secs_max = dist.max(secs)
    value = aggregate_rate([T * args.steps] * dist.world, [secs_max] * dist.world)
    ms_per_step = secs_max / args.steps * 1e3

    # ---------------------------------------------------------------- per-kernel CUDA-event timing
    k_steps = max(3, min(args.steps, 50))
    binding.moe_prefill_set_profiling(layer.plan, True)
    binding.moe_prefill_kernel_times(layer.plan)  # clear
    for _ in range(k_steps):
        step(x, out)
    times = binding.moe_prefill_kernel_times(layer.plan)
    binding.moe_prefill_set_profiling(layer.plan, False)
    peaks = load_peaks()
    gu_ms, gu_n = times["gate_up"]
    dn_ms, dn_n = times["down"]
    # per chunk (offloaded experts run one launch per window of the ring: add up a chunk's launches)
    gu_avg_s = gu_ms / (n_chunks * k_steps if wl.offload_slots else gu_n) / 1e3
    dn_avg_s = dn_ms / (n_chunks * k_steps if wl.offload_slots else dn_n) / 1e3
    gu_bytes, gu_flops = gate_up_bytes_and_flops(wl, offs_host, chunk_sizes, wb)
    gu_staged, _ = gate_up_bytes_and_flops(wl, offs_host, chunk_sizes, wb, staged_rows=True)
    dn_bytes, dn_flops = down_bytes_and_flops(wl, offs_host, chunk_sizes, wb)
    achieved = gu_bytes / gu_avg_s / 1e9
    roofline = {"bound": "hbm", "kernel": "grouped gate/up GEMM + SwiGLU", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": ncu_traffic(wl.name + ("" if args.weights == "bf16" else "_" + args.weights), chunk),
                "algorithmic_bytes_per_launch": gu_bytes, "designed_bytes_per_launch": gu_staged,
                "avg_launch_ms": gu_avg_s * 1e3, "peak_source": peaks["source"] + " (hbm_gbs)"}
    # the GEMMs run for a fraction of a millisecond inside the step: the burst peak applies
    tc_peak = peaks["bf16_tflops"]
    tc_sus = peaks["bf16_tflops_sustained"]
    grouped = {
        "gate_up": {"avg_ms": gu_avg_s * 1e3, "tflops": gu_flops / gu_avg_s / 1e12,
                    "tc_frac_of_burst_bf16": gu_flops / gu_avg_s / 1e12 / tc_peak,
                    "gbs": achieved, "hbm_frac": achieved / peaks["hbm_gbs"]},
        "down": {"avg_ms": dn_avg_s * 1e3, "tflops": dn_flops / dn_avg_s / 1e12,
                 "tc_frac_of_burst_bf16": dn_flops / dn_avg_s / 1e12 / tc_peak,
                 "gbs": dn_bytes / dn_avg_s / 1e9, "hbm_frac": dn_bytes / dn_avg_s / 1e9 / peaks["hbm_gbs"]},
        "per_kernel_ms_per_step": {k: v[0] / k_steps for k, v in times.items()},
        "profiled_steps": k_steps,
    }
    R = T * wl.top_k
    grouped["combine_gbs"] = (R * wl.hidden * 4 + T * wl.hidden * (4 + 2)) / (times["combine"][0] / k_steps / 1e3) / 1e9
    grouped["topk_gbs"] = (T * wl.n_experts * 4 + T * wl.hidden * 2 + T * wl.top_k * 8) / \
        (times["topk"][0] / k_steps / 1e3) / 1e9
    comb_s = times["combine"][0] / max(times["combine"][1], 1) / 1e3
    comb_bytes = (T * wl.top_k * wl.hidden * 4 + T * wl.hidden * (4 + 2)) / n_chunks
    combine = {"mode": "f64-tree" if args.combine == "f64" else "f32-canonical", "avg_launch_ms": comb_s * 1e3,
               "algorithmic_bytes_per_launch": comb_bytes, "gbs": comb_bytes / comb_s / 1e9,
               "hbm_frac": comb_bytes / comb_s / 1e9 / peaks["hbm_gbs"],
               "note": "timed inside the step, on the side stream, overlapping the expert GEMMs"}
    if args.combine == "f64":
        ids_all = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
        layer.run(x, chunk, out=out, topk_id=ids_all)
        ids_np = ids_all.cpu().numpy()
        ops = sum(tree_fp64_ops(r, wl.n_experts) for r in ids_np) + (T if wl.shared_inter else 0)
        ops_per_launch = ops * wl.hidden / n_chunks
        sm_mhz = (clocks_info or {}).get("sm_mhz") or 2070.0
        fp64_peak = torch.cuda.get_device_properties(0).multi_processor_count * 2 * sm_mhz * 1e6 / 1e9
        combine.update({"bound": "alu", "fp64_ops_per_launch": ops_per_launch,
                        "fp64_gops": ops_per_launch / comb_s / 1e9, "fp64_peak_gops": fp64_peak,
                        "fp64_frac": ops_per_launch / comb_s / 1e9 / fp64_peak,
                        "peak_source": "2 float64 operations per SM per clock x SMs x median SM clock of the run"})
    grouped["combine"] = combine

    # ---------------------------------------------------------------- end to end: host buffers through the ABI
    x_host = inp["x"].pin_memory()
    out_host = torch.empty(x_host.shape, dtype=x_host.dtype).pin_memory()
    x_dev = torch.empty_like(x)
    e2e_steps = max(3, min(args.steps, 50))
    out_dev = torch.empty_like(out)

    def host_step():
        # the library copies X rows in and out rows back chunk by chunk, beside the compute
        layer.run_host(x_host, chunk, x_dev, out_dev, out_host)

    for _ in range(2):
        host_step()
    torch.cuda.synchronize()
    dist.barrier()
    ev0.record(stream)
    for _ in range(e2e_steps):
        host_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_secs = dist.max(ev0.elapsed_time(ev1) / 1e3)
    e2e = {"value": T * e2e_steps * dist.world / e2e_secs, "unit": UNIT,
           "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
           "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
           "api": "moe_prefill_run_host: X rows in and out rows back chunk by chunk, overlapped with the compute"}

    # ---------------------------------------------------------------- optional single pass (chunk = T)
    single = None
    if args.single_pass:
        step(x, out, ch=T)
        torch.cuda.synchronize()
        binding.moe_prefill_set_profiling(layer.plan, True)
        binding.moe_prefill_kernel_times(layer.plan)
        sp_steps = 20
        ev0.record(stream)
        for _ in range(sp_steps):
            step(x, out, ch=T)
        ev1.record(stream)
        torch.cuda.synchronize()
        sp_secs = ev0.elapsed_time(ev1) / 1e3
        t2 = binding.moe_prefill_kernel_times(layer.plan)
        binding.moe_prefill_set_profiling(layer.plan, False)
        offs1 = torch.empty((1, wl.n_experts + 1), dtype=torch.int32, device="cuda")
        step(x, out, ch=T, offs_buf=offs1)
        o1 = offs1.cpu().numpy()
        b1, f1 = gate_up_bytes_and_flops(wl, o1, [T], wb)
        b2, f2 = down_bytes_and_flops(wl, o1, [T], wb)
        g_s = t2["gate_up"][0] / t2["gate_up"][1] / 1e3
        d_s = t2["down"][0] / t2["down"][1] / 1e3
        single = {"tokens_per_s": T * sp_steps / sp_secs, "ms_per_step": sp_secs / sp_steps * 1e3,
                  "gate_up": {"avg_ms": g_s * 1e3, "tflops": f1 / g_s / 1e12,
                              "tc_frac_of_burst_bf16": f1 / g_s / 1e12 / tc_peak,
                              "tc_frac_of_sustained_bf16": f1 / g_s / 1e12 / tc_sus,
                              "hbm_frac": b1 / g_s / 1e9 / peaks["hbm_gbs"]},
                  "down": {"avg_ms": d_s * 1e3, "tflops": f2 / d_s / 1e12,
                           "tc_frac_of_burst_bf16": f2 / d_s / 1e12 / tc_peak,
                           "tc_frac_of_sustained_bf16": f2 / d_s / 1e12 / tc_sus,
                           "hbm_frac": b2 / d_s / 1e9 / peaks["hbm_gbs"]},
                  "grouped_tc_frac_of_burst_bf16": (f1 + f2) / (g_s + d_s) / 1e12 / tc_peak,
                  "tc_peak_tflops": tc_peak, "tc_peak_source": peaks["source"] + " (bf16_tflops, burst)",
                  "note": "chunk = T: about T*k/E rows per expert, where the grouped GEMMs are tensor-bound"}
        layer.raise_on_device_error()

    # ---------------------------------------------------------------- decode sizes (1 and 8 tokens, same kernels)
    decode = None
    if not args.no_decode and not wl.offload_slots:
        decode = {}
        for n_dec in (1, 8):
            xd = x[:n_dec].contiguous()
            od = torch.empty_like(xd)
            offs_d = torch.empty((1, wl.n_experts + 1), dtype=torch.int32, device="cuda")
            layer.run(xd, n_dec, out=od, expert_offsets=offs_d)
            for _ in range(5):
                layer.run(xd, n_dec, out=od)
            torch.cuda.synchronize()
            reps = 200
            ev0.record(stream)
            for _ in range(reps):
                layer.run(xd, n_dec, out=od)
            ev1.record(stream)
            torch.cuda.synchronize()
            dsec = ev0.elapsed_time(ev1) / 1e3 / reps
            o = offs_d.cpu().numpy()[0]
            touched = int(((o[1:] - o[:-1]) > 0).sum())
            wbytes = touched * 3 * wl.inter * wl.hidden * wb + wl.n_experts * wl.hidden * 2 + \
                3 * wl.shared_inter * wl.hidden * 2
            decode[f"tokens_{n_dec}"] = {"ms_per_call": dsec * 1e3, "tokens_per_s": n_dec / dsec,
                                         "weight_bytes": wbytes, "gbs": wbytes / dsec / 1e9,
                                         "hbm_frac": wbytes / dsec / 1e9 / peaks["hbm_gbs"]}
        layer.raise_on_device_error()

    route_stats = layer.stats()
    offload = None
    if wl.offload_slots:
        # bytes over the host link per step, against a plain pinned copy: the routed experts of every chunk
        # (routed staging, counted on the device), else every expert of every chunk (copy engines)
        code_bytes = {"bf16": 2.0, "mxfp8": 1.0, "nvfp4": 0.5}[args.weights]  # the banks hold codes only
        bank = int((inp["w_gu"].numel() + inp["w_down"].numel()) * code_bytes)
        per_expert = bank // wl.n_experts
        if args.offload_copy == "routed":
            h2d_bytes = route_stats["experts_copied"] * per_expert
        else:
            h2d_bytes = bank * n_chunks
        probe = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        dprobe = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
        for _ in range(2):
            dprobe.copy_(probe, non_blocking=True)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(5):
            dprobe.copy_(probe, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        link_gbs = 5 * (1 << 30) / (ev0.elapsed_time(ev1) / 1e3) / 1e9
        achieved_link = h2d_bytes / (ms_per_step / 1e3) / 1e9
        offload = {"slots": wl.offload_slots, "copy": args.offload_copy, "h2d_bytes_per_step": h2d_bytes,
                   "experts_copied": route_stats["experts_copied"], "experts_skipped": route_stats["experts_skipped"],
                   "hot_experts": len(hot), "experts_hot": route_stats.get("experts_hot", 0),
                   "prefetch": prefetch,
                   "hot_set_bytes_once": len(hot) * per_expert,
                   "h2d_gbs": achieved_link,
                   "pinned_copy_gbs": link_gbs, "link_frac": achieved_link / link_gbs}
        kname = ("routed-expert staging kernel (reads the pinned banks)" if args.offload_copy == "routed"
                 else "expert staging copies (copy engines)")
        roofline = {"bound": "h2d", "kernel": kname, "achieved": achieved_link,
                    "peak": link_gbs, "unit": "GB/s", "frac": achieved_link / link_gbs, "traffic": None,
                    "peak_source": "measured in this run: pinned host->device cudaMemcpyAsync of 1 GiB"}
        del probe, dprobe

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu_inp = inp
        if quant:  # the oracle runs on the decoded weights
            cpu_inp = decoded_weights(inp, q, args.weights)
        cpu = cpu_baseline(cpu_inp, wl)

    if dist.rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(wl, chunk, dist.world),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
                "clocks": clocks_info, "grouped_gemm": grouped,
                "routing_last_run": route_stats}
        line["config"]["combine"] = "f64-tree" if args.combine == "f64" else "f32-canonical"
        line["config"]["weights"] = WEIGHT_DESC[args.weights]
        if wl.offload_slots:
            line["config"]["offload_copy"] = args.offload_copy
        wbytes = layer_weight_bytes(wl, offs_host, wb)
        line["layer_hbm_frac"] = {"weight_bytes_per_step": wbytes, "gbs": wbytes / (ms_per_step / 1e3) / 1e9,
                                  "frac": wbytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "note": "weight bytes the step must stream / ms_per_step / hbm_gbs"}
        if single is not None:
            line["single_pass"] = single
        if decode is not None:
            line["decode"] = decode
        if offload is not None:
            line["offload"] = offload
        print(json.dumps(line), flush=True)
    del layer
    dist.close()


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_ours(args, dist)


if __name__ == "__main__":
    main()
