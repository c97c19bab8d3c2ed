"""Helpers shared by the GPU layer tests: input caches, one call of the layer through the C ABI, and the
comparison against the float64 oracle."""

from __future__ import annotations

import functools
import math

import numpy as np
import torch

from expert_major_chunked_gb300 import workloads

# Output tolerances against the oracle's BF16 output (the layer's acceptance bound).
MAX_ABS = 2e-2
REL_L2 = 1e-3


@functools.lru_cache(maxsize=4)
def cpu_inputs(name: str, tokens: int | None = None, seed: int | None = None):
    wl = workloads.WORKLOADS[name]
    return wl, workloads.generate(wl, tokens=tokens, seed=seed)


class GpuLayer:
    """Weights on the device plus a plan sized for max_chunk."""

    def __init__(self, inputs: dict, top_k: int, max_chunk: int):
        from expert_major_chunked_gb300 import binding
        self.dev = {k: v.cuda() for k, v in inputs.items()}
        w = {k: self.dev[k] for k in ("w_router", "w_gu", "w_down", "ws_gu", "ws_down") if k in self.dev}
        self.layer = binding.MoePrefill(w, top_k=top_k, max_chunk=max_chunk)
        self.k = top_k
        self.E = inputs["w_router"].shape[0]
        self.H = inputs["w_router"].shape[1]

    def run(self, chunk: int, x=None):
        x = self.dev["x"] if x is None else x
        T = x.shape[0]
        n_chunks = (T + chunk - 1) // chunk
        out = torch.empty_like(x)
        ids = torch.full((T, self.k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, self.k), float("nan"), dtype=torch.float32, device="cuda")
        offs = torch.full((n_chunks, self.E + 1), -1, dtype=torch.int32, device="cuda")
        row_token = torch.full((T * self.k,), -1, dtype=torch.int32, device="cuda")
        self.layer.run(x, chunk, out=out, topk_id=ids, topk_w=w, expert_offsets=offs, row_token=row_token)
        self.layer.raise_on_device_error()
        return {"out": out.cpu(), "ids": ids.cpu().numpy(), "w": w.cpu().numpy(), "offs": offs.cpu().numpy(),
                "row_token": row_token.cpu().numpy()}


def out_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def compare_out(got_bf16: torch.Tensor, ref_bits: np.ndarray, oracle_lib):
    """Returns (max_abs, rel_l2) of the GPU BF16 output against the oracle's BF16 output."""
    g = got_bf16.to(torch.float64).numpy()
    r = oracle_lib.bf16_to_double(ref_bits)
    diff = g - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def tau_bound(x_bf16: torch.Tensor, w_router_bf16: torch.Tensor) -> np.ndarray:
    """Per-token bound on |fp32 tensor-core logit - float64 logit| used by the routing kernel."""
    H = x_bf16.shape[1]
    xn = np.linalg.norm(x_bf16.double().numpy(), axis=1)
    wn = np.linalg.norm(w_router_bf16.double().numpy(), axis=1).max()
    return (H // 16 + 1) * 2.0 ** -23 * xn * wn


def sample_tokens(T: int, chunks, extra: int, seed: int = 0):
    """Tokens at every chunk boundary (first/last of each chunk) for every chunk size, plus random ones."""
    s = {0, T - 1}
    for c in chunks:
        for c0 in range(0, T, c):
            s.add(c0)
            s.add(min(c0 + c, T) - 1)
    rng = np.random.default_rng(seed)
    s.update(rng.choice(T, size=min(extra, T), replace=False).tolist())
    return np.array(sorted(s), dtype=np.int64)


def check_routing(res, ref_ids, ref_w, x_bf16, wr_bf16, E, chunk, oracle_lib):
    """Top-k ids, expert offsets and row->token map bit-exact; weights within the logit error bound."""
    np.testing.assert_array_equal(res["ids"], ref_ids)
    offs, row_token, _ = oracle_lib.permutation(ref_ids, E, chunk)
    np.testing.assert_array_equal(res["offs"], offs)
    np.testing.assert_array_equal(res["row_token"], row_token)
    tau = tau_bound(x_bf16, wr_bf16)
    bound = ref_w * (2 * tau[:, None]) + 2e-6
    werr = np.abs(res["w"].astype(np.float64) - ref_w)
    assert np.all(werr <= bound), float(np.max(werr - bound))
