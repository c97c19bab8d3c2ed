"""Seeded synthetic inputs for the MoE prefill layer.

This module only draws numbers. It holds none of the layer's arithmetic (no router, no top-k, no SwiGLU, no
combine), so both the CUDA path and the float64 oracle can take their inputs from it without sharing any part of
the method.

The pages this layer comes from ("EXL3 Flash Next: deep prefill" and "exact deep prefill") measure whole-model
serving on a private checkpoint and private prompts. Those are not available, so every input here is synthetic:
prompt lengths follow the pages' prompts (40-token "short" prompt, the 3001/12001-token prompt-time cells, the
4099-token chunk-equality gate and the 16,022-token "zig" prompt), and the weights are Gaussian draws in BF16.

Draw recipe (one torch CPU generator per workload, seeded once, draws taken in this order):
X, W_router, W_gu (expert by expert), W_down (expert by expert), W_shared_gu, W_shared_down. Every draw is
float32 and then rounded to bfloat16 (round to nearest, ties to even); both sides of a comparison receive the same
BF16 bytes.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class Workload:
    """Sizes and draw parameters of one synthetic MoE layer workload."""

    name: str
    tokens: int            # T
    hidden: int            # H
    n_experts: int         # E (routed)
    inter: int             # I (routed expert intermediate size)
    top_k: int             # k
    shared_inter: int      # I_s (0 = no shared expert)
    chunks: tuple = ()     # chunk sizes the workload is run at (besides the single pass)
    x_std: float = 1.0
    w_std: float = 0.02
    router_std: float = 0.02
    zipf_prior: float = 0.0     # >0: channel 0 of X is 1.0 and W_router[:, 0] holds log-popularity
    offload_slots: int = 0
    seed: int = 0
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the layer (prompt lengths from the pages; dims from the layer family studied there).
WORKLOADS: Dict[str, Workload] = {
    # Tiny layer: activations and weights N(0, 0.02^2); router scaled so that logits are N(0, 1).
    "tiny": Workload("tiny", tokens=40, hidden=256, n_experts=16, inter=128, top_k=2, shared_inter=128,
                     chunks=(8, 16, 40), x_std=0.02, w_std=0.02, router_std=1.0 / (0.02 * math.sqrt(256)),
                     note="40-token short prompt; fp32 draws rounded to bf16"),
    # 3001-token prompt-time cell: 128 experts, inter 768, top-8, shared inter 2048.
    "e128_t3001": Workload("e128_t3001", tokens=3001, hidden=2048, n_experts=128, inter=768, top_k=8,
                           shared_inter=2048, chunks=(256, 1024, 2048), x_std=1.0, w_std=0.02, router_std=0.02,
                           note="3001-token prompt; router N(0, 0.02^2)"),
    # 4099-token chunk-equality prompt with a Zipf(1.1) expert-popularity prior in the router.
    "e512_zipf_t4099": Workload("e512_zipf_t4099", tokens=4099, hidden=2048, n_experts=512, inter=512, top_k=10,
                                shared_inter=512, chunks=(256, 1024, 2048), x_std=1.0, w_std=0.02,
                                router_std=1.0 / math.sqrt(2047), zipf_prior=1.1,
                                note="4099-token prompt; Zipf(1.1) popularity prior on channel 0"),
    # 16,022-token long prompt, uniform router (logits N(0, 1)), chunk 2048.
    "e512_t16022": Workload("e512_t16022", tokens=16022, hidden=2048, n_experts=512, inter=512, top_k=10,
                            shared_inter=512, chunks=(2048,), x_std=1.0, w_std=0.02,
                            router_std=1.0 / math.sqrt(2048),
                            note="16,022-token long prompt; logits N(0, 1)"),
    # Offloaded experts: 12,001 tokens, chunk 1024, expert weights in pinned host memory, 32-slot ring.
    "e512_offload_t12001": Workload("e512_offload_t12001", tokens=12001, hidden=2048, n_experts=512, inter=512,
                                    top_k=10, shared_inter=512, chunks=(1024,), x_std=1.0, w_std=0.02,
                                    router_std=1.0 / math.sqrt(2048), offload_slots=32,
                                    note="12,001-token prompt; experts staged from pinned host memory"),
    # The same offloaded layer under the Zipf(1.1) popularity prior: skewed routing leaves experts of a chunk
    # without rows, which the routed staging mode does not copy.
    "e512_zipf_offload_t12001": Workload("e512_zipf_offload_t12001", tokens=12001, hidden=2048, n_experts=512,
                                         inter=512, top_k=10, shared_inter=512, chunks=(1024,), x_std=1.0,
                                         w_std=0.02, router_std=1.0 / math.sqrt(2047), zipf_prior=1.1,
                                         offload_slots=32,
                                         note="12,001-token prompt, Zipf(1.1) prior; experts staged from pinned host"
                                              " memory"),
}


def _randn_bf16(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def zipf_log_popularity(n_experts: int, s: float) -> torch.Tensor:
    """log p_r for ranks r = 1..E of a Zipf(s) popularity law, p_r = r^-s / sum_j j^-s (float64)."""
    ranks = torch.arange(1, n_experts + 1, dtype=torch.float64)
    w = ranks.pow(-s)
    return torch.log(w / w.sum())


def generate(wl: Workload, tokens: Optional[int] = None, seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw the inputs of a workload as BF16 CPU tensors.

    Returns a dict with x [T][H], w_router [E][H], w_gu [E][2I][H] (rows 0..I-1 gate, I..2I-1 up),
    w_down [E][H][I], and (when shared_inter > 0) ws_gu [2I_s][H], ws_down [H][I_s].
    """
    T = wl.tokens if tokens is None else tokens
    H, E, I, Is = wl.hidden, wl.n_experts, wl.inter, wl.shared_inter
    gen = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    out: Dict[str, torch.Tensor] = {}
    x = torch.randn((T, H), generator=gen, dtype=torch.float32) * wl.x_std
    if wl.zipf_prior > 0:
        x[:, 0] = 1.0
    out["x"] = x.to(torch.bfloat16)
    del x
    wr = torch.randn((E, H), generator=gen, dtype=torch.float32) * wl.router_std
    if wl.zipf_prior > 0:
        perm = torch.randperm(E, generator=gen)
        logp = zipf_log_popularity(E, wl.zipf_prior)
        wr[:, 0] = logp[perm].to(torch.float32)
    out["w_router"] = wr.to(torch.bfloat16)
    del wr
    w_gu = torch.empty((E, 2 * I, H), dtype=torch.bfloat16)
    for e in range(E):
        w_gu[e] = _randn_bf16(gen, (2 * I, H), wl.w_std)
    out["w_gu"] = w_gu
    w_down = torch.empty((E, H, I), dtype=torch.bfloat16)
    for e in range(E):
        w_down[e] = _randn_bf16(gen, (H, I), wl.w_std)
    out["w_down"] = w_down
    if Is > 0:
        out["ws_gu"] = _randn_bf16(gen, (2 * Is, H), wl.w_std)
        out["ws_down"] = _randn_bf16(gen, (H, Is), wl.w_std)
    return out


def draw_x(wl: Workload, tokens: int, seed: int) -> torch.Tensor:
    """A fresh activation matrix [tokens][H] (BF16) with the workload's distribution, from its own seed."""
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn((tokens, wl.hidden), generator=gen, dtype=torch.float32) * wl.x_std
    if wl.zipf_prior > 0:
        x[:, 0] = 1.0
    return x.to(torch.bfloat16)


def quantize_mxfp8(w: torch.Tensor):
    """Block-scaled FP8 (MXFP8) form of expert weights [E][R][K], K a multiple of 32: E4M3 codes [E][R][K] (uint8)
    and E8M0 scales [E][K/32][R] (uint8, one plane per 32-wide K block).

    This is an input format, not part of the layer: each block of 32 weights along K shares the power of two
    2^(s-127) (OCP Microscaling v1.0 E8M0) with s - 127 the least exponent that keeps max |w| / 2^(s-127) <= 448,
    the largest E4M3 value (so no weight is clipped), kept in [10, 246] so that every code times its scale is
    exactly a normal bf16 value; the weights divided by the scale are rounded to E4M3 (nearest, ties to even).
    """
    E, R, K = w.shape
    assert K % 32 == 0
    codes = torch.empty((E, R, K), dtype=torch.uint8)
    scales = torch.empty((E, K // 32, R), dtype=torch.uint8)
    for e in range(E):
        blk = w[e].to(torch.float32).reshape(R, K // 32, 32)
        amax = blk.abs().amax(dim=2)
        expo = torch.where(amax > 0, torch.ceil(torch.log2(amax.clamp_min(1e-38).double() / 448.0)).float(),
                           torch.zeros_like(amax))
        s = (expo + 127).clamp(10, 246)
        q = (blk / torch.exp2(s - 127).unsqueeze(2)).clamp(-448.0, 448.0)
        codes[e] = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, K)
        scales[e] = s.to(torch.uint8).t()
    return codes, scales


def mxfp8_weights(inp: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """The routed expert weights of a drawn workload in MXFP8 form: w_gu_q/w_gu_s, w_down_q/w_down_s."""
    gu_q, gu_s = quantize_mxfp8(inp["w_gu"])
    dn_q, dn_s = quantize_mxfp8(inp["w_down"])
    return {"w_gu_q": gu_q, "w_gu_s": gu_s, "w_down_q": dn_q, "w_down_s": dn_s}


_E2M1_GRID = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float32)


def quantize_nvfp4(w: torch.Tensor):
    """Block-scaled FP4 (NVFP4) form of expert weights [E][R][K], K a multiple of 16: E2M1 codes [E][R][K/2] (uint8,
    element 2j in the low nibble of byte j) and E4M3 scales [E][K/16][R] (uint8, one plane per 16-wide K block).

    An input format, not part of the layer: each block of 16 weights along K gets the least E4M3 scale that is at
    least max |w| / 6 (6 = the largest E2M1 value, so nothing is clipped), and every weight divided by its scale is
    rounded to the nearest E2M1 value, ties to the even code. No tensor-wide scale.
    """
    E, R, K = w.shape
    assert K % 16 == 0
    codes = torch.empty((E, R, K // 2), dtype=torch.uint8)
    scales = torch.empty((E, K // 16, R), dtype=torch.uint8)
    grid = _E2M1_GRID
    for e in range(E):
        blk = w[e].to(torch.float32).reshape(R, K // 16, 16)
        need = blk.abs().amax(dim=2) / 6.0
        s8 = need.to(torch.float8_e4m3fn)
        s = s8.to(torch.float32)
        bump = s < need  # round the scale up to the next E4M3 value
        s8 = torch.where(bump, (s8.view(torch.uint8) + 1).view(torch.float8_e4m3fn), s8)
        s = s8.to(torch.float32)
        s = torch.where(s > 0, s, torch.ones_like(s))  # an all-zero block: any scale
        s8 = s.to(torch.float8_e4m3fn)
        q = (blk / s.unsqueeze(2)).clamp(-6.0, 6.0)
        mag = q.abs()
        d = (mag.unsqueeze(-1) - grid).abs()  # distance to each grid value
        best = d.argmin(dim=-1)
        # ties between two grid neighbours go to the even code (fraction bit 0): argmin keeps the lower index,
        # which is the even one for the ties 0.25, 1.25, 2.5, 5; for 0.75, 1.75, 3.5 the even code is the upper
        tie_up = torch.zeros_like(mag, dtype=torch.bool)
        for t in (0.75, 1.75, 3.5):
            tie_up |= mag == t
        best = torch.where(tie_up, best + 1, best)
        nib = best.to(torch.uint8) | ((q < 0).to(torch.uint8) << 3)
        nib = nib.reshape(R, K)
        codes[e] = nib[:, 0::2] | (nib[:, 1::2] << 4)
        scales[e] = s8.view(torch.uint8).t()
    return codes, scales


def nvfp4_weights(inp: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """The routed expert weights of a drawn workload in NVFP4 form: w_gu_q/w_gu_s, w_down_q/w_down_s."""
    gu_q, gu_s = quantize_nvfp4(inp["w_gu"])
    dn_q, dn_s = quantize_nvfp4(inp["w_down"])
    return {"w_gu_q": gu_q, "w_gu_s": gu_s, "w_down_q": dn_q, "w_down_s": dn_s}
