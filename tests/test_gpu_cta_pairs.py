"""The expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2, weights as the 256-row operand, an expert's member rows
in steps of 32) against the single-CTA kernel (member rows as the 128-row operand), on the GPU.

Both accumulate every output element over K in the same order (64-wide stages, 16 per instruction), so the layer's
output must be the same bytes whichever kernel runs each projection (gate/up, down, both, neither), at every chunk
size, with or without the shared expert, resident or offloaded; and within the layer's bound of the float64 oracle.
The shapes give experts with one short token tile, with several tiles of up to 256 rows and a ragged last one, and
empty experts.
"""

import numpy as np
import pytest
import torch

from layer_helpers import MAX_ABS, REL_L2, GpuLayer, compare_out, out_bits

pytestmark = pytest.mark.gpu

MASKS = (0, 1, 2, 3)  # bit 0: gate/up on pairs, bit 1: down on pairs


def _inputs(seed, T, H, E, I, Is, router_std=0.3):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    d = {"x": r(T, H, std=1.0), "w_router": r(E, H, std=router_std), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I)}
    if Is > 0:
        d["ws_gu"] = r(2 * Is, H)
        d["ws_down"] = r(H, Is)
    return d


SHAPES = {
    # T, H, E, I, Is, k
    "small_shared": (300, 256, 64, 128, 128, 4),
    "no_shared": (517, 512, 32, 256, 0, 3),
    "long_tiles": (1000, 512, 16, 384, 256, 8),   # ~500 rows per expert: two token tiles each
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_pairs_equal_single_cta_every_chunk(name, oracle_lib):
    from expert_major_chunked_gb300 import binding
    T, H, E, I, Is, k = SHAPES[name]
    inp = _inputs(3, T, H, E, I, Is)
    g = GpuLayer(inp, k, max_chunk=T)
    assert g.layer.cta_pairs == binding.PAIRS_GATE_UP, "the default for these dimensions"
    first = None
    for chunk in (1, 37, 128, T):
        outs = {}
        for mask in MASKS:
            g.layer.cta_pairs = mask
            outs[mask] = g.run(chunk)
        for mask in MASKS[1:]:
            np.testing.assert_array_equal(out_bits(outs[mask]["out"]), out_bits(outs[0]["out"]),
                                          err_msg=f"chunk {chunk} mask {mask}")
            np.testing.assert_array_equal(outs[mask]["row_token"], outs[0]["row_token"])
        if first is None:
            first = out_bits(outs[0]["out"])
        else:  # rows do not depend on the chunk size
            np.testing.assert_array_equal(out_bits(outs[0]["out"]), first, err_msg=f"chunk {chunk}")
    g.layer.cta_pairs = binding.PAIRS_GATE_UP | binding.PAIRS_DOWN
    _, ref_bf, _, _ = oracle_lib.moe_forward(inp, k)
    max_abs, rel = compare_out(g.run(T)["out"], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)


def test_pairs_skewed_routing():
    # a router that sends most tokens to a few experts: tiles of 256 rows, several per expert, many empty experts
    T, H, E, I, Is, k = 2000, 256, 64, 128, 128, 2
    inp = _inputs(5, T, H, E, I, Is, router_std=0.05)
    # positive activations; experts 0..2 favoured by every token, experts 48.. disfavoured by every token
    inp["x"] = (inp["x"].float().abs() + 0.5).to(torch.bfloat16)
    inp["w_router"][:3] += torch.tensor(0.05, dtype=torch.bfloat16)
    inp["w_router"][48:] = -inp["w_router"][48:].float().abs().to(torch.bfloat16) - 0.05
    g = GpuLayer(inp, k, max_chunk=T)
    res = {}
    for mask in MASKS:
        g.layer.cta_pairs = mask
        res[mask] = g.run(T)
    counts = np.diff(res[0]["offs"][0])
    assert counts.max() > 512 and (counts == 0).any(), counts
    for mask in MASKS[1:]:
        np.testing.assert_array_equal(out_bits(res[mask]["out"]), out_bits(res[0]["out"]), err_msg=f"mask {mask}")


def test_pairs_offloaded_equal_resident_single():
    from expert_major_chunked_gb300 import binding
    T, H, E, I, Is, k, chunk = 300, 256, 64, 128, 128, 4, 64
    inp = _inputs(7, T, H, E, I, Is)
    names = ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")
    dev = {n: inp[n].cuda() for n in names}
    resident = binding.MoePrefill(dev, top_k=k, max_chunk=chunk)
    resident.cta_pairs = 0
    host = {n: (inp[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in names}
    offload = binding.MoePrefill(host, top_k=k, max_chunk=chunk, offload_slots=8)
    offload.set_hot_experts([3, 9, 60])
    x = inp["x"].cuda()
    a = resident.run(x, chunk).cpu()
    resident.raise_on_device_error()
    for mask in (binding.PAIRS_GATE_UP, binding.PAIRS_GATE_UP | binding.PAIRS_DOWN):
        offload.cta_pairs = mask
        b = offload.run(x, chunk).cpu()
        offload.raise_on_device_error()
        np.testing.assert_array_equal(out_bits(a), out_bits(b), err_msg=f"mask {mask}")


def test_pairs_refused_where_dimensions_do_not_allow():
    from expert_major_chunked_gb300 import binding
    inp = _inputs(1, 64, 256, 16, 64, 0)  # inter = 64: not a multiple of 128
    g = GpuLayer(inp, 2, max_chunk=64)
    assert g.layer.cta_pairs == 0
    with pytest.raises(binding.MoeError):
        g.layer.cta_pairs = binding.PAIRS_GATE_UP
    with pytest.raises(binding.MoeError):
        g.layer.cta_pairs = 4
    g.layer.cta_pairs = 0


@pytest.mark.parametrize("name,tokens,chunks", [("e512_t16022", 4096, (2048, 4096)),
                                                ("e128_t3001", 3001, (256, 3001))])
def test_pairs_equal_single_cta_on_workload_shapes(name, tokens, chunks):
    """The two GEMM kernels on the workloads' own dimensions (H = 2048; E = 512, I = 512, k = 10 or E = 128,
    I = 768, I_s = 2048, k = 8), at a chunk size the workload uses and in one pass: the same output bytes for every
    choice of kernel per projection."""
    from layer_helpers import cpu_inputs
    wl, inp = cpu_inputs(name, tokens=tokens)
    g = GpuLayer(inp, wl.top_k, max_chunk=max(chunks))
    for chunk in chunks:
        outs = {}
        for mask in MASKS:
            g.layer.cta_pairs = mask
            outs[mask] = out_bits(g.run(chunk)["out"])
        for mask in MASKS[1:]:
            np.testing.assert_array_equal(outs[mask], outs[0], err_msg=f"{name} chunk {chunk} mask {mask}")
