"""Cross-layer prefetch of offloaded experts on the GPU.

Umbrella PR #1113 ("Latest measured follow-up") counts cross-layer prefetch among the expert copies: while one
layer computes, the next layer's first experts move. moe_prefill_prefetch stages the first window of a plan's next
run ahead of it; the run then skips that window's staging. Only where the weights come from changes, so two
offloaded layers run back to back with prefetches must equal their resident runs byte for byte, in both staging
modes, with a hot set, and when the prefetch is dropped (another workspace, a new hot set).
"""

import numpy as np
import pytest
import torch

from layer_helpers import out_bits

pytestmark = pytest.mark.gpu


def _weights(seed, E=64, H=256, I=128, Is=128):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I), "ws_gu": r(2 * Is, H),
            "ws_down": r(H, Is)}


def _pair(w, k, max_chunk, slots):
    from expert_major_chunked_gb300 import binding
    dev = {n: t.cuda() for n, t in w.items()}
    resident = binding.MoePrefill(dev, top_k=k, max_chunk=max_chunk)
    host = {n: (w[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in w}
    return resident, binding.MoePrefill(host, top_k=k, max_chunk=max_chunk, offload_slots=slots)


def _chain(layers, x, chunk, prefetch, copy_stream=None):
    """Layer i's output feeds layer i+1; with prefetch, each layer's first window is staged while the one before
    runs (and layer 0's while the last one runs, for the next pass)."""
    h = x
    for i, layer in enumerate(layers):
        h = layer.run(h, chunk)
        if prefetch:
            layers[(i + 1) % len(layers)].prefetch(copy_stream)
    for layer in layers:
        layer.raise_on_device_error()
    return h.cpu()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("slots", [2, 16])
def test_two_layers_with_prefetch_equal_resident(mode, slots):
    k, T, chunk = 4, 300, 64
    gen = torch.Generator().manual_seed(21)
    x = (torch.randn(T, 256, generator=gen)).to(torch.bfloat16).cuda()
    r0, o0 = _pair(_weights(22), k, chunk, slots)
    r1, o1 = _pair(_weights(23), k, chunk, slots)
    for o in (o0, o1):
        o.set_offload_copy(mode)
    ref = _chain([r0, r1], x, chunk, prefetch=False)
    cs = torch.cuda.Stream()
    for _ in range(3):
        np.testing.assert_array_equal(out_bits(_chain([o0, o1], x, chunk, prefetch=True)), out_bits(ref))
        np.testing.assert_array_equal(out_bits(_chain([o0, o1], x, chunk, prefetch=True, copy_stream=cs)),
                                      out_bits(ref))


def test_prefetch_with_hot_set_and_dropped_prefetches():
    k, T, chunk = 4, 257, 64
    gen = torch.Generator().manual_seed(24)
    x = (torch.randn(T, 256, generator=gen)).to(torch.bfloat16).cuda()
    res, off = _pair(_weights(25), k, chunk, 8)
    ref = res.run(x, chunk).cpu()
    off.set_hot_experts([0, 2, 9, 33])              # hot experts inside and outside the first window
    off.prefetch()
    np.testing.assert_array_equal(out_bits(off.run(x, chunk).cpu()), out_bits(ref))
    off.prefetch()
    off.set_hot_experts([1, 5])                     # drops the prefetch (the ring's layout changes)
    np.testing.assert_array_equal(out_bits(off.run(x, chunk).cpu()), out_bits(ref))
    off.prefetch()
    off.workspace = torch.empty_like(off.workspace)  # the run uses another workspace: prefetch not consumed
    np.testing.assert_array_equal(out_bits(off.run(x, chunk).cpu()), out_bits(ref))
    off.prefetch()
    off.prefetch()                                  # twice: still one consistent window
    np.testing.assert_array_equal(out_bits(off.run(x, chunk).cpu()), out_bits(ref))
    off.raise_on_device_error()


def test_prefetch_rejections():
    from expert_major_chunked_gb300 import binding
    res, off = _pair(_weights(26), 4, 64, 8)
    with pytest.raises(binding.MoeError):
        res.prefetch()                              # no offloaded experts
    too_small = binding.lib().moe_prefill_prefetch(off.plan, off.workspace.data_ptr(), 16, None)
    assert too_small == -3  # MOE_ERR_WORKSPACE
    misaligned = binding.lib().moe_prefill_prefetch(off.plan, off.workspace.data_ptr() + 16, off.workspace_bytes, None)
    assert misaligned == -1
