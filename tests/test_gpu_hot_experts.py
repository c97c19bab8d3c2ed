"""A resident hot set of offloaded experts on the GPU.

Umbrella PR #1113 keeps per-expert use counts as placement priors ("Persistent expert-profile checkpoint") and
accounts the copied bytes by category ("Latest measured follow-up"). Here the caller names experts to keep in HBM
slots after the ring; they are staged once per workspace and the per-chunk staging skips them. The set changes only
where their weights are read from, so every run must equal the resident-weight run byte for byte, and the staging
counts must split the routed (chunk, expert) pairs exactly into copied and hot ones.
"""

import numpy as np
import pytest
import torch

from layer_helpers import cpu_inputs, out_bits

pytestmark = pytest.mark.gpu


def _small(seed, T=300, H=256, E=64, I=128, Is=128):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"x": r(T, H, std=1.0), "w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I),
            "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


def _pair(inp, k, max_chunk, slots):
    from expert_major_chunked_gb300 import binding
    names = ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")
    dev = {n: inp[n].cuda() for n in names}
    resident = binding.MoePrefill(dev, top_k=k, max_chunk=max_chunk)
    host = {n: (inp[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in names}
    offload = binding.MoePrefill(host, top_k=k, max_chunk=max_chunk, offload_slots=slots)
    return resident, offload


def _run(layer, x, chunk, k, offs=None):
    out = layer.run(x, chunk, expert_offsets=offs)
    layer.raise_on_device_error()
    return out.cpu()


def _counts(offs):
    return np.diff(offs.cpu().numpy(), axis=1)  # [chunks][E] rows per (chunk, expert)


@pytest.mark.parametrize("slots", [2, 8])
@pytest.mark.parametrize("hot", [[5], [0, 1, 2, 3], [63, 7, 30, 12, 44, 1, 9, 20, 33, 50], list(range(64))])
def test_hot_set_equals_resident_and_counts(slots, hot):
    from expert_major_chunked_gb300 import binding
    k, E, T, chunk = 4, 64, 300, 64
    inp = _small(11)
    x = inp["x"].cuda()
    resident, offload = _pair(inp, k, chunk, slots)
    a = _run(resident, x, chunk, k)
    offload.set_hot_experts(hot)
    n_chunks = (T + chunk - 1) // chunk
    offs = torch.empty((n_chunks, E + 1), dtype=torch.int32, device="cuda")
    for mode in (binding.OFFLOAD_COPY_ROUTED, binding.OFFLOAD_COPY_ALL, binding.OFFLOAD_COPY_ROUTED):
        offload.set_offload_copy(mode)
        b = _run(offload, x, chunk, k, offs)
        np.testing.assert_array_equal(out_bits(b), out_bits(a))
    st = offload.stats()  # of the last (routed) run
    routed = _counts(offs) > 0
    is_hot = np.zeros(E, dtype=bool)
    is_hot[hot] = True
    assert st["experts_hot"] == int(routed[:, is_hot].sum())
    assert st["experts_copied"] == int(routed[:, ~is_hot].sum())
    assert st["experts_copied"] + st["experts_skipped"] + st["experts_hot"] == n_chunks * E


def test_hot_set_changes_and_new_workspace():
    """A set replaced by another, removed, and a run on a fresh workspace (the set is staged again)."""
    k, T, chunk = 4, 257, 64
    inp = _small(12, T=T)
    x = inp["x"].cuda()
    resident, offload = _pair(inp, k, chunk, 8)
    a = _run(resident, x, chunk, k)
    base_ws = offload.workspace_bytes
    for hot in ([3, 4], [10, 20, 30, 40, 50, 60], [], [0]):
        offload.set_hot_experts(hot)
        assert offload.workspace_bytes >= base_ws
        for _ in range(2):
            np.testing.assert_array_equal(out_bits(_run(offload, x, chunk, k)), out_bits(a))
    offload.workspace = torch.empty_like(offload.workspace)  # another workspace: maps and hot slots rebuilt
    np.testing.assert_array_equal(out_bits(_run(offload, x, chunk, k)), out_bits(a))


def test_hot_set_with_mxfp8_codes():
    from expert_major_chunked_gb300 import binding, workloads
    k, chunk = 4, 64
    inp = _small(13)
    q = workloads.mxfp8_weights(inp)
    common = {n: inp[n].cuda() for n in ("w_router", "ws_gu", "ws_down")}
    x = inp["x"].cuda()
    resident = binding.MoePrefill(dict(common, **{n: t.cuda() for n, t in q.items()}), top_k=k, max_chunk=chunk)
    host = dict(common, w_gu_q=q["w_gu_q"].pin_memory(), w_down_q=q["w_down_q"].pin_memory(),
                w_gu_s=q["w_gu_s"].cuda(), w_down_s=q["w_down_s"].cuda())
    offload = binding.MoePrefill(host, top_k=k, max_chunk=chunk, offload_slots=8)
    offload.set_hot_experts([1, 2, 3, 40, 41])
    a = _run(resident, x, chunk, k)
    np.testing.assert_array_equal(out_bits(_run(offload, x, chunk, k)), out_bits(a))


def test_hot_set_rejections():
    from expert_major_chunked_gb300 import binding
    k, chunk = 4, 64
    inp = _small(14, T=64)
    resident, offload = _pair(inp, k, chunk, 8)
    with pytest.raises(binding.MoeError):
        resident.set_hot_experts([1])          # no offloaded experts
    for bad in ([1, 1], [64], [-1], list(range(65))):
        with pytest.raises(binding.MoeError):
            offload.set_hot_experts(bad)
    # the plan is unchanged after a rejected set
    x = inp["x"].cuda()
    np.testing.assert_array_equal(out_bits(_run(offload, x, chunk, k)), out_bits(_run(resident, x, chunk, k)))


def test_zipf_offload_with_popular_experts_resident():
    """12,001 tokens under the Zipf(1.1) router, 32-slot ring: the 64 experts routed in the most chunks of a first
    run, kept resident, take their (chunk, expert) pairs off the staging list; output bytes unchanged."""
    wl, inp = cpu_inputs("e512_zipf_offload_t12001")
    chunk = wl.chunks[0]
    x = inp["x"].cuda()
    resident, offload = _pair(inp, wl.top_k, chunk, wl.offload_slots)
    a = _run(resident, x, chunk, wl.top_k)
    n_chunks = (wl.tokens + chunk - 1) // chunk
    offs = torch.empty((n_chunks, wl.n_experts + 1), dtype=torch.int32, device="cuda")
    b = _run(offload, x, chunk, wl.top_k, offs)
    np.testing.assert_array_equal(out_bits(b), out_bits(a))
    before = offload.stats()["experts_copied"]
    routed = _counts(offs) > 0
    order = np.lexsort((np.arange(wl.n_experts), -_counts(offs).sum(0), -routed.sum(0)))
    hot = order[:64]
    offload.set_hot_experts(hot)
    b = _run(offload, x, chunk, wl.top_k)
    np.testing.assert_array_equal(out_bits(b), out_bits(a))
    st = offload.stats()
    assert st["experts_hot"] == int(routed[:, hot].sum())
    assert st["experts_copied"] == before - st["experts_hot"]
