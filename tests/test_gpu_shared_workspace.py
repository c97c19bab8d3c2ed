"""Layers that share one workspace, on the GPU.

Umbrella PR #1113, "Memory and execution split", *Expert movement*: the deep-prefill ring reuses one pool of device
storage across layers. Here several plans (layers) take turns on one workspace. What a run leaves there for later
runs (a hot set's slots, the slot map, a first window staged ahead by a prefetch) is valid only for the plan and
hot set that put it there, so every run must still equal its layer's resident-weight run byte for byte: when
plans alternate A, B, A, when their hot sets differ, when one layer prefetches into the workspace the other is
still running on, and when a prefetch is made by one plan and dropped by another plan's run.
"""

import numpy as np
import pytest
import torch

from layer_helpers import MAX_ABS, REL_L2, compare_out, cpu_inputs, out_bits, sample_tokens

pytestmark = pytest.mark.gpu

NAMES = ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")


def _weights(seed, E=64, H=256, I=128, Is=128):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I), "ws_gu": r(2 * Is, H),
            "ws_down": r(H, Is)}


def _pair(w, k, max_chunk, slots, hot=None, mode=None):
    """(resident layer, offloaded layer) on the same weights; the offloaded one with an optional hot set."""
    from expert_major_chunked_gb300 import binding
    dev = {n: t.cuda() for n, t in w.items()}
    resident = binding.MoePrefill(dev, top_k=k, max_chunk=max_chunk)
    host = {n: (w[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in w}
    off = binding.MoePrefill(host, top_k=k, max_chunk=max_chunk, offload_slots=slots)
    if hot:
        off.set_hot_experts(hot)
    if mode is not None:
        off.set_offload_copy(mode)
    return resident, off


def _share(layers):
    """Point every layer at one workspace as large as the largest of theirs."""
    n = max(layer.workspace_bytes for layer in layers)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    for layer in layers:
        layer.workspace = ws
    return ws


def _x(seed, T, H=256):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(T, H, generator=gen).to(torch.bfloat16).cuda()


def _run(layer, x, chunk):
    out = layer.run(x, chunk)
    layer.raise_on_device_error()
    return out_bits(out.cpu())


@pytest.mark.parametrize("mode", [0, 1])
def test_two_offloaded_plans_alternate_on_one_workspace(mode):
    """A, B, A, B, A on one workspace, with different weights and different hot sets (of different sizes, so the
    ring's down slots lie at different offsets): each run equals its resident run."""
    k, T, chunk = 4, 300, 64
    ra, oa = _pair(_weights(31), k, chunk, 8, hot=[0, 3, 9, 17, 40], mode=mode)
    rb, ob = _pair(_weights(32), k, chunk, 8, hot=[3, 0, 50], mode=mode)
    xa, xb = _x(33, T), _x(34, T)
    ref_a, ref_b = _run(ra, xa, chunk), _run(rb, xb, chunk)
    _share([oa, ob])
    for i in range(5):
        if i % 2 == 0:
            np.testing.assert_array_equal(_run(oa, xa, chunk), ref_a)
        else:
            np.testing.assert_array_equal(_run(ob, xb, chunk), ref_b)


def test_same_plan_runs_again_after_another_workspace():
    """A on workspace 1, A on workspace 2, B on workspace 1, A on workspace 1: the hot set kept in workspace 1 is
    used only while A was the last plan to run there."""
    k, T, chunk = 4, 257, 64
    ra, oa = _pair(_weights(41), k, chunk, 8, hot=[1, 2, 3, 4])
    rb, ob = _pair(_weights(42), k, chunk, 8, hot=[4, 3, 2, 1])
    x = _x(43, T)
    ref_a, ref_b = _run(ra, x, chunk), _run(rb, x, chunk)
    ws1 = _share([oa, ob])
    ws2 = torch.empty_like(ws1)
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
    oa.workspace = ws2
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
    np.testing.assert_array_equal(_run(ob, x, chunk), ref_b)   # on ws1
    oa.workspace = ws1
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)   # A again: its hot set is reused, not restaged


def test_offloaded_and_resident_plans_share_a_workspace():
    k, T, chunk = 4, 300, 128
    ra, oa = _pair(_weights(51), k, chunk, 8, hot=[7, 8])
    rc, _ = _pair(_weights(52), k, chunk, 8)
    x = _x(53, T)
    ref_a, ref_c = _run(ra, x, chunk), _run(rc, x, chunk)
    # the resident plan's layout is shorter: its h and y lie over the offloaded plan's ring, hot slots and slot map
    _share([oa, rc])
    for _ in range(2):
        np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
        np.testing.assert_array_equal(_run(rc, x, chunk), ref_c)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("slots,hot", [(2, None), (16, None), (8, ([0, 5, 33], [2, 61]))])
def test_chain_with_prefetch_on_one_workspace(mode, slots, hot):
    """Two layers on one workspace, each prefetching the other's first window while the other runs: the prefetch
    of layer 1 overlaps the tail of layer 0's run on the same bytes' workspace."""
    k, T, chunk = 4, 300, 64
    r0, o0 = _pair(_weights(61), k, chunk, slots, hot=hot[0] if hot else None, mode=mode)
    r1, o1 = _pair(_weights(62), k, chunk, slots, hot=hot[1] if hot else None, mode=mode)
    x = _x(63, T)
    ref = out_bits(r1.run(r0.run(x, chunk), chunk).cpu())
    _share([o0, o1])
    cs = torch.cuda.Stream()
    o0.prefetch(cs)
    for _ in range(3):
        h = o0.run(x, chunk)
        o1.prefetch(cs)
        h = o1.run(h, chunk)
        o0.prefetch(cs)
        np.testing.assert_array_equal(out_bits(h.cpu()), ref)
    o0.raise_on_device_error()


def test_prefetch_dropped_by_another_plans_run():
    """B prefetches into the workspace, A runs there (dropping B's window and overwriting the ring), B runs: B must
    stage its first window again. Also two prefetches in a row by different plans."""
    k, T, chunk = 4, 257, 64
    ra, oa = _pair(_weights(71), k, chunk, 8)
    rb, ob = _pair(_weights(72), k, chunk, 8, hot=[0, 1])
    x = _x(73, T)
    ref_a, ref_b = _run(ra, x, chunk), _run(rb, x, chunk)
    _share([oa, ob])
    ob.prefetch()
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
    np.testing.assert_array_equal(_run(ob, x, chunk), ref_b)
    ob.prefetch()
    oa.prefetch()                          # A's window replaces B's in the same slots
    np.testing.assert_array_equal(_run(ob, x, chunk), ref_b)
    oa.prefetch()
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)


def test_full_offload_workload_two_hot_sets_on_one_workspace(oracle_lib):
    """The 12,001-token offloaded workload (512 experts, 32-slot ring, chunk 1024): two plans on the same banks with
    disjoint 64-expert hot sets take turns on one workspace, so each run finds the other set in its hot slots.
    Every run equals the resident run byte for byte and the oracle on sampled tokens."""
    from expert_major_chunked_gb300 import binding
    wl, inp = cpu_inputs("e512_offload_t12001")
    chunk = wl.chunks[0]
    dev = {n: inp[n].cuda() for n in NAMES}
    x = inp["x"].cuda()
    resident = binding.MoePrefill(dev, top_k=wl.top_k, max_chunk=chunk)
    ref = resident.run(x, chunk).cpu()
    resident.raise_on_device_error()
    host = {n: (inp[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in NAMES}
    a = binding.MoePrefill(host, top_k=wl.top_k, max_chunk=chunk, offload_slots=wl.offload_slots)
    b = binding.MoePrefill(host, top_k=wl.top_k, max_chunk=chunk, offload_slots=wl.offload_slots)
    a.set_hot_experts(list(range(0, 128, 2)))
    b.set_hot_experts(list(range(1, 128, 2)))
    _share([a, b])
    outs = []
    for layer in (a, b, a):
        out = layer.run(x, chunk)
        layer.raise_on_device_error()
        outs.append(out.cpu())
        np.testing.assert_array_equal(out_bits(outs[-1]), out_bits(ref))
    sample = sample_tokens(wl.tokens, (chunk,), extra=16)
    _, ref_bf, _, _ = oracle_lib.moe_forward(inp, wl.top_k, token_idx=sample)
    max_abs, rel = compare_out(outs[-1][sample], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2


def test_forgotten_workspace_is_restaged():
    """The library remembers the most recently used workspaces (256); a plan that returns to a workspace whose record
    was dropped, after another plan ran there, must stage its hot set again."""
    k, T, chunk = 4, 130, 64
    ra, oa = _pair(_weights(81), k, chunk, 8, hot=[2, 40])
    rb, ob = _pair(_weights(82), k, chunk, 8, hot=[40, 2])
    x = _x(83, T)
    ref_a, ref_b = _run(ra, x, chunk), _run(rb, x, chunk)
    ws = _share([oa, ob])
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)
    np.testing.assert_array_equal(_run(ob, x, chunk), ref_b)   # B's hot set now in the shared workspace
    # 300 other workspaces (kept alive, so that each has its own address) push the shared one's record out
    n = oa.workspace_bytes
    others = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(300)]
    from expert_major_chunked_gb300 import binding
    for w in others:
        binding.moe_prefill_run(oa.plan, x.data_ptr(), T, chunk, w.data_ptr(), n, torch.empty_like(x).data_ptr())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_run(oa, x, chunk), ref_a)   # must not trust the slots it staged long ago
    np.testing.assert_array_equal(_run(ob, x, chunk), ref_b)
    for w in others:
        binding.moe_prefill_forget_workspace(w.data_ptr())


def test_forget_workspace_before_reuse():
    """A workspace's memory reused for something else after moe_prefill_forget_workspace: the next run of the same
    plan there stages its hot set again instead of trusting what it left."""
    from expert_major_chunked_gb300 import binding
    k, T, chunk = 4, 130, 64
    ra, oa = _pair(_weights(91), k, chunk, 8, hot=[3, 9])
    x = _x(92, T)
    ref = _run(ra, x, chunk)
    ws = oa.workspace
    np.testing.assert_array_equal(_run(oa, x, chunk), ref)
    binding.moe_prefill_forget_workspace(ws.data_ptr())
    ws.fill_(0x7F)                          # someone else's data at the same address
    np.testing.assert_array_equal(_run(oa, x, chunk), ref)
    assert binding.lib().moe_prefill_forget_workspace(None) == -1
