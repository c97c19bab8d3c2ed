"""The allocation-free entry point (moe_prefill_run_noalloc) through the C ABI, against moe_prefill_run (GPU).

It serves callers that cannot allocate device memory where they run the layer (their memory belongs to another
allocator or pool, or allocation is forbidden after start-up). Its scratch is a fixed array inside the library, so
two calls in a row reuse the same bytes: the second call must not see anything of the first. This file is
collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 1e-3


def _inputs(seed, T, H, E, I, Is, std=0.02):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, sd=std: (torch.randn(s, generator=gen) * sd).to(torch.bfloat16)
    return {"x": r(T, H, sd=1.0), "w_router": r(E, H), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I),
            "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


def _noalloc(L, plan, x, T, chunk, out, ids, w, status, stream=None):
    return L.moe_prefill_run_noalloc(plan, x.data_ptr(), T, chunk, out.data_ptr(), ids.data_ptr(), w.data_ptr(),
                                     None, None, status.data_ptr(), stream)


def _close(a, b):
    a64, b64 = a.to(torch.float64), b.to(torch.float64)
    diff = (a64 - b64).abs()
    rel = (a64 - b64).norm() / b64.norm()
    return diff.max().item() <= MAX_ABS and rel.item() <= REL_L2


def test_noalloc_matches_run_twice_in_a_row():
    from expert_major_chunked_gb300 import binding
    L = binding.lib()
    L.moe_prefill_run_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.moe_prefill_run_noalloc.restype = ctypes.c_int
    k, chunk = 8, 256
    inp = _inputs(1, T=700, H=2048, E=128, I=768, Is=2048)
    dev = {n: t.cuda() for n, t in inp.items()}
    layer = binding.MoePrefill({n: dev[n] for n in ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")},
                               top_k=k, max_chunk=chunk)
    assert layer.workspace_bytes <= (64 << 20)
    T = dev["x"].shape[0]
    ids_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_ref = torch.empty((T, k), device="cuda")
    ref = layer.run(dev["x"], chunk, topk_id=ids_ref, topk_w=w_ref)
    layer.raise_on_device_error()

    # a second input for the first no-alloc call, so that the array holds another token set's data when the call
    # under test runs
    other = (torch.randn((T, 2048), generator=torch.Generator().manual_seed(9))).to(torch.bfloat16).cuda()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    outs = []
    for x in (other, dev["x"], dev["x"]):
        out = torch.empty_like(x)
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), device="cuda")
        status.fill_(-1)
        assert _noalloc(L, layer.plan, x, T, chunk, out, ids, w, status) == 0, binding.moe_prefill_last_error()
        torch.cuda.synchronize()
        assert status.item() == 0
        outs.append((out, ids, w))
    for out, ids, w in outs[1:]:
        assert _close(out.cpu(), ref.cpu())
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))   # same kernels, same bytes
        assert torch.equal(ids, ids_ref)
        assert torch.equal(w, w_ref)


def test_noalloc_rejects_plans_larger_than_its_array():
    from expert_major_chunked_gb300 import binding
    L = binding.lib()
    inp = _inputs(2, T=64, H=2048, E=128, I=768, Is=2048)
    dev = {n: t.cuda() for n, t in inp.items()}
    layer = binding.MoePrefill({n: dev[n] for n in ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")},
                               top_k=8, max_chunk=4096)
    assert layer.workspace_bytes > (64 << 20)
    out = torch.empty_like(dev["x"])
    ids = torch.empty((64, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((64, 8), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(L, layer.plan, dev["x"], 64, 64, out, ids, w, status) == -3
    assert b"scratch" in L.moe_prefill_last_error()


def test_noalloc_offloaded_plans_take_turns():
    """Two offloaded layers with different weights and different hot sets, called A, B, A, B through the built-in
    array: each run must find its own hot experts and slot map there, not the other layer's. Each output equals the
    same plan's run on a workspace of its own, byte for byte."""
    from expert_major_chunked_gb300 import binding
    L = binding.lib()
    k, chunk, T = 4, 64, 300
    layers, refs, xs = [], [], []
    for seed, hot in ((11, [0, 3, 9, 17, 40]), (12, [3, 0, 50])):
        inp = _inputs(seed, T=T, H=256, E=64, I=128, Is=128, std=0.05)
        dev = {n: inp[n].cuda() for n in ("w_router", "ws_gu", "ws_down")}
        host = dict(dev, w_gu=inp["w_gu"].pin_memory(), w_down=inp["w_down"].pin_memory())
        layer = binding.MoePrefill(host, top_k=k, max_chunk=chunk, offload_slots=8)
        layer.set_hot_experts(hot)
        assert layer.workspace_bytes <= (64 << 20)
        x = inp["x"].cuda()
        ref = layer.run(x, chunk)
        layer.raise_on_device_error()
        layers.append(layer)
        refs.append(ref.cpu())
        xs.append(x)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for i in range(4):
        j = i % 2
        out = torch.empty_like(xs[j])
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), device="cuda")
        status.fill_(-1)
        assert _noalloc(L, layers[j].plan, xs[j], T, chunk, out, ids, w, status) == 0, binding.moe_prefill_last_error()
        torch.cuda.synchronize()
        assert status.item() == 0
        assert _close(out.cpu(), refs[j])
        assert torch.equal(out.cpu().view(torch.int16), refs[j].view(torch.int16))
