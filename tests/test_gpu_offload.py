"""Offloaded experts (pinned host banks streamed through a ring of HBM slots) on the GPU.

The ring only changes where the expert weights are read from; the kernels and their accumulation order are the
same, so the output must equal the resident-weight run byte for byte, and the oracle within the usual bound.
"""

import numpy as np
import pytest
import torch

from layer_helpers import MAX_ABS, REL_L2, compare_out, cpu_inputs, out_bits, sample_tokens

pytestmark = pytest.mark.gpu


def _small(seed, T=300, H=256, E=64, I=128, Is=128):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"x": r(T, H, std=1.0), "w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I),
            "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


def _layers(inp, k, max_chunk, slots, mode=None):
    from expert_major_chunked_gb300 import binding
    dev = {n: t.cuda() for n, t in inp.items()}
    names = ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")
    resident = binding.MoePrefill({n: dev[n] for n in names}, top_k=k, max_chunk=max_chunk)
    host = {n: (inp[n].pin_memory() if n in ("w_gu", "w_down") else dev[n]) for n in names}
    offload = binding.MoePrefill(host, top_k=k, max_chunk=max_chunk, offload_slots=slots)
    if mode is not None:
        offload.set_offload_copy(mode)
    return dev, resident, offload, host


def _run(layer, x, chunk, k, copy_stream=None):
    T = x.shape[0]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = layer.run(x, chunk, topk_id=ids, copy_stream=copy_stream)
    layer.raise_on_device_error()
    return out.cpu(), ids.cpu()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("slots", [2, 8, 64])
def test_offload_equals_resident_small(oracle_lib, slots, mode):
    k = 4
    inp = _small(1)
    dev, resident, offload, _ = _layers(inp, k, max_chunk=300, slots=slots, mode=mode)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(inp, k)
    for chunk in (64, 300, 17):
        a, ia = _run(resident, dev["x"], chunk, k)
        b, ib = _run(offload, dev["x"], chunk, k)
        np.testing.assert_array_equal(out_bits(b), out_bits(a))
        np.testing.assert_array_equal(ib.numpy(), ref_ids)
        max_abs, rel = compare_out(b, ref_bf, oracle_lib)
        assert max_abs <= MAX_ABS and rel <= REL_L2


@pytest.mark.parametrize("mode", [0, 1])
def test_offload_with_caller_copy_stream_and_repeats(mode):
    k = 4
    inp = _small(2, T=513)
    dev, resident, offload, _ = _layers(inp, k, max_chunk=128, slots=8, mode=mode)
    cs = torch.cuda.Stream()
    a, _ = _run(resident, dev["x"], 128, k)
    for _ in range(3):
        b, _ = _run(offload, dev["x"], 128, k, copy_stream=cs)
        np.testing.assert_array_equal(out_bits(b), out_bits(a))


def test_offload_rejects_device_banks():
    from expert_major_chunked_gb300 import binding
    inp = _small(3, T=16)
    dev = {n: t.cuda() for n, t in inp.items()}
    dims = binding.moe_dims(256, 64, 128, 4, 128, 1, 16, 8)
    with pytest.raises(binding.MoeError) as e:
        binding.moe_prefill_plan(dims, dev["w_router"].data_ptr(), dev["w_gu"].data_ptr(), dev["w_down"].data_ptr(),
                                 dev["ws_gu"].data_ptr(), dev["ws_down"].data_ptr())
    assert e.value.status == -1


def test_offload_full_workload(oracle_lib):
    """The 12,001-token offloaded workload: 512 experts in pinned host memory, a 32-slot ring, chunk 1024."""
    wl, inp = cpu_inputs("e512_offload_t12001")
    chunk = wl.chunks[0]
    dev, resident, offload, _ = _layers(inp, wl.top_k, max_chunk=chunk, slots=wl.offload_slots)
    a, ia = _run(resident, dev["x"], chunk, wl.top_k)
    b, ib = _run(offload, dev["x"], chunk, wl.top_k)
    np.testing.assert_array_equal(out_bits(b), out_bits(a))
    np.testing.assert_array_equal(ib.numpy(), ia.numpy())
    sample = sample_tokens(wl.tokens, (chunk,), extra=32)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(inp, wl.top_k, token_idx=sample)
    np.testing.assert_array_equal(ib.numpy()[sample], ref_ids)
    max_abs, rel = compare_out(b[sample], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2


def test_routed_staging_counts_and_skips():
    """Routed staging copies exactly the (chunk, expert) pairs with rows: checked against the expert offsets that
    the same run reports, under a skewed router (most experts of a chunk get no rows) and with the copy engines."""
    from expert_major_chunked_gb300 import binding
    k, E, T, chunk = 4, 64, 300, 64
    inp = _small(4, T=T, E=E)
    # skew: a large positive router bias for 8 experts through input channel 0
    inp["x"][:, 0] = 1.0
    wr = inp["w_router"].float()
    wr[:, 0] = -40.0
    wr[:8, 0] = 40.0
    inp["w_router"] = wr.to(torch.bfloat16)
    dev, resident, offload, _ = _layers(inp, k, max_chunk=chunk, slots=8, mode=binding.OFFLOAD_COPY_ROUTED)
    a, _ = _run(resident, dev["x"], chunk, k)
    n_chunks = (T + chunk - 1) // chunk
    offs = torch.empty((n_chunks, E + 1), dtype=torch.int32, device="cuda")
    out = offload.run(dev["x"], chunk, expert_offsets=offs)
    offload.raise_on_device_error()
    np.testing.assert_array_equal(out_bits(out.cpu()), out_bits(a))
    st = offload.stats()
    counts = np.diff(offs.cpu().numpy(), axis=1)
    assert st["experts_copied"] == int((counts > 0).sum())
    assert st["experts_copied"] + st["experts_skipped"] == n_chunks * E
    assert st["experts_skipped"] > n_chunks * E // 2
    offload.set_offload_copy(binding.OFFLOAD_COPY_ALL)
    b, _ = _run(offload, dev["x"], chunk, k)
    np.testing.assert_array_equal(out_bits(b), out_bits(a))


def test_offload_copy_mode_rejected_without_offload():
    from expert_major_chunked_gb300 import binding
    inp = _small(5, T=16)
    dev = {n: t.cuda() for n, t in inp.items()}
    layer = binding.MoePrefill({n: dev[n] for n in ("w_router", "w_gu", "w_down", "ws_gu", "ws_down")}, top_k=4,
                               max_chunk=16)
    with pytest.raises(binding.MoeError):
        layer.set_offload_copy(binding.OFFLOAD_COPY_ROUTED)


def test_zipf_offload_workload(oracle_lib):
    """12,001 tokens, Zipf(1.1) router prior, 32-slot ring, chunk 1024, routed staging: equals resident weights
    byte for byte and the oracle on sampled tokens."""
    wl, inp = cpu_inputs("e512_zipf_offload_t12001")
    chunk = wl.chunks[0]
    dev, resident, offload, _ = _layers(inp, wl.top_k, max_chunk=chunk, slots=wl.offload_slots)
    a, ia = _run(resident, dev["x"], chunk, wl.top_k)
    b, ib = _run(offload, dev["x"], chunk, wl.top_k)
    np.testing.assert_array_equal(out_bits(b), out_bits(a))
    np.testing.assert_array_equal(ib.numpy(), ia.numpy())
    st = offload.stats()
    n_chunks = (wl.tokens + chunk - 1) // chunk
    assert st["experts_copied"] + st["experts_skipped"] == n_chunks * wl.n_experts
    sample = sample_tokens(wl.tokens, (chunk,), extra=24)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(inp, wl.top_k, token_idx=sample)
    np.testing.assert_array_equal(ib.numpy()[sample], ref_ids)
    max_abs, rel = compare_out(b[sample], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2
