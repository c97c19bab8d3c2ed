"""Block-scaled FP4 (NVFP4) routed experts on the GPU.

The deep-prefill draft's review ("To land") quantises prompt-tile weights. Here the routed experts' weights are E2M1
codes, two per byte, with one E4M3 scale per 16 weights along K; a code times its scale is exactly a bf16 value, and
the kernels decode tiles to bf16 in shared memory before the tensor-core path. So the layer must equal, byte for
byte, the bf16 layer run on the weights the oracle decodes, stay chunk-invariant, match the float64 oracle on those
weights within the layer's bound, and give the same bytes when the code banks are staged from pinned host memory.
"""

import numpy as np
import pytest
import torch

from layer_helpers import MAX_ABS, REL_L2, compare_out, cpu_inputs, out_bits, sample_tokens

pytestmark = pytest.mark.gpu


def _decoded(oracle_lib, q):
    gu = oracle_lib.dequant_nvfp4(q["w_gu_q"].numpy(), q["w_gu_s"].numpy())
    dn = oracle_lib.dequant_nvfp4(q["w_down_q"].numpy(), q["w_down_s"].numpy())
    return (torch.from_numpy(gu.view(np.int16)).view(torch.bfloat16),
            torch.from_numpy(dn.view(np.int16)).view(torch.bfloat16))


def _layers(oracle_lib, inp, k, max_chunk):
    from expert_major_chunked_gb300 import binding, workloads
    q = workloads.nvfp4_weights(inp)
    gu, dn = _decoded(oracle_lib, q)
    ref_inp = dict(inp, w_gu=gu, w_down=dn)
    dev = {n: t.cuda() for n, t in ref_inp.items()}
    common = {n: dev[n] for n in ("w_router", "ws_gu", "ws_down") if n in dev}
    bf16 = binding.MoePrefill(dict(common, w_gu=dev["w_gu"], w_down=dev["w_down"]), top_k=k, max_chunk=max_chunk)
    fp4 = binding.MoePrefill(dict(common, **{n: t.cuda() for n, t in q.items()}), top_k=k, max_chunk=max_chunk,
                             weight_format="nvfp4")
    return ref_inp, dev, bf16, fp4


def _run(layer, x, chunk, k):
    T = x.shape[0]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = layer.run(x, chunk, topk_id=ids)
    layer.raise_on_device_error()
    return out.cpu(), ids.cpu().numpy()


def _small(seed, T, H, E, I, Is, k):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"x": r(T, H, std=1.0), "w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I),
            "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


@pytest.mark.parametrize("T,H,E,I,Is,k", [(300, 256, 64, 128, 128, 4),    # N tiles 256 (gate/up) and 256 (down)
                                          (257, 320, 32, 192, 64, 3),     # gate/up halves of 64, down N tile 64
                                          (40, 512, 16, 256, 256, 2)])
def test_nvfp4_equals_bf16_on_decoded_weights(oracle_lib, T, H, E, I, Is, k):
    inp = _small(T + H + 1, T, H, E, I, Is, k)
    ref_inp, dev, bf16, fp4 = _layers(oracle_lib, inp, k, max_chunk=T)
    for chunk in (T, min(64, T), 17):
        a, ia = _run(bf16, dev["x"], chunk, k)
        b, ib = _run(fp4, dev["x"], chunk, k)
        np.testing.assert_array_equal(out_bits(b), out_bits(a))
        np.testing.assert_array_equal(ib, ia)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(ref_inp, k)
    np.testing.assert_array_equal(ib, ref_ids)
    max_abs, rel = compare_out(b, ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2


def test_nvfp4_every_code_and_wide_scales(oracle_lib):
    """Weights that use all 16 E2M1 codes in both nibbles, and down-projection scales from the E4M3 subnormal 2^-9
    to its largest value 448, so a swapped nibble order, a dropped sign or a misread scale changes the bytes."""
    from expert_major_chunked_gb300 import binding
    k, T, H, E, I = 2, 64, 256, 16, 128
    gen = torch.Generator().manual_seed(5)
    inp = _small(5, T, H, E, I, 0, k)
    scale_codes = torch.tensor([0x01, 0x08, 0x20, 0x30, 0x38, 0x40, 0x48, 0x7e], dtype=torch.uint8)
    q = {"w_gu_q": torch.randint(0, 256, (E, 2 * I, H // 2), generator=gen, dtype=torch.uint8),
         "w_gu_s": torch.full((E, H // 16, 2 * I), 0x20, dtype=torch.uint8),  # 2^-3 keeps the activations small
         "w_down_q": torch.randint(0, 256, (E, H, I // 2), generator=gen, dtype=torch.uint8),
         "w_down_s": scale_codes[torch.randint(0, 8, (E, I // 16, H), generator=gen)]}
    gu, dn = _decoded(oracle_lib, q)
    dev = {n: t.cuda() for n, t in dict(inp, w_gu=gu, w_down=dn).items()}
    bf16 = binding.MoePrefill({"w_router": dev["w_router"], "w_gu": dev["w_gu"], "w_down": dev["w_down"]},
                              top_k=k, max_chunk=T)
    fp4 = binding.MoePrefill(dict(w_router=dev["w_router"], **{n: t.cuda() for n, t in q.items()}), top_k=k,
                             max_chunk=T, weight_format="nvfp4")
    a, ia = _run(bf16, dev["x"], T, k)
    b, ib = _run(fp4, dev["x"], T, k)
    assert torch.isfinite(a.float()).all()
    np.testing.assert_array_equal(out_bits(b), out_bits(a))
    np.testing.assert_array_equal(ib, ia)


@pytest.mark.parametrize("name", ["e512_zipf_t4099", "e512_t16022"])
def test_nvfp4_workloads(oracle_lib, name):
    wl, inp = cpu_inputs(name)
    ref_inp, dev, bf16, fp4 = _layers(oracle_lib, inp, wl.top_k, max_chunk=max(wl.chunks))
    first = None
    for chunk in wl.chunks:
        b, ib = _run(fp4, dev["x"], chunk, wl.top_k)
        if first is None:
            first = (b, ib)
            a, ia = _run(bf16, dev["x"], chunk, wl.top_k)
            np.testing.assert_array_equal(out_bits(b), out_bits(a))
        else:
            np.testing.assert_array_equal(out_bits(b), out_bits(first[0]))
    sample = sample_tokens(wl.tokens, wl.chunks, extra=24)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(ref_inp, wl.top_k, token_idx=sample)
    np.testing.assert_array_equal(first[1][sample], ref_ids)
    max_abs, rel = compare_out(first[0][sample], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2


def test_nvfp4_offloaded_codes_equal_resident():
    """E2M1 code banks in pinned host memory, staged through a ring (both staging modes), give the bytes of the
    resident NVFP4 layer; scales stay in device memory."""
    from expert_major_chunked_gb300 import binding, workloads
    k = 4
    inp = _small(13, 300, 256, 64, 128, 128, k)
    q = workloads.nvfp4_weights(inp)
    dev = {n: t.cuda() for n, t in inp.items()}
    common = {n: dev[n] for n in ("w_router", "ws_gu", "ws_down")}
    resident = binding.MoePrefill(dict(common, **{n: t.cuda() for n, t in q.items()}), top_k=k, max_chunk=300,
                                  weight_format="nvfp4")
    host = dict(common, w_gu_q=q["w_gu_q"].pin_memory(), w_down_q=q["w_down_q"].pin_memory(),
                w_gu_s=q["w_gu_s"].cuda(), w_down_s=q["w_down_s"].cuda())
    a, ia = _run(resident, dev["x"], 64, k)
    for slots in (2, 16):
        off = binding.MoePrefill(host, top_k=k, max_chunk=300, offload_slots=slots, weight_format="nvfp4")
        for mode in (binding.OFFLOAD_COPY_ROUTED, binding.OFFLOAD_COPY_ALL):
            off.set_offload_copy(mode)
            b, ib = _run(off, dev["x"], 64, k)
            np.testing.assert_array_equal(out_bits(b), out_bits(a))
            np.testing.assert_array_equal(ib, ia)
