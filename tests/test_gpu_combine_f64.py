"""The float64 tree combine (expert-parallel partials) on the GPU, against the oracle, bit for bit.

"EXL3 Flash Next: deep prefill (3/8)" ("What this changes", "Checklist"): the prefill partials of a tensor-parallel
split are float64, summed with one rounding to float32 at the finish, so a split over two GPUs equals one GPU bit for
bit. The kernels here take the same steps as the oracle's dense tree over the expert ids, so every value — the
float64 partials (signed zeros included), the float32 finish and the bf16 output — must match exactly.
"""

import numpy as np
import pytest
import torch

from conftest import read_fixture
from layer_helpers import MAX_ABS, REL_L2, GpuLayer, compare_out, cpu_inputs, out_bits, sample_tokens

pytestmark = pytest.mark.gpu


def _case(seed, n, k, E, H, rows=None, zeros=0.0):
    rng = np.random.default_rng(seed)
    R = rows or n * k
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(n)]).astype(np.int32)  # unsorted slots
    w = rng.random((n, k)).astype(np.float32)
    y = (rng.standard_normal((R, H)) * 10.0 ** rng.integers(-4, 5, size=(R, H))).astype(np.float32)
    if zeros:  # signed zeros and float32 subnormals (the conversions' special paths)
        mask = rng.random((R, H)) < zeros
        specials = np.array([0.0, -0.0, 1e-40, -3e-42, 1.4e-45, -1.2e-38], dtype=np.float32)
        y[mask] = specials[rng.integers(0, len(specials), size=int(mask.sum()))]
    s = rng.standard_normal((n, H)).astype(np.float32)
    tr = rng.integers(0, R, size=(n, k)).astype(np.int32)
    return y, w, tr, ids, s


def _dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


def _gpu_whole(y, w, tr, ids, s, E):
    from expert_major_chunked_gb300 import binding as b
    n, k = w.shape
    H = y.shape[1]
    dy, dw, dtr, dids = _dev(y, w, tr, ids)
    ds = _dev(s)[0] if s is not None else None
    out = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    f32 = torch.empty((n, H), dtype=torch.float32, device="cuda")
    b.moe_prefill_combine_f64(dy.data_ptr(), dw.data_ptr(), dtr.data_ptr(), dids.data_ptr(),
                              ds.data_ptr() if ds is not None else None, n, k, H, E, out.data_ptr(), f32.data_ptr())
    torch.cuda.synchronize()
    return f32.cpu().numpy(), out_bits(out.cpu())


def _gpu_split(y, w, tr, ids, s, E, parts):
    from expert_major_chunked_gb300 import binding as b
    n, k = w.shape
    H = y.shape[1]
    dy, dw, dtr, dids = _dev(y, w, tr, ids)
    ds = _dev(s)[0] if s is not None else None
    pieces = [torch.empty((n, H), dtype=torch.float64, device="cuda") for _ in range(parts)]
    for p, buf in enumerate(pieces):
        b.moe_prefill_combine_partial_f64(dy.data_ptr(), dw.data_ptr(), dtr.data_ptr(), dids.data_ptr(), n, k, H, E,
                                          parts, p, buf.data_ptr())
    out = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    f32 = torch.empty((n, H), dtype=torch.float32, device="cuda")
    b.moe_prefill_combine_finish_f64([t.data_ptr() for t in pieces], ds.data_ptr() if ds is not None else None, n, H,
                                     out.data_ptr(), f32.data_ptr())
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in pieces], f32.cpu().numpy(), out_bits(out.cpu())


def _bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint64 if a.itemsize == 8 else np.uint32)


def test_hand_worked_example_on_gpu():
    fx = read_fixture("hand_worked_tree_combine.txt")
    n, k, E, H = (int(v) for v in fx["dims"])
    pad = lambda a, cols: np.concatenate([a, np.zeros((a.shape[0], cols - a.shape[1]), a.dtype)], axis=1)
    y = pad(np.array(fx["y"], np.float32).reshape(n * k, H), 4)
    s = pad(np.array(fx["s"], np.float32).reshape(n, H), 4)
    w = np.array(fx["w"], np.float32).reshape(n, k)
    tr = np.array(fx["token_row"], np.int32).reshape(n, k)
    ids = np.array(fx["topk_id"], np.int32).reshape(n, k)
    f32, bf = _gpu_whole(y, w, tr, ids, s, E)
    np.testing.assert_array_equal(_bits(f32[:, :H]), _bits(np.array(fx["out_f32"], np.float32).reshape(n, H)))
    np.testing.assert_array_equal(bf[:, :H], np.array(fx["out_bf16"], np.uint16).reshape(n, H))
    pieces, f32s, bfs = _gpu_split(y, w, tr, ids, s, E, 2)
    for p in range(2):
        np.testing.assert_array_equal(_bits(pieces[p][:, :H]),
                                      _bits(np.array(fx[f"part{p}"], np.float64).reshape(n, H)))
    np.testing.assert_array_equal(bfs, bf)
    f32n, bfn = _gpu_whole(y, w, tr, ids, None, E)
    np.testing.assert_array_equal(bfn[:, :H], np.array(fx["out_bf16_no_shared"], np.uint16).reshape(n, H))


@pytest.mark.parametrize("n,k,E,H,zeros", [(257, 8, 512, 256, 0.0), (64, 10, 512, 2048, 0.0), (100, 1, 48, 64, 0.3),
                                           (33, 32, 1024, 128, 0.0), (50, 6, 96, 512, 0.5)])
def test_whole_and_split_equal_oracle(oracle_lib, n, k, E, H, zeros):
    y, w, tr, ids, s = _case(n + k + E, n, k, E, H, zeros=zeros)
    ref_f32, ref_bf = oracle_lib.combine_tree_f64(y, w, tr, ids, E, s)
    f32, bf = _gpu_whole(y, w, tr, ids, s, E)
    np.testing.assert_array_equal(_bits(f32), _bits(ref_f32))
    np.testing.assert_array_equal(bf, ref_bf)
    Ep = 1 << (E - 1).bit_length()
    for parts in sorted({2, 4, min(16, Ep)}):
        pieces, f32s, bfs = _gpu_split(y, w, tr, ids, s, E, parts)
        for p in range(parts):
            ref_p = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E, parts, p)
            np.testing.assert_array_equal(_bits(pieces[p]), _bits(ref_p))
        np.testing.assert_array_equal(_bits(f32s), _bits(f32))
        np.testing.assert_array_equal(bfs, bf)


def test_empty_and_all_outside_part():
    y, w, tr, ids, s = _case(5, 16, 4, 64, 64)
    ids[:] = np.array([0, 1, 2, 3], np.int32)  # every token's experts lie in the first of 4 parts
    pieces, _, _ = _gpu_split(y, w, tr, ids, None, 64, 4)
    for p in (1, 2, 3):
        np.testing.assert_array_equal(_bits(pieces[p]), np.zeros_like(_bits(pieces[p])))  # +0.0 everywhere
    from expert_major_chunked_gb300 import binding as b
    b.moe_prefill_combine_f64(None, None, None, None, None, 0, 4, 64, 64, None)  # n = 0: nothing to do


def test_layer_with_float64_combine(oracle_lib):
    """The layer under MOE_COMBINE_F64_TREE: within the oracle bound, chunk-invariant, decode rows equal."""
    from expert_major_chunked_gb300 import binding
    wl, inp = cpu_inputs("e128_t3001")
    g = GpuLayer(inp, wl.top_k, max_chunk=max(wl.chunks))
    g.layer.set_combine(binding.COMBINE_F64_TREE)
    runs = {c: g.run(c) for c in wl.chunks}
    first = runs[wl.chunks[0]]
    for c in wl.chunks[1:]:
        np.testing.assert_array_equal(out_bits(runs[c]["out"]), out_bits(first["out"]))
    sample = sample_tokens(wl.tokens, wl.chunks, extra=48)
    _, ref_bf, ref_ids, _ = oracle_lib.moe_forward(inp, wl.top_k, token_idx=sample)
    np.testing.assert_array_equal(first["ids"][sample], ref_ids)
    max_abs, rel = compare_out(first["out"][sample], ref_bf, oracle_lib)
    assert max_abs <= MAX_ABS and rel <= REL_L2
    x = g.dev["x"]
    for t in (0, 1234, wl.tokens - 1):
        row = g.run(1, x=x[t:t + 1].contiguous())["out"]
        np.testing.assert_array_equal(out_bits(row)[0], out_bits(first["out"])[t])
    g.layer.set_combine(binding.COMBINE_F32)
    f32_run = g.run(wl.chunks[0])
    assert (out_bits(f32_run["out"]) != out_bits(first["out"])).mean() < 0.01  # another order, same values


def test_split_on_the_layers_routing(oracle_lib):
    """The layer's own routing (ids in ascending order, softmax weights, member-list rows) with random y: the
    two-part split of the pages equals the unsplit kernel and the oracle."""
    from expert_major_chunked_gb300 import binding
    wl, inp = cpu_inputs("tiny")
    g = GpuLayer(inp, wl.top_k, max_chunk=wl.tokens)
    g.layer.set_combine(binding.COMBINE_F64_TREE)
    res = g.run(wl.tokens)
    E, H = inp["w_router"].shape
    ids = res["ids"]
    _, _, token_row = oracle_lib.permutation(ids, E, wl.tokens)
    rng = np.random.default_rng(3)
    y = rng.standard_normal((ids.size, H)).astype(np.float32)
    s = rng.standard_normal((wl.tokens, H)).astype(np.float32)
    whole_f32, whole_bf = _gpu_whole(y, res["w"], token_row, ids, s, E)
    _, f32s, bfs = _gpu_split(y, res["w"], token_row, ids, s, E, 2)
    np.testing.assert_array_equal(_bits(f32s), _bits(whole_f32))
    np.testing.assert_array_equal(bfs, whole_bf)
    ref_f32, ref_bf = oracle_lib.combine_tree_f64(y, res["w"], token_row, ids, E, s)
    np.testing.assert_array_equal(_bits(whole_f32), _bits(ref_f32))
    np.testing.assert_array_equal(whole_bf, ref_bf)
