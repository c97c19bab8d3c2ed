"""Pins of the float64 oracle to things other than itself (CPU only).

Each test checks the oracle against a closed form, a hand-worked instance, an invariant, a library routine or a
brute-force evaluation, chosen so that a plausible slip (a dropped term, a swapped gate/up half, a transposed
matrix, a wrong tie-break or sort key, double rounding) fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

from conftest import bf16_bits, read_fixture


# ---------------------------------------------------------------- bf16 rounding (every BF16 store of the layer)

def _bf16_neighbours(b):
    """(value, next value up) for a positive bf16 bit pattern, as float64."""
    lo = np.array([b], dtype=np.uint32) << 16
    hi = np.array([b + 1], dtype=np.uint32) << 16
    return float(lo.view(np.float32)[0]), float(hi.view(np.float32)[0])


def test_bf16_rounding_midpoints_closed_form(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(1)
    for b in list(rng.integers(0x0080, 0x7F00, size=400)) + [0x3F80, 0x3F81, 0x4000, 0x0080]:
        b = int(b)
        lo, hi = _bf16_neighbours(b)
        mid = (lo + hi) / 2  # exact in double
        even = b if b % 2 == 0 else b + 1
        tiny = (hi - lo) * 2.0 ** -30
        got = o.bf16_from_double([mid, mid + tiny, mid - tiny, lo, -mid, -(mid + tiny)])
        assert got[0] == even, "exact midpoint must round to the even neighbour"
        assert got[1] == b + 1
        assert got[2] == b
        assert got[3] == b
        assert got[4] == (even | 0x8000)
        assert got[5] == ((b + 1) | 0x8000)


def test_bf16_rounding_single_step_not_via_float(oracle_lib):
    # A double just above a bf16 midpoint whose float rounding lands exactly on the midpoint: rounding through
    # float (twice) would give the even neighbour; one correct rounding gives the upper one.
    lo, hi = _bf16_neighbours(0x3F80)  # 1.0 and 1.0078125
    mid = (lo + hi) / 2
    v = mid + 2.0 ** -40  # rounds to `mid` in float32
    assert float(np.float32(v)) == mid
    assert oracle_lib.bf16_from_double([v])[0] == 0x3F81


def test_bf16_rounding_matches_library_on_float32_values(oracle_lib):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_lib.bf16_from_double(v.astype(np.float64))
    np.testing.assert_array_equal(got, lib)


def test_bf16_special_values(oracle_lib):
    got = oracle_lib.bf16_from_double([0.0, -0.0, np.inf, -np.inf, 3.5e38, 2.0 ** -133, 2.0 ** -134 * 3])
    assert list(got[:5]) == [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7F80]
    assert got[5] == 0x0001            # smallest bf16 subnormal
    assert got[6] == 0x0002            # 1.5 * 2^-133 is a tie between 1 and 2 quanta: even -> 2
    back = oracle_lib.bf16_to_double(np.array([0x3F80, 0xC040, 0x0001], dtype=np.uint16))
    assert list(back) == [1.0, -3.0, 2.0 ** -133]


# ---------------------------------------------------------------- router logits

def _rand_bf16(rng, shape, std):
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)


def _as_f64(t):
    return t.to(torch.float64).numpy()


def test_router_logits_match_library_matmul(oracle_lib):
    rng = np.random.default_rng(3)
    x, wr = _rand_bf16(rng, (37, 320), 1.0), _rand_bf16(rng, (24, 320), 0.05)
    got = oracle_lib.router_logits(x, wr)
    ref = _as_f64(x) @ _as_f64(wr).T
    scale = np.abs(_as_f64(x)) @ np.abs(_as_f64(wr)).T
    assert np.all(np.abs(got - ref) <= 1e-13 * scale + 1e-300)
    # a transposed weight matrix would not even match in shape
    assert got.shape == (37, 24)


def test_router_logits_exact_on_integer_inputs(oracle_lib):
    rng = np.random.default_rng(4)
    xi = rng.integers(-8, 9, (9, 64)).astype(np.float32)
    wi = rng.integers(-8, 9, (5, 64)).astype(np.float32)
    got = oracle_lib.router_logits(bf16_bits(xi), bf16_bits(wi))
    np.testing.assert_array_equal(got, xi.astype(np.int64) @ wi.astype(np.int64).T)


# ---------------------------------------------------------------- top-k and weights

def test_topk_invariants(oracle_lib):
    rng = np.random.default_rng(5)
    T, E, k = 300, 40, 6
    l = rng.standard_normal((T, E))
    ids, w = oracle_lib.topk(l, k)
    for t in range(T):
        assert len(set(ids[t])) == k and list(ids[t]) == sorted(ids[t])
        sel = l[t, ids[t]]
        rest = np.delete(l[t], ids[t])
        assert sel.min() > rest.max()
        np.testing.assert_allclose(w[t], softmax(sel), rtol=1e-14, atol=0)
    assert abs(np.sum(w, axis=1) - 1).max() < 1e-15 * 8
    counts = np.bincount(ids.ravel(), minlength=E)
    assert counts.sum() == T * k


def test_topk_matches_stable_library_sort(oracle_lib):
    rng = np.random.default_rng(6)
    # Coarse logits (multiples of 1/4) give many exact ties.
    l = np.round(rng.standard_normal((500, 16)) * 4) / 4
    ids, _ = oracle_lib.topk(l, 5)
    ref = np.sort(np.argsort(-l, axis=1, kind="stable")[:, :5], axis=1)
    np.testing.assert_array_equal(ids, ref)


def test_topk_planted_tie_goes_to_lower_id(oracle_lib):
    l = np.array([[0.5, 2.0, 1.0, 2.0, 1.0, 1.0]])
    ids, w = oracle_lib.topk(l, 3)
    assert list(ids[0]) == [1, 2, 3]
    np.testing.assert_allclose(w[0], softmax([2.0, 1.0, 2.0]), rtol=1e-15)


def test_topk_k_equals_E_is_full_softmax(oracle_lib):
    rng = np.random.default_rng(7)
    l = rng.standard_normal((20, 12)) * 3
    ids, w = oracle_lib.topk(l, 12)
    assert np.all(ids == np.arange(12))
    np.testing.assert_allclose(w, softmax(l, axis=1), rtol=1e-14)


# ---------------------------------------------------------------- SwiGLU expert

def _bf16_round_torch(v64):
    """Library BF16 rounding (through float32). Asserts that no value sits so close to a bf16 midpoint that the
    float32 step could change the result, so it equals one correct rounding of the float64 value."""
    v64 = np.asarray(v64, dtype=np.float64)
    inexact = v64[(v64 != 0) & (v64.astype(np.float32).astype(np.float64) != v64)]  # exact float32: one rounding
    a = np.abs(inexact)
    e = np.floor(np.log2(a)) + 1
    frac = a / 2.0 ** (e - 8)
    assert np.all(np.abs(frac - np.floor(frac) - 0.5) > 2.0 ** -14), "value too close to a bf16 midpoint"
    return torch.from_numpy(v64.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_swiglu_matches_textbook_numpy(oracle_lib):
    rng = np.random.default_rng(8)
    H, I = 96, 40
    x = _rand_bf16(rng, (H,), 1.0)
    wgu = _rand_bf16(rng, (2 * I, H), 0.1)
    wd = _rand_bf16(rng, (H, I), 0.1)
    y, h_bits = oracle_lib.swiglu_ffn(x, wgu, wd)
    X, G, U, D = _as_f64(x), _as_f64(wgu[:I]), _as_f64(wgu[I:]), _as_f64(wd)
    g, u = G @ X, U @ X
    h_exact = g / (1 + np.exp(-g)) * u
    h = oracle_lib.bf16_to_double(h_bits)
    # RNE: |round(v) - v| <= half the bf16 spacing at v (2^-8 relative at most)
    assert np.all(np.abs(h - h_exact) <= np.abs(h_exact) * 2.0 ** -8 + 1e-300)
    np.testing.assert_allclose(h, _bf16_round_torch(h_exact), rtol=0, atol=0)
    np.testing.assert_allclose(y, D @ h, rtol=1e-13, atol=1e-15)
    # swapping the gate and up halves changes the result: the pin distinguishes the two orders
    h_swapped = u / (1 + np.exp(-u)) * g
    assert not np.allclose(h_swapped, h_exact)


def test_single_expert_layer_is_textbook_ffn(oracle_lib):
    rng = np.random.default_rng(9)
    H, I, T = 64, 32, 11
    inp = {"x": _rand_bf16(rng, (T, H), 1.0), "w_router": _rand_bf16(rng, (1, H), 0.1),
           "w_gu": _rand_bf16(rng, (1, 2 * I, H), 0.1), "w_down": _rand_bf16(rng, (1, H, I), 0.1)}
    out_ref, out_bf, ids, w = oracle_lib.moe_forward(inp, top_k=1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    X = _as_f64(inp["x"])
    G, U, D = _as_f64(inp["w_gu"][0, :I]), _as_f64(inp["w_gu"][0, I:]), _as_f64(inp["w_down"][0])
    g, u = X @ G.T, X @ U.T
    h = _bf16_round_torch(g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(out_ref, h @ D.T, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- whole layer

def _dense_masked_numpy(inp, k, oracle_round):
    """Brute force: every expert evaluated on every token; unselected experts get weight 0."""
    X = _as_f64(inp["x"])
    Wr = _as_f64(inp["w_router"])
    E = Wr.shape[0]
    I = inp["w_gu"].shape[1] // 2
    l = X @ Wr.T
    order = np.argsort(-l, axis=1, kind="stable")
    mask = np.zeros_like(l, dtype=bool)
    np.put_along_axis(mask, order[:, :k], True, axis=1)
    lsel = np.where(mask, l, -np.inf)
    wfull = np.exp(lsel - lsel.max(axis=1, keepdims=True))
    wfull /= wfull.sum(axis=1, keepdims=True)
    acc = np.zeros((X.shape[0], X.shape[1]))
    for e in range(E):
        G, U, D = _as_f64(inp["w_gu"][e, :I]), _as_f64(inp["w_gu"][e, I:]), _as_f64(inp["w_down"][e])
        g, u = X @ G.T, X @ U.T
        h = oracle_round(g / (1 + np.exp(-g)) * u)
        acc += wfull[:, e:e + 1] * (h @ D.T)
    if inp.get("ws_gu") is not None:
        Is = inp["ws_gu"].shape[0] // 2
        G, U, D = _as_f64(inp["ws_gu"][:Is]), _as_f64(inp["ws_gu"][Is:]), _as_f64(inp["ws_down"])
        g, u = X @ G.T, X @ U.T
        acc += oracle_round(g / (1 + np.exp(-g)) * u) @ D.T
    return acc, np.sort(order[:, :k], axis=1), l


def _tiny_inputs(rng, T=23, H=64, E=8, I=32, Is=16):
    return {"x": _rand_bf16(rng, (T, H), 1.0), "w_router": _rand_bf16(rng, (E, H), 0.3),
            "w_gu": _rand_bf16(rng, (E, 2 * I, H), 0.1), "w_down": _rand_bf16(rng, (E, H, I), 0.1),
            "ws_gu": _rand_bf16(rng, (2 * Is, H), 0.1), "ws_down": _rand_bf16(rng, (H, Is), 0.1)}


def test_layer_matches_dense_masked_brute_force(oracle_lib):
    rng = np.random.default_rng(10)
    inp = _tiny_inputs(rng)
    k = 3
    rnd = lambda v: oracle_lib.bf16_to_double(oracle_lib.bf16_from_double(v))
    dense, ids_dense, l = _dense_masked_numpy(inp, k, rnd)
    # the numpy logits differ from the oracle's sequential sums in the last bits: make sure no selection is that close
    srt = np.sort(l, axis=1)[:, ::-1]
    assert np.min(srt[:, k - 1] - srt[:, k]) > 1e-9
    out_ref, out_bf, ids, w = oracle_lib.moe_forward(inp, top_k=k)
    np.testing.assert_array_equal(ids, ids_dense)
    np.testing.assert_allclose(out_ref, dense, rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(out_bf, oracle_lib.bf16_from_double(out_ref))


def test_layer_hand_worked_example(oracle_lib):
    fx = read_fixture("hand_worked_layer.txt")
    H, E, I, k, Is = (int(v) for v in fx["dims"])
    inp = {"x": bf16_bits(np.reshape(fx["x"], (2, H))),
           "w_router": bf16_bits(np.reshape(fx["w_router"], (E, H))),
           "w_gu": bf16_bits(np.reshape(fx["w_gu"], (E, 2 * I, H))),
           "w_down": bf16_bits(np.reshape(fx["w_down"], (E, H, I))),
           "ws_gu": bf16_bits(np.reshape(fx["ws_gu"], (2 * Is, H))),
           "ws_down": bf16_bits(np.reshape(fx["ws_down"], (H, Is)))}
    out_ref, out_bf, ids, w = oracle_lib.moe_forward(inp, top_k=k)
    np.testing.assert_array_equal(ids.ravel(), np.array(fx["topk_id"], dtype=np.int32))
    a, b = 1 / (1 + math.e), math.e / (1 + math.e)
    np.testing.assert_allclose(w, [[a, b], [a, b]], rtol=1e-15)
    for t, o, ca, cb, c0 in fx["closed"]:
        assert out_ref[int(t), int(o)] == pytest.approx(ca * a + cb * b + c0, rel=1e-15, abs=1e-16)
    np.testing.assert_array_equal(out_bf.ravel(), bf16_bits(fx["out_bf16"]))
    _, h1 = oracle_lib.swiglu_ffn(inp["x"][0], inp["w_gu"][1], inp["w_down"][1])
    assert oracle_lib.bf16_to_double(h1)[0] == fx["h_e1_t0"][0]


def test_layer_token_subset_equals_full(oracle_lib):
    rng = np.random.default_rng(11)
    inp = _tiny_inputs(rng, T=17)
    full = oracle_lib.moe_forward(inp, top_k=2)
    idx = [16, 3, 3, 0]
    sub = oracle_lib.moe_forward(inp, top_k=2, token_idx=idx)
    for a, b in zip(full, sub):
        np.testing.assert_array_equal(a[idx], b)


def test_layer_zero_routed_down_gives_shared_only(oracle_lib):
    rng = np.random.default_rng(12)
    inp = _tiny_inputs(rng, T=9)
    inp["w_down"] = torch.zeros_like(inp["w_down"])
    out_ref, _, _, _ = oracle_lib.moe_forward(inp, top_k=2)
    X = _as_f64(inp["x"])
    Is = inp["ws_gu"].shape[0] // 2
    ys = np.stack([oracle_lib.swiglu_ffn(inp["x"][t], inp["ws_gu"], inp["ws_down"])[0] for t in range(X.shape[0])])
    np.testing.assert_array_equal(out_ref, ys)


def test_layer_identical_experts_weights_sum_to_one(oracle_lib):
    rng = np.random.default_rng(13)
    inp = _tiny_inputs(rng, T=7)
    inp["w_gu"] = inp["w_gu"][:1].repeat(inp["w_gu"].shape[0], 1, 1)
    inp["w_down"] = inp["w_down"][:1].repeat(inp["w_down"].shape[0], 1, 1)
    del inp["ws_gu"], inp["ws_down"]
    out_ref, _, _, _ = oracle_lib.moe_forward(inp, top_k=4)
    y0 = np.stack([oracle_lib.swiglu_ffn(inp["x"][t], inp["w_gu"][0], inp["w_down"][0])[0] for t in range(7)])
    np.testing.assert_allclose(out_ref, y0, rtol=1e-14, atol=1e-16)


# ---------------------------------------------------------------- member lists

def test_permutation_hand_worked_example(oracle_lib):
    fx = read_fixture("hand_worked_permutation.txt")
    T, k, E, chunk = (int(v) for v in fx["dims"])
    ids = np.array(fx["topk_id"], dtype=np.int32).reshape(T, k)
    offs, row_token, token_row = oracle_lib.permutation(ids, E, chunk)
    np.testing.assert_array_equal(offs.ravel(), np.array(fx["expert_offsets"], dtype=np.int32))
    np.testing.assert_array_equal(row_token, np.array(fx["row_token"], dtype=np.int32))
    np.testing.assert_array_equal(token_row.ravel(), np.array(fx["token_row"], dtype=np.int32))


@pytest.mark.parametrize("chunk", [1, 7, 64, 1000])
def test_permutation_is_stable_sort_per_chunk(oracle_lib, chunk):
    rng = np.random.default_rng(14)
    T, E, k = 301, 24, 4
    ids = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    offs, row_token, token_row = oracle_lib.permutation(ids, E, chunk)
    for c in range((T + chunk - 1) // chunk):
        t0, t1 = c * chunk, min((c + 1) * chunk, T)
        flat = ids[t0:t1].ravel()
        order = np.argsort(flat, kind="stable")
        np.testing.assert_array_equal(row_token[t0 * k: t1 * k], t0 + order // k)
        np.testing.assert_array_equal(offs[c], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        rows = token_row[t0:t1].ravel()
        assert sorted(rows) == list(range((t1 - t0) * k))        # a bijection onto the chunk's rows
        np.testing.assert_array_equal(np.argsort(rows), order)


# ---------------------------------------------------------------- combine

def test_combine_f32_canonical_exact_cases(oracle_lib):
    rng = np.random.default_rng(15)
    n, k, H = 50, 4, 33
    y = rng.integers(-64, 65, (n * k, H)).astype(np.float32)
    w = (2.0 ** rng.integers(-3, 2, (n, k))).astype(np.float32)
    s = rng.integers(-64, 65, (n, H)).astype(np.float32)
    tr = rng.permutation(n * k).reshape(n, k).astype(np.int32)
    out = oracle_lib.combine_f32_canonical(y, w, tr, s)
    exact = np.einsum("nk,nkh->nh", w.astype(np.float64), y[tr].astype(np.float64)) + s
    np.testing.assert_array_equal(oracle_lib.bf16_to_double(out), _bf16_round_torch(exact))
    ref, out64 = oracle_lib.combine_f64(y, w, tr, s)
    np.testing.assert_array_equal(ref, exact)
    np.testing.assert_array_equal(out64, out)


def test_combine_f32_canonical_order_and_rounding(oracle_lib):
    # slot order matters in float32: (1e8 + 1) - 1e8 = 0, but (1e8 - 1e8) + 1 = 1
    y = np.array([[1.0e8], [1.0], [-1.0e8]], dtype=np.float32)
    w = np.ones((1, 3), dtype=np.float32)
    tr = np.array([[0, 1, 2]], dtype=np.int32)
    assert oracle_lib.bf16_to_double(oracle_lib.combine_f32_canonical(y, w, tr))[0, 0] == 0.0
    tr_swap = np.array([[0, 2, 1]], dtype=np.int32)
    assert oracle_lib.bf16_to_double(oracle_lib.combine_f32_canonical(y, w, tr_swap))[0, 0] == 1.0
    # the shared term is added last, after the routed sum
    s = np.array([[-1.0e8]], dtype=np.float32)
    y2 = np.array([[1.0e8], [1.0]], dtype=np.float32)
    out = oracle_lib.combine_f32_canonical(y2, np.ones((1, 2), np.float32), np.array([[0, 1]], np.int32), s)
    assert oracle_lib.bf16_to_double(out)[0, 0] == 0.0
    # a float32 result exactly on a bf16 midpoint rounds to even: 1 + 2^-8 -> 1.0 ; 1 + 3*2^-8 -> 1 + 2^-6
    y3 = np.array([[1.0], [2.0 ** -8]], dtype=np.float32)
    o3 = oracle_lib.combine_f32_canonical(y3, np.ones((1, 2), np.float32), np.array([[0, 1]], np.int32))
    assert oracle_lib.bf16_to_double(o3)[0, 0] == 1.0
    y4 = np.array([[1.0], [3 * 2.0 ** -8]], dtype=np.float32)
    o4 = oracle_lib.combine_f32_canonical(y4, np.ones((1, 2), np.float32), np.array([[0, 1]], np.int32))
    assert oracle_lib.bf16_to_double(o4)[0, 0] == 1.0 + 2.0 ** -6


def test_combine_f64_matches_library(oracle_lib):
    rng = np.random.default_rng(16)
    n, k, H = 40, 5, 24
    y = rng.standard_normal((n * k, H)).astype(np.float32)
    w = rng.random((n, k)).astype(np.float32)
    s = rng.standard_normal((n, H)).astype(np.float32)
    tr = rng.permutation(n * k).reshape(n, k).astype(np.int32)
    ref, _ = oracle_lib.combine_f64(y, w, tr, s)
    exact = np.einsum("nk,nkh->nh", w.astype(np.float64), y[tr].astype(np.float64)) + s
    np.testing.assert_allclose(ref, exact, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- float64 tree combine (expert-parallel partials)

def _tree_fixture():
    fx = read_fixture("hand_worked_tree_combine.txt")
    n, k, E, H = (int(v) for v in fx["dims"])
    f = lambda key, dt: np.array(fx[key], dtype=dt)
    return (n, k, E, H, f("y", np.float32).reshape(n * k, H), f("w", np.float32).reshape(n, k),
            f("token_row", np.int32).reshape(n, k), f("topk_id", np.int32).reshape(n, k),
            f("s", np.float32).reshape(n, H), fx)


def _same_bits(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b, dtype=a.dtype)
    np.testing.assert_array_equal(a.view(np.uint64 if a.itemsize == 8 else np.uint32),
                                  b.view(np.uint64 if b.itemsize == 8 else np.uint32))


def test_tree_combine_hand_worked_example(oracle_lib):
    n, k, E, H, y, w, tr, ids, s, fx = _tree_fixture()
    for part in (0, 1):
        got = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E, n_parts=2, part=part)
        _same_bits(got, np.array(fx[f"part{part}"], dtype=np.float64).reshape(n, H))  # signed zeros included
    whole = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E)
    f32, bf = oracle_lib.combine_tree_finish_f64([whole])
    _same_bits(f32, np.array(fx["out_f32_no_shared"], dtype=np.float32).reshape(n, H))
    np.testing.assert_array_equal(bf, np.array(fx["out_bf16_no_shared"], dtype=np.uint16).reshape(n, H))
    for parts in (1, 2, 4):
        pieces = [oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E, parts, p) for p in range(parts)]
        f32, bf = oracle_lib.combine_tree_finish_f64(pieces, s)
        _same_bits(f32, np.array(fx["out_f32"], dtype=np.float32).reshape(n, H))
        np.testing.assert_array_equal(bf, np.array(fx["out_bf16"], dtype=np.uint16).reshape(n, H))
    # the ascending-id float64 sum of the same slots differs in t0 c0: the order is part of the definition
    ref, _ = oracle_lib.combine_f64(y, w, tr)
    assert ref[0, 0] == 0.0 and whole[0, 0] == 1.0


@pytest.mark.parametrize("E,k", [(48, 6), (64, 8), (16, 1)])
def test_tree_combine_exact_integer_sums(oracle_lib, E, k):
    """Integer y and power-of-two weights keep every partial sum exact, so any tree equals the exact sum."""
    rng = np.random.default_rng(21 + E)
    n, H = 37, 12
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(n)]).astype(np.int32)
    w = (2.0 ** rng.integers(-4, 3, size=(n, k))).astype(np.float32)
    y = rng.integers(-2 ** 20, 2 ** 20, size=(n * k, H)).astype(np.float32)
    s = rng.integers(-2 ** 20, 2 ** 20, size=(n, H)).astype(np.float32)
    tr = rng.permutation(n * k).reshape(n, k).astype(np.int32)
    exact = [[sum(int(y[tr[t, j], o]) * float(w[t, j]) for j in range(k)) for o in range(H)] for t in range(n)]
    whole = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E)
    np.testing.assert_array_equal(whole, np.array(exact))
    f32, bf = oracle_lib.combine_tree_finish_f64([whole], s)
    np.testing.assert_array_equal(f32.astype(np.float64), (np.array(exact) + s).astype(np.float32))
    np.testing.assert_array_equal(oracle_lib.bf16_to_double(bf), _bf16_round_torch(f32.astype(np.float64)))
    Ep = 1 << (E - 1).bit_length()
    for parts in (2, Ep):
        lo = [p * Ep // parts for p in range(parts)]
        for p in range(parts):
            got = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E, parts, p)
            inside = (ids >= lo[p]) & (ids < lo[p] + Ep // parts)
            want = np.einsum("nk,nkh->nh", np.where(inside, w, 0).astype(np.float64), y[tr].astype(np.float64))
            np.testing.assert_array_equal(got, want)


def test_tree_combine_split_reproduces_whole(oracle_lib):
    rng = np.random.default_rng(22)
    n, k, E, H = 29, 8, 96, 20
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(n)]).astype(np.int32)
    w = rng.random((n, k)).astype(np.float32)
    y = (rng.standard_normal((n * k, H)) * 10.0 ** rng.integers(-6, 7, size=(n * k, H))).astype(np.float32)
    s = rng.standard_normal((n, H)).astype(np.float32)
    tr = rng.permutation(n * k).reshape(n, k).astype(np.int32)
    f_whole, b_whole = oracle_lib.combine_tree_f64(y, w, tr, ids, E, s)
    for parts in (2, 4, 8, 32, 128):
        pieces = [oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E, parts, p) for p in range(parts)]
        f32, bf = oracle_lib.combine_tree_finish_f64(pieces, s)
        _same_bits(f32, f_whole)
        np.testing.assert_array_equal(bf, b_whole)
    # within the float64 error bound of the exact sum (math.fsum), then one float32 rounding
    whole = oracle_lib.combine_tree_partial_f64(y, w, tr, ids, E)
    depth = 7  # log2(128)
    for t in range(n):
        for o in range(H):
            terms = [float(w[t, j]) * float(y[tr[t, j], o]) for j in range(k)]
            bound = depth * 2.0 ** -53 * sum(abs(v) for v in terms)
            assert abs(whole[t, o] - math.fsum(terms)) <= bound


def test_tree_combine_rejects_bad_arguments(oracle_lib):
    y = np.ones((4, 2), np.float32)
    w = np.ones((2, 2), np.float32)
    tr = np.array([[0, 1], [2, 3]], np.int32)
    with pytest.raises(ValueError):
        oracle_lib.combine_tree_partial_f64(y, w, tr, np.array([[1, 1], [0, 2]], np.int32), 4)   # repeated id
    with pytest.raises(ValueError):
        oracle_lib.combine_tree_partial_f64(y, w, tr, np.array([[0, 4], [1, 2]], np.int32), 4)   # id >= E
    with pytest.raises(ValueError):
        oracle_lib.combine_tree_partial_f64(y, w, tr, np.array([[0, 1], [1, 2]], np.int32), 4, 3, 0)  # 3 parts


# ---------------------------------------------------------------- MXFP8 weights (E4M3 codes, E8M0 block scales)

def _fixture_lines(name):
    import os
    from conftest import GOLDEN
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split()[1:])
    return rows


def test_mxfp8_hand_worked_codes(oracle_lib):
    for code, scale, value in _fixture_lines("e4m3_codes.txt"):
        codes = np.zeros((1, 1, 32), np.uint8)
        codes[0, 0, 5] = int(code)
        scales = np.full((1, 1, 1), int(scale), np.uint8)
        got = float(oracle_lib.bf16_to_double(oracle_lib.dequant_mxfp8(codes, scales)[0, 0, 5:6])[0])
        want = float(value)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, scale, got, want)


def test_mxfp8_matches_library_decoding(oracle_lib):
    """Every non-NaN code against torch's float8_e4m3fn decoding, times 2^(s-127) for scales across the range."""
    rng = np.random.default_rng(31)
    codes_all = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    R, K = 8, 256
    codes = rng.choice(codes_all, size=(2, R, K)).astype(np.uint8)
    codes[0, 0, :len(codes_all)] = codes_all
    scales = rng.integers(10, 247, size=(2, K // 32, R)).astype(np.uint8)
    got = oracle_lib.bf16_to_double(oracle_lib.dequant_mxfp8(codes, scales))
    lib_vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s_full = np.repeat(scales.transpose(0, 2, 1), 32, axis=2).astype(np.int64)  # [E][R][K]
    want = np.ldexp(lib_vals, s_full - 127)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(want))


def test_mxfp8_rejects_nan_and_unrepresentable(oracle_lib):
    base = np.zeros((1, 2, 32), np.uint8)
    ok = np.full((1, 1, 2), 127, np.uint8)
    oracle_lib.dequant_mxfp8(base, ok)
    for code in (0x7F, 0xFF):
        bad = base.copy()
        bad[0, 1, 3] = code
        with pytest.raises(ValueError):
            oracle_lib.dequant_mxfp8(bad, ok)
    with pytest.raises(ValueError):
        oracle_lib.dequant_mxfp8(base, np.full((1, 1, 2), 255, np.uint8))
    tiny = base.copy()
    tiny[0, 0, 0] = 0x01
    with pytest.raises(ValueError):  # 2^-9 * 2^-127 is below every bf16 value
        oracle_lib.dequant_mxfp8(tiny, np.full((1, 1, 2), 0, np.uint8))


def test_mxfp8_quantizer_round_trip(oracle_lib):
    """The synthetic MXFP8 inputs decode (oracle) to within half an E4M3 step of the drawn weights, and every
    block's largest weight lands in (224, 448] after scaling (the least scale that clips nothing)."""
    from expert_major_chunked_gb300 import workloads
    g = torch.Generator().manual_seed(5)
    w = (torch.randn((3, 16, 128), generator=g) * 0.02).to(torch.bfloat16)
    codes, scales = workloads.quantize_mxfp8(w)
    got = oracle_lib.bf16_to_double(oracle_lib.dequant_mxfp8(codes.numpy(), scales.numpy()))
    ref = w.double().numpy()
    blk_scale = np.repeat(np.ldexp(1.0, scales.numpy().astype(np.int64) - 127).transpose(0, 2, 1), 32, axis=2)
    # E4M3 spacing at magnitude |q| = |w| / scale is 2^(floor(log2|q|) - 3) (normal) or 2^-9 (subnormal)
    q = np.abs(ref) / blk_scale
    step = np.where(q >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(got - ref) <= 0.5 * step * blk_scale + 1e-30)
    amax = np.abs(ref).reshape(3, 16, 4, 32).max(axis=3)
    qmax = amax / np.ldexp(1.0, scales.numpy().astype(np.int64).transpose(0, 2, 1) - 127)
    assert np.all((qmax > 224) & (qmax <= 448))


# ---------------------------------------------------------------- NVFP4 weights (E2M1 codes, E4M3 block scales)

def test_nvfp4_hand_worked_codes(oracle_lib):
    table = {int(c): float(v) for c, v in _fixture_lines("e2m1_codes.txt")}
    assert len(table) == 16
    for lo in range(16):
        hi = 15 - lo
        codes = np.zeros((1, 1, 8), np.uint8)
        codes[0, 0, 3] = lo | (hi << 4)  # elements 6 (low nibble) and 7 (high nibble)
        scales = np.full((1, 1, 1), 0x38, np.uint8)  # E4M3 1.0
        got = oracle_lib.bf16_to_double(oracle_lib.dequant_nvfp4(codes, scales)[0, 0, 6:8])
        for g, want in zip(got, (table[lo], table[hi])):
            assert g == want and math.copysign(1, g) == math.copysign(1, want), (lo, hi, got)


def test_nvfp4_matches_library_scale_decoding(oracle_lib):
    """Every code with E4M3 scales across the format (subnormal to 448, either sign), against the hand table times
    torch's float8_e4m3fn decoding of the scale; every product is exact in bf16."""
    table = np.array([float(v) for _, v in _fixture_lines("e2m1_codes.txt")])
    rng = np.random.default_rng(41)
    R, K = 6, 512
    codes = rng.integers(0, 256, size=(2, R, K // 2)).astype(np.uint8)
    scale_codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    scales = rng.choice(scale_codes, size=(2, K // 16, R)).astype(np.uint8)
    scales[0, :, 0] = scale_codes[:K // 16]
    got = oracle_lib.bf16_to_double(oracle_lib.dequant_nvfp4(codes, scales))
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(2, R, K)
    s_val = torch.from_numpy(scales).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    want = table[nib] * np.repeat(s_val.transpose(0, 2, 1), 16, axis=2)
    np.testing.assert_array_equal(got, want)


def test_nvfp4_rejects_nan_scale(oracle_lib):
    codes = np.zeros((1, 2, 8), np.uint8)
    with pytest.raises(ValueError):
        oracle_lib.dequant_nvfp4(codes, np.full((1, 1, 2), 0x7F, np.uint8))


def test_nvfp4_quantizer_round_trip(oracle_lib):
    """The synthetic NVFP4 inputs decode (oracle) to the nearest E2M1 multiple of the block scale (ties even), and
    every block's scale is the least E4M3 value >= max |w| / 6."""
    from expert_major_chunked_gb300 import workloads
    g = torch.Generator().manual_seed(6)
    w = (torch.randn((2, 8, 64), generator=g) * 0.02).to(torch.bfloat16)
    codes, scales = workloads.quantize_nvfp4(w)
    got = oracle_lib.bf16_to_double(oracle_lib.dequant_nvfp4(codes.numpy(), scales.numpy()))
    ref = w.double().numpy()
    s = torch.from_numpy(scales.numpy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()  # [E][K/16][R]
    s_full = np.repeat(s.transpose(0, 2, 1), 16, axis=2)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    q = np.abs(ref) / s_full
    nearest = np.min(np.abs(q[..., None] - grid), axis=-1)
    assert np.all(np.abs(np.abs(got) / s_full - q) <= nearest + 1e-12)
    amax = np.abs(ref).reshape(2, 8, 4, 16).max(axis=3).transpose(0, 2, 1)  # [E][K/16][R]
    assert np.all(s * 6.0 >= amax)
    smaller = torch.from_numpy((scales.numpy() - 1).astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    assert np.all((smaller.numpy() * 6.0 < amax) | (scales.numpy() == 0))
