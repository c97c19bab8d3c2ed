"""Routing under adversarial router inputs, on the GPU.

The routing kernel trusts the fp32 tensor-core logits of a token when its k-th and (k+1)-th logits are more than
2 tau apart, with tau = (H/16 + 1) 2^-23 ||x|| max_e ||w_e||: a model of the accumulation error (at most one float32
rounding per 16-wide K step of a partial sum bounded by sum |x_i w_i| <= ||x|| ||w||), not a documented bound of the
tensor cores. Every other token is decided in float64 by levels that are rigorous. These inputs are built to push
the model: same-sign products (every partial sum as large as it can be), heavy cancellation (large partial sums, small
logits), a wide exponent spread within bf16, and many experts with logits a few ulps apart (long recheck lists).
Each must give the oracle's routing bit for bit, and the measured logit error must stay below tau.
"""

import numpy as np
import pytest
import torch

from layer_helpers import GpuLayer

pytestmark = pytest.mark.gpu

T, H, E, I, K = 512, 2048, 64, 64, 8


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _case(name, seed=0):
    rng = np.random.default_rng(seed)
    if name == "same_sign":
        x = rng.uniform(0.5, 1.5, (T, H))
        w = rng.uniform(0.5, 1.5, (E, H))
    elif name == "cancellation":
        # the first half of K adds large positive products, the second half takes them away again
        x = rng.uniform(0.5, 1.5, (T, H)) * 2.0 ** 6
        mag = rng.uniform(0.5, 1.5, (E, H // 2))
        w = np.concatenate([mag, -mag[:, rng.permutation(H // 2)]], axis=1)
        w += rng.normal(0, 0.01, (E, H))
    elif name == "exponent_spread":
        x = rng.normal(0, 1, (T, H)) * 2.0 ** rng.integers(-30, 31, (T, H))
        w = rng.normal(0, 1, (E, H)) * 2.0 ** rng.integers(-30, 31, (E, H))
    elif name == "near_equal":
        # 48 of the experts share one router row up to a single bf16 step in one coordinate each
        x = rng.normal(0, 1, (T, H))
        w = rng.normal(0, 0.02, (E, H))
        base = _bf16(rng.normal(0, 0.02, H)).float().numpy().astype(np.float64)
        for e in range(48):
            row = base.copy()
            j = rng.integers(0, H)
            row[j] = np.nextafter(np.float32(row[j]), np.float32(np.inf if e % 2 else -np.inf))
            w[e] = row
    else:
        raise ValueError(name)
    xb, wb = _bf16(x), _bf16(w)
    zeros = lambda *s: torch.zeros(s, dtype=torch.bfloat16)
    # zero expert weights: the layer's outputs stay finite whatever the activations' range; only routing is checked
    return {"x": xb, "w_router": wb, "w_gu": zeros(E, 2 * I, H), "w_down": zeros(E, H, I)}


@pytest.mark.parametrize("name", ["same_sign", "cancellation", "exponent_spread", "near_equal"])
def test_routing_bit_exact_and_error_below_tau(oracle_lib, name):
    from expert_major_chunked_gb300 import binding
    inp = _case(name)
    g = GpuLayer(inp, K, max_chunk=256)
    res = g.run(256)
    logits64 = oracle_lib.router_logits(inp["x"], inp["w_router"])
    ids, _ = oracle_lib.topk(logits64, K)
    np.testing.assert_array_equal(res["ids"], ids)
    offs, row_token, _ = oracle_lib.permutation(ids, E, 256)
    np.testing.assert_array_equal(res["offs"], offs)
    np.testing.assert_array_equal(res["row_token"], row_token)
    stats = g.layer.stats()

    # the fp32 tensor-core logits themselves, through the same GEMM kernel
    logits = torch.empty((T, E), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.moe_prefill_debug_gemm(g.dev["x"].data_ptr(), g.dev["w_router"].data_ptr(), logits.data_ptr(), T, E, H,
                                   0, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    xn = np.linalg.norm(inp["x"].double().numpy(), axis=1)
    wn = np.linalg.norm(inp["w_router"].double().numpy(), axis=1).max()
    ratio = (np.abs(logits.cpu().double().numpy() - logits64) / (xn[:, None] * wn)).max()
    coef = (H // 16 + 1) * 2.0 ** -23
    print(f"\n[{name}] max |fp32 - float64| / (||x|| max||w||) = 2^{np.log2(max(ratio, 1e-300)):.2f}, "
          f"tau coefficient 2^{np.log2(coef):.2f} (margin {coef / max(ratio, 1e-300):.1f}x); "
          f"flagged {stats['flagged']} of {T}, by float {stats['by_float']}, double {stats['by_double']}, "
          f"sequential {stats['by_sequential']}, many {stats['by_many']}")
    assert ratio <= coef / 2, (name, ratio, coef)
