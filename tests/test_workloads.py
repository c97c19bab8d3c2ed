"""The synthetic inputs follow the recipe stated for each workload (CPU only).

The pages measure on a private checkpoint and private prompts; the workloads stand in for them with the pages'
prompt lengths and the layer sizes of the model family. These tests check the recipe itself: sizes and chunk
lists, the router logit spread each workload states, the Zipf(1.1) expert-popularity prior of the skewed ones
(against a table computed here from its definition), and that the draws are seeded and repeatable.
"""

import math

import numpy as np
import pytest
import torch

from expert_major_chunked_gb300 import workloads as W

# name: (T, H, E, I, k, I_s, chunks, offload slots)
RECIPE = {
    "tiny": (40, 256, 16, 128, 2, 128, (8, 16, 40), 0),
    "e128_t3001": (3001, 2048, 128, 768, 8, 2048, (256, 1024, 2048), 0),
    "e512_zipf_t4099": (4099, 2048, 512, 512, 10, 512, (256, 1024, 2048), 0),
    "e512_t16022": (16022, 2048, 512, 512, 10, 512, (2048,), 0),
    "e512_offload_t12001": (12001, 2048, 512, 512, 10, 512, (1024,), 32),
    "e512_zipf_offload_t12001": (12001, 2048, 512, 512, 10, 512, (1024,), 32),
}


def _light(name, tokens=512):
    """x and W_router of a workload at full H and E (they are drawn first, so smaller expert sizes leave them
    unchanged); the expert weights are shrunk to keep the draw quick."""
    wl = W.WORKLOADS[name]
    return W.generate(wl.with_(inter=64, shared_inter=0), tokens=tokens)


@pytest.mark.parametrize("name", sorted(RECIPE))
def test_sizes_and_chunks(name):
    wl = W.WORKLOADS[name]
    T, H, E, I, k, Is, chunks, slots = RECIPE[name]
    assert (wl.tokens, wl.hidden, wl.n_experts, wl.inter, wl.top_k, wl.shared_inter) == (T, H, E, I, k, Is)
    assert tuple(wl.chunks) == chunks and wl.offload_slots == slots
    assert H % 64 == 0 and I % 64 == 0 and E % 16 == 0 and 1 <= k <= E


def test_tiny_draw_shapes_dtypes_and_repeatability():
    wl = W.WORKLOADS["tiny"]
    a, b = W.generate(wl), W.generate(wl)
    shapes = {"x": (40, 256), "w_router": (16, 256), "w_gu": (16, 256, 256), "w_down": (16, 256, 128),
              "ws_gu": (256, 256), "ws_down": (256, 128)}
    for n, shape in shapes.items():
        assert a[n].dtype == torch.bfloat16 and tuple(a[n].shape) == shape
        assert torch.equal(a[n].view(torch.int16), b[n].view(torch.int16))
    c = W.generate(wl, seed=1)
    assert not torch.equal(a["x"].view(torch.int16), c["x"].view(torch.int16))


@pytest.mark.parametrize("name,std", [("tiny", 1.0), ("e128_t3001", 0.02 * math.sqrt(2048)),
                                      ("e512_t16022", 1.0), ("e512_offload_t12001", 1.0)])
def test_router_logit_spread(name, std):
    """Logits x . W_r^T have the spread the recipe states: N(0, 1) for the tiny and uniform-router workloads,
    0.02 * sqrt(2048) ~ 0.905 for the 3001-token one (router N(0, 0.02^2) on N(0, 1) activations)."""
    inp = _light(name, tokens=40 if name == "tiny" else 512)
    x = inp["x"].double().numpy()
    wr = inp["w_router"].double().numpy()
    logits = x @ wr.T
    assert abs(logits.mean()) < 0.05 * std + 0.02
    assert 0.9 * std < logits.std() < 1.1 * std


@pytest.mark.parametrize("name", ["e512_zipf_t4099", "e512_zipf_offload_t12001"])
def test_zipf_popularity_prior(name):
    """Channel 0 of x is 1.0 and W_router[:, 0] holds log p_r of a Zipf(1.1) law over the 512 ranks, permuted
    over the experts; the other channels give N(0, 1) noise logits."""
    inp = _light(name)
    x = inp["x"].double().numpy()
    wr = inp["w_router"].double().numpy()
    assert np.all(x[:, 0] == 1.0)
    E = wr.shape[0]
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** -1.1 / np.sum(ranks ** -1.1)
    expected = torch.from_numpy(np.log(p)).float().to(torch.bfloat16).double().numpy()
    got = np.sort(wr[:, 0])[::-1]
    np.testing.assert_array_equal(got, np.sort(expected)[::-1])
    assert abs(np.exp(wr[:, 0]).sum() - 1.0) < 1e-2          # a distribution, up to the bf16 rounding of log p
    assert 1.6 < -got[0] < 1.7 and 8.4 < -got[-1] < 8.6      # ln p_1 ~ -1.65, ln p_512 ~ -8.52
    noise = x[:, 1:] @ wr[:, 1:].T
    assert 0.9 < noise.std() < 1.1


def test_draw_x_uses_the_workload_distribution():
    wl = W.WORKLOADS["e512_zipf_t4099"]
    x = W.draw_x(wl, 256, seed=5).double().numpy()
    assert np.all(x[:, 0] == 1.0)
    assert 0.95 < x[:, 1:].std() < 1.05
