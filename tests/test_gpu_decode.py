"""Decode-row equality on the GPU.

The maintainer review of the deep-prefill draft, slice 3 of 7 ("To land"), asks that the prompt kernels produce the
decode kernels' bytes for every row, whatever the chunk or segment length. Here decoding a token is the same layer call
with T = 1 (or a small batch), through the same kernels: every row of a long prefill must equal, byte for byte,
the row obtained by running that token alone or inside any small batch.
"""

import numpy as np
import pytest
import torch

from layer_helpers import GpuLayer, cpu_inputs, out_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,prefill_chunk", [("tiny", 40), ("e512_zipf_t4099", 2048), ("e512_t16022", 2048)])
def test_decode_rows_equal_prefill_rows(name, prefill_chunk):
    wl, inp = cpu_inputs(name)
    g = GpuLayer(inp, wl.top_k, max_chunk=prefill_chunk)
    prefill = out_bits(g.run(prefill_chunk)["out"])
    x = g.dev["x"]
    rng = np.random.default_rng(7)
    singles = sorted(set(rng.choice(wl.tokens, size=min(24, wl.tokens), replace=False).tolist()) | {0, wl.tokens - 1})
    for t in singles:
        row = g.run(1, x=x[t:t + 1].contiguous())["out"]
        np.testing.assert_array_equal(out_bits(row)[0], prefill[t], err_msg=f"{name}: token {t} decoded alone")
    for size in (2, 5, 16, 33):
        idx = torch.tensor(np.sort(rng.choice(wl.tokens, size=min(size, wl.tokens), replace=False)))
        batch = g.run(min(size, prefill_chunk), x=x[idx.cuda()].contiguous())["out"]
        np.testing.assert_array_equal(out_bits(batch), prefill[idx.numpy()],
                                      err_msg=f"{name}: batch of {size} tokens")
