"""The benchmark's byte and FLOP accounting (CPU): the figures behind roofline.achieved and layer_hbm_frac, checked
against the closed forms for the 16,022-token layer (512 experts, H = 2048, I = 512, k = 10, I_s = 512) at
chunk 2048 with every expert touched."""

import numpy as np
import pytest


def _wl():
    from expert_major_chunked_gb300 import workloads
    return workloads.WORKLOADS["e512_t16022"]


def _offs_all_touched(n_chunks, E, rows):
    return np.tile(np.arange(E + 1, dtype=np.int64) * rows, (n_chunks, 1))


def test_gate_up_minimum_and_staged_bytes():
    import bench
    wl = _wl()
    H, I, Is, k, E = wl.hidden, wl.inter, wl.shared_inter, wl.top_k, wl.n_experts
    n = 2048
    offs = _offs_all_touched(1, E, n * k // E)
    b, f = bench.gate_up_bytes_and_flops(wl, offs, [n])
    bs, _ = bench.gate_up_bytes_and_flops(wl, offs, [n], staged_rows=True)
    weights = E * 2 * I * H * 2 + 2 * Is * H * 2
    assert b == weights + n * H * 2 + (n * k * I + n * Is) * 2        # x read once, h written once
    assert bs - b == (n * k + n - n) * H * 2                            # plus the gathered copy of the rows
    assert b == pytest.approx(2.183e9, rel=1e-3)
    assert f == 2.0 * n * k * H * 2 * I + 2.0 * n * H * 2 * Is


def test_layer_weight_bytes_per_step():
    import bench
    wl = _wl()
    chunks = [min(2048, wl.tokens - c0) for c0 in range(0, wl.tokens, 2048)]
    assert len(chunks) == 8
    offs = _offs_all_touched(8, wl.n_experts, 40)
    per_chunk = 6 * wl.inter * wl.hidden * wl.n_experts + 6 * wl.shared_inter * wl.hidden + 2 * wl.n_experts * wl.hidden
    assert bench.layer_weight_bytes(wl, offs) == 8 * per_chunk
    assert 8 * per_chunk == pytest.approx(25.8e9, rel=0.01)
    # an expert with no rows in a chunk is not streamed
    offs[0, 1] = 0      # expert 0 gets no rows in chunk 0 (expert 1 gets its 40)
    assert bench.layer_weight_bytes(wl, offs) == 8 * per_chunk - 6 * wl.inter * wl.hidden
