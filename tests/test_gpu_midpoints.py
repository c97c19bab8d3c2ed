"""Ties in the two BF16 roundings of the layer, on the GPU: inputs whose float32 results land exactly halfway
between two bf16 values, so that only the ties-to-even rule decides the stored bits.

The reading of every BF16 store of the layer is round to nearest, ties to even (the oracle's bf16 rounding is pinned
to closed-form midpoint cases on the CPU). The combine kernel (the layer's output rounding) and the SwiGLU epilogue of
the gate/up GEMM (the rounding of h) must make the same choice as the oracle on every tie.
"""

import numpy as np
import pytest

import parity_checks as pc

pytestmark = pytest.mark.gpu


def test_combine_rounds_ties_to_even(oracle_lib):
    y, w, tr, s = pc.combine_midpoint_inputs()
    pc.check_combine_bits(pc.gpu_combine(y, w, tr, s), y, w, tr, s, oracle_lib)


def test_swiglu_epilogue_rounds_ties_to_even(oracle_lib):
    a, b = pc.swiglu_midpoint_inputs()
    pc.check_swiglu_bits(pc.gpu_swiglu(a, b), a, b, oracle_lib)


def test_midpoint_fixtures_are_ties(oracle_lib):
    """Every constructed value is exactly a bf16 midpoint (so the two tests above test the tie rule)."""
    y, w, tr, s = pc.combine_midpoint_inputs()
    acc = s.astype(np.float64) + sum(w[:, j:j + 1].astype(np.float64) * y[tr[:, j]].astype(np.float64)
                                     for j in range(w.shape[1]))
    a, b = pc.swiglu_midpoint_inputs()
    n = b.shape[0] // 2
    af, bf = a.double().numpy(), b.double().numpy()
    h = (af @ bf[:n].T) * (af @ bf[n:].T)
    for v in (acc.ravel(), h.ravel()):
        m, e = np.frexp(np.abs(v))               # |v| = m 2^e, m in [0.5, 1)
        q = m * 2.0 ** 9                          # 9 significant bits: the bf16 grid has 8
        assert np.all(q == np.floor(q)) and np.all(np.floor(q) % 2 == 1)
