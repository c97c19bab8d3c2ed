"""Planted controls: every GPU-vs-oracle gate goes red when the oracle carries a plausible mistake.

"EXL3 Flash Next: deep prefill (3/8)", *Device results*, reports its controls all red, and "Flash Next EXL3: exact
deep prefill", *Independent numerical-phase audit*, plants controls the same way. The GPU runs only the correct
kernels, once; each gate is then evaluated against the real oracle (green) and against copies of oracle.c, each with
one planted mistake, compiled on the CPU (tests/planted.py): the gate named for the mistake must fail. A mistake that
no gate could see would show up here as a control that stays green.
"""

import numpy as np
import pytest

import parity_checks as pc
import planted
from layer_helpers import GpuLayer

pytestmark = pytest.mark.gpu

K_SMALL, CHUNK = 4, 33


def _small_inputs(seed, T=100, H=128, E=32, I=64, Is=64, router_std=0.3):
    import torch
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"x": r(T, H, std=1.0), "w_router": r(E, H, std=router_std), "w_gu": r(E, 2 * I, H),
            "w_down": r(E, H, I), "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


@pytest.fixture(scope="module")
def gpu():
    """All GPU results the gates need, computed once with the real kernels."""
    res = {}
    inp = _small_inputs(1)
    res["layer"] = (inp, GpuLayer(inp, K_SMALL, max_chunk=CHUNK).run(CHUNK))
    tie = _small_inputs(5)
    wr = tie["w_router"].clone()
    for a, b in ((3, 7), (10, 11), (20, 30), (0, 31)):
        wr[b] = wr[a]                                   # identical router rows: exactly equal logits
    tie["w_router"] = wr
    res["ties"] = (tie, GpuLayer(tie, K_SMALL, max_chunk=CHUNK).run(CHUNK))
    for key, make in (("combine", pc.combine_random_inputs), ("combine_mid", pc.combine_midpoint_inputs)):
        args = make()
        res[key] = (args, pc.gpu_combine(*args))
    a, b = pc.swiglu_midpoint_inputs()
    res["swiglu_mid"] = ((a, b), pc.gpu_swiglu(a, b))
    res["swiglu_mid_pairs"] = ((a, b), pc.gpu_swiglu_pairs(a, b))
    # dimensions where the gate/up projection runs on CTA pairs (the default for them)
    wide = _small_inputs(2, H=256, I=128, Is=128)
    res["layer_pairs"] = (wide, GpuLayer(wide, K_SMALL, max_chunk=CHUNK).run(CHUNK))
    return res


GATES = {
    "routing_ids_planted_ties": lambda g, o: pc.check_routing_ids(g["ties"][1], g["ties"][0], K_SMALL, o),
    "permutation": lambda g, o: pc.check_permutation(g["layer"][1], g["layer"][0], K_SMALL, CHUNK, o),
    "routing_weights": lambda g, o: pc.check_weights(g["layer"][1], g["layer"][0], K_SMALL, o),
    "layer_output": lambda g, o: pc.check_output(g["layer"][1], g["layer"][0], K_SMALL, o),
    "combine_bits": lambda g, o: pc.check_combine_bits(g["combine"][1], *g["combine"][0], o),
    "combine_ties": lambda g, o: pc.check_combine_bits(g["combine_mid"][1], *g["combine_mid"][0], o),
    "swiglu_ties": lambda g, o: pc.check_swiglu_bits(g["swiglu_mid"][1], *g["swiglu_mid"][0], o),
    "swiglu_ties_pairs": lambda g, o: pc.check_swiglu_bits(g["swiglu_mid_pairs"][1], *g["swiglu_mid_pairs"][0], o),
    "layer_output_pairs": lambda g, o: pc.check_output(g["layer_pairs"][1], g["layer_pairs"][0], K_SMALL, o),
}

# planted mistake -> the gates that must go red on it
RED = {
    "combine_descending": ["combine_bits"],
    "shared_added_first": ["combine_bits"],
    "tie_to_higher_id": ["routing_ids_planted_ties"],
    "scan_base_off_by_one": ["permutation"],
    "round_half_away": ["combine_ties", "swiglu_ties", "swiglu_ties_pairs", "combine_bits"],
    "h_not_rounded": ["layer_output", "layer_output_pairs"],
    "gate_up_swapped": ["layer_output", "layer_output_pairs"],
    "no_renormalise": ["routing_weights", "layer_output", "layer_output_pairs"],
    "shared_dropped": ["layer_output", "layer_output_pairs"],
    "silu_sign_flipped": ["layer_output", "layer_output_pairs"],
}


def test_every_planted_mistake_has_a_gate():
    assert set(RED) == set(planted.PLANTED)
    assert all(g in GATES for gates in RED.values() for g in gates)


@pytest.mark.parametrize("gate", sorted(GATES))
def test_gate_green_against_the_oracle(gpu, oracle_lib, gate):
    GATES[gate](gpu, oracle_lib)


@pytest.mark.parametrize("name", sorted(planted.PLANTED))
def test_planted_mistake_turns_its_gate_red(gpu, name):
    with planted.planted_oracle(name) as bad:
        for gate in RED[name]:
            with pytest.raises(AssertionError):
                GATES[gate](gpu, bad)
