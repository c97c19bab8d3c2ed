"""The planted controls themselves, on the CPU: each copy of oracle.c with its planted mistake compiles, and the
mistake changes the oracle's answer on the inputs of the gate that is meant to catch it (a control that changed
nothing would prove nothing). The GPU side is tests/test_gpu_planted.py."""

import numpy as np
import pytest
import torch

import parity_checks as pc
import planted


def _small(seed, T=60, H=128, E=32, I=64, Is=64):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s, std=0.05: (torch.randn(s, generator=gen) * std).to(torch.bfloat16)
    return {"x": r(T, H, std=1.0), "w_router": r(E, H, std=0.3), "w_gu": r(E, 2 * I, H), "w_down": r(E, H, I),
            "ws_gu": r(2 * Is, H), "ws_down": r(H, Is)}


def _answers(orc):
    inp = _small(1)
    tie = _small(5)
    wr = tie["w_router"].clone()
    for a, b in ((3, 7), (10, 11), (20, 30), (0, 31)):
        wr[b] = wr[a]
    tie["w_router"] = wr
    _, out, ids, w = orc.moe_forward(inp, 4)
    _, _, tie_ids, _ = orc.moe_forward(tie, 4)
    offs, row_token, _ = orc.permutation(ids, 32, 7)
    comb = orc.combine_f32_canonical(*pc.combine_random_inputs(n=64, H=512))
    mid = orc.combine_f32_canonical(*pc.combine_midpoint_inputs(n=32, H=256))
    return {"out": out, "w": w, "tie_ids": tie_ids, "offs": offs, "combine": comb, "combine_mid": mid}


@pytest.mark.parametrize("name", sorted(planted.PLANTED))
def test_planted_copy_builds_and_changes_an_answer(oracle_lib, name):
    good = _answers(oracle_lib)
    with planted.planted_oracle(name) as bad_orc:
        bad = _answers(bad_orc)
    changed = [k for k in good if not np.array_equal(good[k], bad[k])]
    assert changed, f"planted mistake {name!r} changes none of the oracle's answers"


def test_planted_text_must_match_exactly():
    for name in planted.PLANTED:
        src = planted.planted_source(name)
        assert src != open(f"{planted.ORACLE_DIR}/oracle.c").read()
