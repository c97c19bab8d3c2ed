"""The CTA-pair GEMM kernel on its own, through moe_prefill_debug_gemm_pairs (GPU).

Exact-integer inputs make every product and partial sum exactly representable in float32, so the result must equal
the integer matmul bit for bit whatever the accumulation order: a wrong descriptor, box, K block, peer half or tile
offset shows up as a mismatch. On float inputs the pair kernel must give the single-CTA kernel's bytes (same K order);
the SwiGLU epilogue must round exact bf16 midpoints to even, as the oracle does. The bounded-wait test makes the load
warps wait on a flag that nothing sets: both CTAs of every pair give up, report the stall site, and the context stays
usable.
"""

import numpy as np
import pytest
import torch

import parity_checks as pc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from expert_major_chunked_gb300 import binding
    binding.lib()
    return binding


def _ints_bf16(gen, shape, lo, hi):
    v = torch.randint(lo, hi, shape, generator=gen, dtype=torch.int32)
    return v.to(torch.bfloat16), v.to(torch.int64)


def _pairs(B, a, b, m, n, k, epi, flag=None, timeout_ns=0, out=None):
    dt = torch.float32 if epi == 0 else torch.bfloat16
    c = out if out is not None else torch.full((m, n), float("nan"), dtype=dt, device="cuda")
    need = B.moe_prefill_debug_gemm_pairs_scratch(m, n, epi)
    scratch = torch.zeros(need // 4 + 4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da, db = a.cuda(), b.cuda()
    B.moe_prefill_debug_gemm_pairs(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, k, epi, scratch.data_ptr(),
                                   scratch.numel() * 4, err.data_ptr(), None if flag is None else flag.data_ptr(),
                                   timeout_ns)
    torch.cuda.synchronize()
    return c, err.item()


def _single(B, a, b, m, n, k, epi):
    dt = torch.float32 if epi == 0 else torch.bfloat16
    c = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da, db = a.cuda(), b.cuda()
    B.moe_prefill_debug_gemm(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, k, epi, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    return c


def _bits(t):
    return t.cpu().contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy()


# token counts: one short tile, exactly 256, 257 (two tiles of 160/97), ragged several-tile cases
@pytest.mark.parametrize("m,n,k", [(1, 256, 128), (31, 256, 128), (77, 512, 256), (256, 256, 128), (257, 256, 256),
                                   (300, 768, 2048), (513, 1024, 256)])
def test_pair_gemm_exact_integers(B, m, n, k):
    gen = torch.Generator().manual_seed(m * 7 + n * 13 + k)
    a, ai = _ints_bf16(gen, (m, k), -3, 4)
    b, bi = _ints_bf16(gen, (n, k), -3, 4)
    ref = (ai @ bi.T).to(torch.float64)
    assert ref.abs().max() < 2 ** 24
    c, err = _pairs(B, a, b, m, n, k, 0)
    assert err == 0
    np.testing.assert_array_equal(c.cpu().to(torch.float64).numpy(), ref.numpy())


@pytest.mark.parametrize("m,n,k", [(200, 256, 2048), (333, 512, 256), (1, 256, 128)])
def test_pair_gemm_float_inputs_equal_single_cta(B, m, n, k):
    gen = torch.Generator().manual_seed(m + n + k)
    a = torch.randn((m, k), generator=gen).to(torch.bfloat16)
    b = (torch.randn((n, k), generator=gen) * 0.02).to(torch.bfloat16)
    c, err = _pairs(B, a, b, m, n, k, 0)
    assert err == 0
    np.testing.assert_array_equal(_bits(c), _bits(_single(B, a, b, m, n, k, 0)))


@pytest.mark.parametrize("m,n,k", [(50, 128, 128), (256, 256, 256), (130, 512, 2048), (1, 768, 128)])
def test_pair_gemm_swiglu_equal_single_cta_and_near_oracle(B, oracle_lib, m, n, k):
    gen = torch.Generator().manual_seed(m + n + k)
    a, ai = _ints_bf16(gen, (m, k), -2, 3)
    b, bi = _ints_bf16(gen, (2 * n, k), -2, 3)
    scale = 2.0 ** -5
    a = (a.float() * scale).to(torch.bfloat16)
    gu = (ai @ bi.T).to(torch.float64) * scale   # exact
    g, u = gu[:, :n].numpy(), gu[:, n:].numpy()
    h_ref = oracle_lib.bf16_to_double(oracle_lib.bf16_from_double(g / (1 + np.exp(-g)) * u))
    c, err = _pairs(B, a, b, m, n, k, 1)
    assert err == 0
    np.testing.assert_array_equal(_bits(c), _bits(_single(B, a, b, m, n, k, 1)))
    diff = np.abs(c.cpu().double().numpy() - h_ref)
    assert np.all(diff <= np.abs(h_ref) * 2.0 ** -7 + 1e-30)
    assert np.mean(diff == 0) > 0.995


def test_pair_swiglu_midpoints_round_to_even(oracle_lib):
    a, b = pc.swiglu_midpoint_inputs()
    pc.check_swiglu_bits(pc.gpu_swiglu_pairs(a, b), a, b, oracle_lib)


def test_pair_bounded_wait_gives_up_and_context_survives(B):
    m, n, k = 64, 256, 128
    a = torch.ones((m, k), dtype=torch.bfloat16)
    b = torch.ones((n, k), dtype=torch.bfloat16)
    c = torch.zeros((m, n), device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")   # nothing ever sets it
    _, code = _pairs(B, a, b, m, n, k, 0, flag=flag, timeout_ns=20_000_000, out=c)
    assert code & 0xFF == 1            # timeout
    assert (code >> 8) & 0xFF == 5     # at the stall-flag wait
    assert torch.all(c == 0)           # nothing was stored
    flag.fill_(1)
    c2, code = _pairs(B, a, b, m, n, k, 0, flag=flag, timeout_ns=2_000_000_000)
    assert code == 0
    assert torch.all(c2 == k)
