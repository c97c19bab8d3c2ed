"""The tcgen05 GEMM kernel on its own, through the C ABI's diagnostic entry point (GPU).

Exact-integer inputs make every product and every partial sum exactly representable in float32, so whatever
order the tensor cores accumulate in, the result must equal the integer matmul bit for bit: a wrong descriptor,
swizzle, K step or tile offset shows up as a mismatch.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from expert_major_chunked_gb300 import binding
    binding.lib()
    return binding


def _ints_bf16(gen, shape, lo, hi):
    v = torch.randint(lo, hi, shape, generator=gen, dtype=torch.int32)
    return v.to(torch.bfloat16), v.to(torch.int64)


@pytest.mark.parametrize("m,n,k", [(1, 16, 64), (77, 48, 128), (128, 256, 64), (300, 320, 192), (1000, 512, 2048),
                                   (129, 16, 512), (333, 1024, 256)])
def test_debug_gemm_exact_integers(B, m, n, k):
    gen = torch.Generator().manual_seed(m * 7 + n * 13 + k)
    a, ai = _ints_bf16(gen, (m, k), -3, 4)
    b, bi = _ints_bf16(gen, (n, k), -3, 4)
    ref = (ai @ bi.T).to(torch.float64)
    assert ref.abs().max() < 2 ** 24
    da, db = a.cuda(), b.cuda()
    c = torch.full((m, n), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_prefill_debug_gemm(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, k, 0, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_array_equal(c.cpu().to(torch.float64).numpy(), ref.numpy())


def test_debug_gemm_float_inputs_close_to_float64(B):
    gen = torch.Generator().manual_seed(5)
    m, n, k = 200, 256, 2048
    a = torch.randn((m, k), generator=gen).to(torch.bfloat16)
    b = (torch.randn((n, k), generator=gen) * 0.02).to(torch.bfloat16)
    ref = a.double() @ b.double().T
    c = torch.empty((m, n), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da, db = a.cuda(), b.cuda()   # keep the device copies alive until the kernel has run
    B.moe_prefill_debug_gemm(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, k, 0, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    scale = a.double().abs() @ b.double().abs().T
    rel = ((c.cpu().double() - ref).abs() / scale).max().item()
    # fp32 accumulation: far below one part in 2^16 of sum |a_i b_i|
    assert rel < 2.0 ** -16, rel


@pytest.mark.parametrize("m,n,k", [(50, 64, 128), (256, 128, 256), (130, 512, 2048), (1, 768, 64)])
def test_debug_gemm_swiglu_epilogue(B, oracle_lib, m, n, k):
    gen = torch.Generator().manual_seed(m + n + k)
    a, ai = _ints_bf16(gen, (m, k), -2, 3)
    b, bi = _ints_bf16(gen, (2 * n, k), -2, 3)
    scale = 2.0 ** -5  # keeps silu in its curved range; exact power of two
    a = (a.float() * scale).to(torch.bfloat16)
    gu = (ai @ bi.T).to(torch.float64) * scale   # exact
    g, u = gu[:, :n].numpy(), gu[:, n:].numpy()
    h_ref = oracle_lib.bf16_to_double(oracle_lib.bf16_from_double(g / (1 + np.exp(-g)) * u))
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    da, db = a.cuda(), b.cuda()
    B.moe_prefill_debug_gemm(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, k, 1, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    got = c.cpu().double().numpy()
    # g and u are exact; silu in float32 vs float64 can move h across a bf16 rounding boundary only rarely,
    # and then by one bf16 step (2^-8 relative)
    diff = np.abs(got - h_ref)
    assert np.all(diff <= np.abs(h_ref) * 2.0 ** -7 + 1e-30)
    assert np.mean(diff == 0) > 0.995


def test_bounded_wait_gives_up_and_context_survives(B):
    m, n, k = 64, 32, 64
    a = torch.ones((m, k), dtype=torch.bfloat16, device="cuda")
    b = torch.ones((n, k), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((m, n), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")   # nothing ever sets it
    B.moe_prefill_debug_gemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), m, n, k, 0, err.data_ptr(),
                             flag.data_ptr(), 20_000_000)
    torch.cuda.synchronize()
    code = err.item()
    assert code & 0xFF == 1            # timeout
    assert (code >> 8) & 0xFF == 5     # at the stall-flag wait
    assert torch.all(c == 0)           # nothing was computed
    # the context is still usable
    err.zero_()
    flag.fill_(1)
    B.moe_prefill_debug_gemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), m, n, k, 0, err.data_ptr(),
                             flag.data_ptr(), 2_000_000_000)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.all(c == k)
