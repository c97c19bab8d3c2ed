"""GPU-vs-oracle parity gates as plain functions: GPU results in, an oracle module in, AssertionError when they
disagree. The GPU tests call them with the oracle; tests/test_gpu_planted.py calls the same functions with
planted copies of the oracle (tests/planted.py) to show that each gate goes red on the mistake it is meant to catch.

Also the inputs whose float32 results land exactly on bf16 rounding midpoints (ties), for the combine kernel and the
SwiGLU epilogue: on random data an exact tie practically never occurs, so the ties-to-even rule is otherwise
untested on the GPU.
"""

from __future__ import annotations

import numpy as np
import torch

from layer_helpers import MAX_ABS, REL_L2, compare_out, out_bits, tau_bound


# ------------------------------------------------------------------------------------------------ layer gates

def check_routing_ids(res, inp, k, orc):
    """Top-k ids bit-exact (ties to the lower expert id)."""
    logits = orc.router_logits(inp["x"], inp["w_router"])
    ids, _ = orc.topk(logits, k)
    np.testing.assert_array_equal(res["ids"], ids)


def check_permutation(res, inp, k, chunk, orc):
    """Per-chunk expert offsets and the row->token map bit-exact."""
    logits = orc.router_logits(inp["x"], inp["w_router"])
    ids, _ = orc.topk(logits, k)
    offs, row_token, _ = orc.permutation(ids, inp["w_router"].shape[0], chunk)
    np.testing.assert_array_equal(res["offs"], offs)
    np.testing.assert_array_equal(res["row_token"], row_token)


def check_weights(res, inp, k, orc):
    """Routing weights within the logit-error bound of the oracle's (first-order softmax sensitivity)."""
    logits = orc.router_logits(inp["x"], inp["w_router"])
    _, w = orc.topk(logits, k)
    tau = tau_bound(inp["x"], inp["w_router"])
    bound = w * (2 * tau[:, None]) + 2e-6
    err = np.abs(res["w"].astype(np.float64) - w)
    assert np.all(err <= bound), float(np.max(err - bound))


def check_output(res, inp, k, orc):
    """BF16 output within max-abs 2e-2 and relative L2 1e-3 of the oracle's BF16 output."""
    _, ref_bf, _, _ = orc.moe_forward(inp, k)
    max_abs, rel = compare_out(res["out"], ref_bf, orc)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)


# ------------------------------------------------------------------------------------------------ combine

def combine_random_inputs(seed=11, n=333, k=10, H=2048):
    gen = torch.Generator().manual_seed(seed)
    R = n * k
    y = torch.randn((R, H), generator=gen)
    w = torch.rand((n, k), generator=gen)
    w = w / w.sum(1, keepdim=True)
    s = torch.randn((n, H), generator=gen)
    tr = torch.randperm(R, generator=gen).reshape(n, k).to(torch.int32)
    return y.numpy(), w.numpy(), tr.numpy(), s.numpy()


def combine_midpoint_inputs(seed=12, n=200, H=512):
    """Four slots with power-of-two weights (1/2, 1/4, 1/8, 1/8, permuted per token) and a shared term, built so
    that every product and partial sum is exact in float32 and the final sum is exactly halfway between two
    neighbouring bf16 values: v = (2j + 1) 2^(e-8) with j in [128, 254], e in [-6, 6], either sign. Half of the
    cases (j even) round down under ties-to-even and up under ties-away-from-zero."""
    rng = np.random.default_rng(seed)
    k = 4
    R = n * k
    base_w = np.array([0.5, 0.25, 0.125, 0.125], dtype=np.float32)
    w = np.stack([rng.permutation(base_w) for _ in range(n)]).astype(np.float32)
    tr = rng.permutation(R).reshape(n, k).astype(np.int32)
    j = rng.integers(128, 255, size=(n, H))
    e = rng.integers(-6, 7, size=(n, H))
    sign = rng.choice([-1, 1], size=(n, H))
    unit = np.ldexp(1.0, e - 8)
    target = sign * (2 * j + 1)
    c = rng.integers(-300, 301, size=(n, k, H))
    c_shared = target - c.sum(axis=1)
    y = np.zeros((R, H), dtype=np.float32)
    for s in range(k):
        y[tr[:, s]] = (c[:, s] * unit / w[:, s:s + 1]).astype(np.float32)
    s_sh = (c_shared * unit).astype(np.float32)
    # the construction is exact: check it in float64
    acc = np.zeros((n, H))
    for s in range(k):
        acc = acc + w[:, s:s + 1].astype(np.float64) * y[tr[:, s]].astype(np.float64)
    assert np.array_equal(acc + s_sh, target * unit)
    return y, w, tr, s_sh


def gpu_combine(y, w, tr, s):
    from expert_major_chunked_gb300 import binding
    n, k = w.shape
    H = y.shape[1]
    dy, dw, dtr = torch.from_numpy(y).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(tr).cuda()
    ds = torch.from_numpy(s).cuda() if s is not None else None
    out = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    binding.moe_prefill_combine(dy.data_ptr(), dw.data_ptr(), dtr.data_ptr(), ds.data_ptr() if ds is not None else None,
                                n, k, H, out.data_ptr())
    torch.cuda.synchronize()
    return out_bits(out.cpu())


def check_combine_bits(gpu_bits, y, w, tr, s, orc):
    """The combine kernel's bytes equal the oracle's float32 canonical reduction."""
    np.testing.assert_array_equal(gpu_bits, orc.combine_f32_canonical(y, w, tr, s))


# ------------------------------------------------------------------------------------------------ SwiGLU epilogue

def swiglu_midpoint_inputs(seed=13, m=128, n=512, K=64):
    """Operands of one gate/up GEMM (a [m][K], b [2n][K] = gate rows then up rows) whose SwiGLU outputs are exact
    bf16 midpoints: g = 64 * 2^(r % 4) exactly (so 1 + exp(-g) == 1 in float32 and float64 and silu(g) = g), and
    u = 2^(r % 4) * (b_c + h_c) with b_c a bf16 value and h_c = +-half of its last place, so silu(g) * u is exact
    and halfway between two bf16 values."""
    rng = np.random.default_rng(seed)
    a = np.zeros((m, K), dtype=np.float32)
    scale = np.ldexp(1.0, np.arange(m) % 4)
    a[:, 0] = a[:, 1] = a[:, 2] = scale
    b = np.zeros((2 * n, K), dtype=np.float32)
    b[:n, 0] = 64.0
    jb = rng.integers(128, 256, size=n)
    eb = rng.integers(-6, 3, size=n)
    sb = rng.choice([-1.0, 1.0], size=n)
    bc = sb * jb * np.ldexp(1.0, eb - 7)                      # |b_c| = jb/128 * 2^eb: 8 significant bits
    hsign = np.where(jb == 128, 1.0, rng.choice([-1.0, 1.0], size=n))
    hc = sb * hsign * np.ldexp(1.0, eb - 8)                    # half of b_c's last place
    b[n:, 1] = bc
    b[n:, 2] = hc
    at = torch.from_numpy(a).to(torch.bfloat16)
    bt = torch.from_numpy(b).to(torch.bfloat16)
    assert torch.equal(at.float(), torch.from_numpy(a)) and torch.equal(bt.float(), torch.from_numpy(b))
    return at, bt


def gpu_swiglu(a, b):
    from expert_major_chunked_gb300 import binding
    m, K = a.shape
    n = b.shape[0] // 2
    da, db = a.cuda(), b.cuda()
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.moe_prefill_debug_gemm(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, K, 1, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    return out_bits(c.cpu())


def gpu_swiglu_pairs(a, b):
    """The same SwiGLU GEMM through the CTA-pair kernel (K padded with zeros to its multiple of 128)."""
    from expert_major_chunked_gb300 import binding
    m, K = a.shape
    n = b.shape[0] // 2
    Kp = (K + 127) // 128 * 128
    ap = torch.zeros((m, Kp), dtype=torch.bfloat16)
    bp = torch.zeros((2 * n, Kp), dtype=torch.bfloat16)
    ap[:, :K] = a
    bp[:, :K] = b
    da, db = ap.cuda(), bp.cuda()
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    need = binding.moe_prefill_debug_gemm_pairs_scratch(m, n, 1)
    scratch = torch.zeros(need // 4 + 4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.moe_prefill_debug_gemm_pairs(da.data_ptr(), db.data_ptr(), c.data_ptr(), m, n, Kp, 1, scratch.data_ptr(),
                                         scratch.numel() * 4, err.data_ptr())
    torch.cuda.synchronize()
    assert err.item() == 0
    return out_bits(c.cpu())


def check_swiglu_bits(gpu_bits, a, b, orc):
    """The SwiGLU epilogue's bf16 h equals the oracle's h (one expert FFN, h = bf16(silu(g) * u)) bit for bit."""
    m, K = a.shape
    n = b.shape[0] // 2
    zeros_down = np.zeros((K, n), dtype=np.uint16)
    want = np.stack([orc.swiglu_ffn(a[r], b, zeros_down)[1] for r in range(m)])
    np.testing.assert_array_equal(gpu_bits, want)
