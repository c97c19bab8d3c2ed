"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function that
include/moe_prefill.h declares, and rejects bad arguments before touching the device."""

import ctypes
import os
import re
import subprocess
import threading

import pytest

from conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from expert_major_chunked_gb300 import binding
    return binding.lib()


def test_header_declares_the_layer_entry_points():
    names = declared_functions()
    for required in ("moe_prefill_plan", "moe_prefill_run", "moe_prefill_combine", "moe_prefill_check",
                     "moe_prefill_destroy", "moe_prefill_last_error"):
        assert required in names
    assert len(names) >= 12


def test_library_exports_every_declared_symbol(L):
    from expert_major_chunked_gb300 import binding
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()], capture_output=True, text=True)
    exported = set(re.findall(r"\s[TW]\s(moe_[a-z0-9_]+)$", out.stdout, flags=re.M))
    assert set(declared_functions()) <= exported
    # every exported moe_* symbol is declared (nothing undocumented leaks out of the library)
    assert exported <= set(declared_functions())


def test_plan_rejects_bad_dims_before_device_use(L):
    from expert_major_chunked_gb300 import binding as b
    plan = ctypes.c_void_p(None)
    ws = ctypes.c_size_t(0)
    assert L.moe_prefill_plan(None, None, None, None, None, None, ctypes.byref(ws), ctypes.byref(plan)) == -1
    assert b"dims" in L.moe_prefill_last_error()
    cases = [
        (b.moe_dims(100, 16, 128, 2, 0, 1, 64, 0), -2),      # hidden not a multiple of 64
        (b.moe_dims(256, 20, 128, 2, 0, 1, 64, 0), -2),      # experts not a multiple of 16
        (b.moe_dims(256, 16, 128, 17, 0, 1, 64, 0), -2),     # k > E
        (b.moe_dims(256, 2048, 128, 2, 0, 1, 64, 0), -2),    # E > 1024
        (b.moe_dims(256, 64, 128, 33, 0, 1, 64, 0), -2),     # k > 32
        (b.moe_dims(256, 16, 128, 2, 0, 0, 64, 0), -2),      # renormalize must be 1
        (b.moe_dims(256, 16, 128, 2, 0, 1, 0, 0), -1),       # max_chunk < 1
        (b.moe_dims(-256, 16, 128, 2, 0, 1, 64, 0), -1),     # negative size
        (b.moe_dims(256, 16, 128, 2, 32, 1, 64, 0), -2),     # shared_inter not a multiple of 64
        (b.moe_dims(256, 16, 128, 2, 0, 1, 64, 3), -2),      # odd ring size
        (b.moe_dims(256, 16, 128, 2, 0, 1, 64, 6), -2),      # half the ring (3) does not divide 16 experts
        (b.moe_dims(256, 16, 128, 2, 0, 1, 64, 32), -2),     # ring larger than the expert count
    ]
    fake = ctypes.c_void_p(0x1000)
    for dims, want in cases:
        st = L.moe_prefill_plan(ctypes.byref(dims), fake, fake, fake, None, None, ctypes.byref(ws),
                                ctypes.byref(plan))
        assert st == want, (dims.hidden, dims.n_experts, dims.top_k, st)
        assert plan.value is None
        assert L.moe_prefill_last_error()
    good = b.moe_dims(256, 16, 128, 2, 128, 1, 64, 0)
    # shared weights missing although shared_inter > 0
    assert L.moe_prefill_plan(ctypes.byref(good), fake, fake, fake, None, None, ctypes.byref(ws),
                              ctypes.byref(plan)) == -1
    # misaligned weight pointer
    odd = ctypes.c_void_p(0x1001)
    assert L.moe_prefill_plan(ctypes.byref(good), odd, fake, fake, fake, fake, ctypes.byref(ws),
                              ctypes.byref(plan)) == -1


def test_plan_without_a_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from expert_major_chunked_gb300 import binding as b
    plan = ctypes.c_void_p(None)
    ws = ctypes.c_size_t(0)
    fake = ctypes.c_void_p(0x1000)
    dims = b.moe_dims(256, 16, 128, 2, 128, 1, 64, 0)
    st = L.moe_prefill_plan(ctypes.byref(dims), fake, fake, fake, fake, fake, ctypes.byref(ws), ctypes.byref(plan))
    assert st in (-4, -6)  # no CUDA device: a CUDA error, never a crash or a fallback
    assert plan.value is None


def test_run_combine_and_misc_reject_bad_arguments(L):
    assert L.moe_prefill_run(None, None, 0, 1, None, 0, None, None, None, None, None, None, None) == -1
    fake = ctypes.c_void_p(0x1000)
    assert L.moe_prefill_combine(fake, fake, fake, None, 4, 0, 64, fake, None) == -1     # k = 0
    assert L.moe_prefill_combine(fake, fake, fake, None, 4, 33, 64, fake, None) == -1    # k > 32
    assert L.moe_prefill_combine(fake, fake, fake, None, 4, 2, 62, fake, None) == -1     # H % 4
    assert L.moe_prefill_combine(fake, fake, fake, None, -1, 2, 64, fake, None) == -1
    assert L.moe_prefill_combine(None, None, None, None, 0, 2, 64, None, None) == 0      # n == 0: no-op
    assert L.moe_prefill_check(None, None) == -1
    assert L.moe_prefill_set_profiling(None, 1) == -1
    assert L.moe_prefill_kernel_times(None, None, None) == -1
    assert L.moe_prefill_launch_count(None) == 0
    assert L.moe_prefill_set_wait_timeout(None, 5) == -1
    L.moe_prefill_destroy(None)
    assert L.moe_prefill_debug_gemm(None, None, None, 1, 16, 64, 0, None, None, 0, None) == -1
    assert L.moe_prefill_debug_gemm(fake, fake, fake, 1, 16, 60, 0, fake, None, 0, None) == -1  # k % 64


def test_float64_combine_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    part = L.moe_prefill_combine_partial_f64
    assert part(fake, fake, fake, fake, 4, 0, 64, 64, 1, 0, fake, None) == -1      # k = 0
    assert part(fake, fake, fake, fake, 4, 2, 62, 64, 1, 0, fake, None) == -1      # H % 4
    assert part(fake, fake, fake, fake, 4, 2, 64, 0, 1, 0, fake, None) == -1       # no experts
    assert part(fake, fake, fake, fake, 4, 2, 64, 2048, 1, 0, fake, None) == -1    # > 1024 experts
    assert part(fake, fake, fake, fake, 4, 2, 64, 64, 3, 0, fake, None) == -1      # 3 parts
    assert part(fake, fake, fake, fake, 4, 2, 64, 48, 128, 0, fake, None) == -1    # more parts than Ep = 64
    assert part(fake, fake, fake, fake, 4, 2, 64, 64, 4, 4, fake, None) == -1      # part out of range
    assert part(fake, fake, fake, fake, 4, 2, 64, 64, 4, 1, None, None) == -1      # no output
    assert part(fake, fake, fake, fake, 4, 2, 64, 64, 4, 1, ctypes.c_void_p(0x1008), None) == -1  # misaligned
    assert part(None, None, None, None, 0, 2, 64, 64, 4, 1, None, None) == 0       # n == 0: no-op
    finish = L.moe_prefill_combine_finish_f64
    ptrs = (ctypes.c_void_p * 32)(*([0x1000] * 32))
    assert finish(ptrs, 32, None, 4, 64, fake, None, None) == -1                   # more than 16 parts
    assert finish(ptrs, 3, None, 4, 64, fake, None, None) == -1                    # not a power of two
    assert finish(ptrs, 2, None, 4, 64, None, None, None) == -1                    # no output
    bad = (ctypes.c_void_p * 2)(0x1000, 0)
    assert finish(bad, 2, None, 4, 64, fake, None, None) == -1                     # a NULL part
    assert finish(None, 2, None, 0, 64, None, None, None) == 0                     # n == 0: no-op
    whole = L.moe_prefill_combine_f64
    assert whole(fake, fake, fake, fake, None, 4, 33, 64, 64, fake, None, None) == -1  # k > 32
    assert whole(fake, fake, fake, fake, None, 4, 2, 64, 64, None, None, None) == -1   # no output
    assert L.moe_prefill_set_combine(None, 1) == -1
    assert b"plan" in L.moe_prefill_last_error()


def test_hot_experts_reject_a_missing_plan(L):
    ids = (ctypes.c_int32 * 2)(1, 2)
    ws = ctypes.c_size_t(7)
    assert L.moe_prefill_set_hot_experts(None, ids, 2, ctypes.byref(ws)) == -1
    assert b"plan" in L.moe_prefill_last_error()
    assert ws.value == 7  # untouched on error
    assert L.moe_prefill_prefetch(None, ctypes.c_void_p(0x1000), 1 << 20, None) == -1
    assert b"plan" in L.moe_prefill_last_error()


def test_last_error_is_per_thread(L):
    L.moe_prefill_combine(None, None, None, None, 4, 0, 64, None, None)
    main_msg = L.moe_prefill_last_error()
    assert main_msg
    seen = {}

    def other():
        seen["msg"] = L.moe_prefill_last_error()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == b""
    assert L.moe_prefill_last_error() == main_msg


def declared_parameter_counts():
    """Number of parameters of every function the headers declare ("(void)" counts as none)."""
    counts = {}
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(HEADER_DIR, fn)).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(([^)]*)\)\s*;",
                             text, flags=re.M):
            params = " ".join(m.group(2).split())
            counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_signatures_match_the_header():
    """The Python binding marshals every declared entry point with as many arguments as the header declares, and
    declares nothing the header does not."""
    from expert_major_chunked_gb300 import binding
    counts = declared_parameter_counts()
    assert set(counts) == set(declared_functions())
    sigs = binding._SIGS
    assert set(sigs) == set(counts), sorted(set(sigs) ^ set(counts))
    for name, (argtypes, _) in sigs.items():
        assert len(argtypes) == counts[name], (name, len(argtypes), counts[name])


def test_debug_gemm_pairs_scratch_and_argument_checks(L):
    """The pair kernel's diagnostic entry: scratch sizes, and arguments rejected before any device use (the
    pointers below are never dereferenced)."""
    from expert_major_chunked_gb300 import binding as b
    # 313 token rows: two token tiles (160 + 153); n = 512: two F32 weight blocks of 256, four SwiGLU blocks of 128
    assert b.moe_prefill_debug_gemm_pairs_scratch(313, 512, 0) == 16 * (2 * 2 + 1)
    assert b.moe_prefill_debug_gemm_pairs_scratch(313, 512, 1) == 16 * (2 * 4 + 1)
    assert b.moe_prefill_debug_gemm_pairs_scratch(257, 256, 0) == 16 * (2 + 1)
    assert b.moe_prefill_debug_gemm_pairs_scratch(256, 256, 0) == 16 * (1 + 1)
    assert b.moe_prefill_debug_gemm_pairs_scratch(0, 512, 0) == 0
    assert b.moe_prefill_debug_gemm_pairs_scratch(1, 256, 2) == 0
    p = ctypes.c_void_p(1 << 20)
    f = L.moe_prefill_debug_gemm_pairs
    assert f(None, p, p, 1, 256, 128, 0, p, 64, p, None, 0, None) == -1      # NULL a
    assert f(p, p, p, 1, 256, 64, 0, p, 64, p, None, 0, None) == -1          # k_dim % 128
    assert f(p, p, p, 1, 128, 128, 0, p, 64, p, None, 0, None) == -2         # F32 needs n % 256
    assert f(p, p, p, 1, 192, 128, 1, p, 64, p, None, 0, None) == -2         # SwiGLU needs n % 128
    assert f(p, p, p, 1, 256, 128, 3, p, 64, p, None, 0, None) == -1         # unknown epilogue
    assert f(p, p, p, 300, 512, 128, 0, p, 16, p, None, 0, None) == -3       # scratch too small
    assert b"scratch" in L.moe_prefill_last_error()
