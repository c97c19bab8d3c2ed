"""Planted mistakes in the oracle (CPU), to show that the GPU parity gates go red on a wrong answer.

"EXL3 Flash Next: deep prefill (3/8)", *Device results*, reports its controls all red; "Flash Next EXL3: exact deep
prefill", *Independent numerical-phase audit*, plants controls the same way. Here a control is a copy of oracle.c
with one plausible mistake substituted into its text, compiled on the CPU into a library of its own. The GPU runs
only the correct kernels. A gate that compares the GPU with the oracle must pass against the real oracle and fail
against each planted copy that it is meant to catch. The kernels themselves are never altered.

Each entry: the mistake, the passage of the pages (or the reading of it) it breaks, and exact text substitutions
(old, new) in oracle.c. Every `old` must occur exactly once, so a change to oracle.c that moves the text makes the
control fail loudly instead of silently testing nothing.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import shutil
import subprocess
import threading

import oracle

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))
BUILD_DIR = os.path.join(ORACLE_DIR, "lib", "planted")

PLANTED = {
    # "Flash Next EXL3: exact deep prefill" (introduction): the routed contributions are reduced in one canonical
    # order; the reading is ascending expert id. Reversed order rounds differently.
    "combine_descending": [
        ("      for (int32_t s = 0; s < top_k; ++s) {\n        volatile float prod",
         "      for (int32_t s = top_k - 1; s >= 0; --s) {\n        volatile float prod"),
    ],
    # The shared expert is indexed after the routed experts (umbrella PR #1113, "Memory and execution split"): it is
    # added last. Adding it first changes the float32 rounding sequence.
    "shared_added_first": [
        ("      volatile float acc = 0.0f;\n      for (int32_t s = 0; s < top_k; ++s) {",
         "      volatile float acc = s_shared ? s_shared[t * hidden + o] : 0.0f;\n"
         "      for (int32_t s = 0; s < top_k; ++s) {"),
        ("      if (s_shared) acc = acc + s_shared[t * hidden + o];\n      out_bf16[t * hidden + o]",
         "      out_bf16[t * hidden + o]"),
    ],
    # Reading of the top-k: an exact tie goes to the lower expert id.
    "tie_to_higher_id": [
        ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;"),
    ],
    # Member lists ("Latest prefill efficiency candidate": per-expert member lists per chunk): an exclusive scan of
    # the per-expert counts. Off by one after the first expert.
    "scan_base_off_by_one": [
        ("if (expert_offsets) expert_offsets[c * (n_experts + 1) + e] = run;",
         "if (expert_offsets) expert_offsets[c * (n_experts + 1) + e] = run + (e > 0 ? 1 : 0);"),
    ],
    # Reading of every BF16 store: round to nearest, ties to even. C's round() sends ties away from zero.
    "round_half_away": [
        ("double r = rint(a / q) * q;", "double r = round(a / q) * q;"),
    ],
    # "Flash Next EXL3: exact deep prefill", *Independent numerical-phase audit*: the gate/up kernel writes complete
    # scratch bytes that the down kernel reads, i.e. h is stored (BF16) between the projections. Not rounding it
    # changes the layer output.
    "h_not_rounded": [
        ("    h[j] = oracle_bf16_to_double(hb);", "    h[j] = silu * u;"),
    ],
    # Reading of the fused gate/up matrix: gate rows first, then up rows.
    "gate_up_swapped": [
        ("    const uint16_t* wg = w_gu + (int64_t)j * hidden;\n"
         "    const uint16_t* wu = w_gu + (int64_t)(inter + j) * hidden;",
         "    const uint16_t* wu = w_gu + (int64_t)j * hidden;\n"
         "    const uint16_t* wg = w_gu + (int64_t)(inter + j) * hidden;"),
    ],
    # The 3001-token workload states softmax-renormalised weights: the softmax over the selected experts only.
    "no_renormalise": [
        ("for (int32_t s = 0; s < k; ++s) denom += exp(l[ids[s]] - lmax);",
         "for (int32_t s = 0; s < E; ++s) denom += exp(l[s] - lmax);"),
    ],
    # The layer adds the shared expert to every token.
    "shared_dropped": [
        ("      if (Is > 0) {\n        oracle_swiglu_ffn(xr, ws_gu", "      if (0) {\n        oracle_swiglu_ffn(xr, ws_gu"),
    ],
    # silu(z) = z / (1 + exp(-z)).
    "silu_sign_flipped": [
        ("double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    ],
}

_lock = threading.Lock()
_libs: dict = {}


def planted_source(name: str) -> str:
    with open(os.path.join(ORACLE_DIR, "oracle.c")) as f:
        src = f.read()
    for old, new in PLANTED[name]:
        n = src.count(old)
        if n != 1:
            raise AssertionError(f"planted control {name!r}: expected text found {n} times in oracle.c")
        src = src.replace(old, new)
    return src


def build(name: str) -> str:
    """Compile oracle.c with the named mistake (same compiler and flags as the oracle) and return the library path."""
    out_dir = os.path.join(BUILD_DIR, name)
    os.makedirs(out_dir, exist_ok=True)
    src_path = os.path.join(out_dir, "oracle.c")
    with open(src_path, "w") as f:
        f.write(planted_source(name))
    shutil.copyfile(os.path.join(ORACLE_DIR, "oracle.h"), os.path.join(out_dir, "oracle.h"))
    lib_path = os.path.join(out_dir, f"liboracle_{name}.so")
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", tmp, src_path, "-lm"], check=True)
    os.replace(tmp, lib_path)
    return lib_path


def load(name: str):
    with _lock:
        if name not in _libs:
            _libs[name] = oracle.bind(ctypes.CDLL(build(name)))
        return _libs[name]


@contextlib.contextmanager
def planted_oracle(name: str):
    """The oracle module with its library swapped for the planted copy, for the duration of the block."""
    L = load(name)
    oracle.lib()  # make sure the real library is loaded first, so it is what gets restored
    saved = oracle._lib
    oracle._lib = L
    try:
        yield oracle
    finally:
        oracle._lib = saved
