"""ctypes wrapper of the float64 reference oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the benchmark's CPU-baseline and
reference legs. The product library never imports or loads it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.c")]
_lock = threading.Lock()
_lib = None


CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall",
          "-Wextra"]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/lib/liboracle.so (gcc, OpenMP, no floating-point contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(p) for p in _SOURCES + [os.path.join(_HERE, "oracle.h")])
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest_src:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp] + _SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(L):
    """Declare the C signatures on a loaded oracle library (this one, or a test's rebuilt copy of oracle.c)."""
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    L.oracle_num_threads.restype = ctypes.c_int
    L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    L.oracle_bf16_from_double.restype = ctypes.c_uint16
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_bf16_round_array.argtypes = [P, P, i64]
    L.oracle_router_logits.argtypes = [P, P, i64, i32, i32, P]
    L.oracle_topk.argtypes = [P, i64, i32, i32, P, P]
    L.oracle_swiglu_ffn.argtypes = [P, P, P, i32, i32, P, P]
    L.oracle_moe_forward.argtypes = [P, P, P, P, P, P, P, i64, P, i64, P, P, P, P]
    L.oracle_permutation.argtypes = [P, i64, i32, i32, i32, P, P, P]
    L.oracle_combine_f64.argtypes = [P, P, P, P, i64, i32, i32, P, P]
    L.oracle_combine_f32_canonical.argtypes = [P, P, P, P, i64, i32, i32, P]
    L.oracle_combine_tree_partial_f64.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, i32, P]
    L.oracle_combine_tree_finish_f64.argtypes = [P, i32, P, i64, i32, P, P]
    L.oracle_dequant_mxfp8.argtypes = [P, P, i64, i64, P]
    L.oracle_dequant_nvfp4.argtypes = [P, P, i64, i64, P]
    for name in ("oracle_bf16_round_array", "oracle_router_logits", "oracle_topk", "oracle_swiglu_ffn",
                 "oracle_moe_forward", "oracle_permutation", "oracle_combine_f64",
                 "oracle_combine_f32_canonical", "oracle_combine_tree_partial_f64",
                 "oracle_combine_tree_finish_f64", "oracle_dequant_mxfp8",
                 "oracle_dequant_nvfp4"):
        getattr(L, name).restype = ctypes.c_int
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(ctypes.CDLL(_LIB_PATH))
    return _lib


class _Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("shared_inter", ctypes.c_int32)]


def _u16(a) -> np.ndarray:
    """BF16 data as a contiguous uint16 numpy array (accepts torch bf16 tensors or uint16 arrays)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(a.contiguous().view(torch.int16).numpy().view(np.uint16))
    arr = np.asarray(a)
    if arr.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {arr.dtype}")
    return np.ascontiguousarray(arr)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected its arguments (rc={rc})")


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def bf16_from_double(v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    _check(lib().oracle_bf16_round_array(_ptr(v), _ptr(out), v.size), "bf16_round")
    return out


def bf16_to_double(b) -> np.ndarray:
    b = _u16(b)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def router_logits(x, w_router) -> np.ndarray:
    x, wr = _u16(x), _u16(w_router)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _check(lib().oracle_router_logits(_ptr(x), _ptr(wr), T, H, E, _ptr(out)), "router_logits")
    return out


def topk(logits: np.ndarray, k: int):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = l.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().oracle_topk(_ptr(l), T, E, k, _ptr(ids), _ptr(w)), "topk")
    return ids, w


def swiglu_ffn(x_row, w_gu, w_down):
    x, g, d = _u16(x_row), _u16(w_gu), _u16(w_down)
    H = x.shape[-1]
    I = g.shape[0] // 2
    y = np.empty(H, dtype=np.float64)
    h = np.empty(I, dtype=np.uint16)
    _check(lib().oracle_swiglu_ffn(_ptr(x), _ptr(g), _ptr(d), H, I, _ptr(y), _ptr(h)), "swiglu_ffn")
    return y, h


def moe_forward(inputs: dict, top_k: int, token_idx=None):
    """Evaluate the layer on the listed tokens (all when token_idx is None).

    Returns (out_ref float64 [n][H], out_bf16 uint16 [n][H], topk_id int32 [n][k], topk_w float64 [n][k]).
    """
    x, wr, wgu, wd = (_u16(inputs[k]) for k in ("x", "w_router", "w_gu", "w_down"))
    T, H = x.shape
    E = wr.shape[0]
    I = wgu.shape[1] // 2
    has_shared = inputs.get("ws_gu") is not None
    wsg = _u16(inputs["ws_gu"]) if has_shared else None
    wsd = _u16(inputs["ws_down"]) if has_shared else None
    Is = wsg.shape[0] // 2 if has_shared else 0
    dims = _Dims(H, E, I, top_k, Is)
    if token_idx is None:
        idx_arr, n = None, T
    else:
        idx_arr = np.ascontiguousarray(np.asarray(token_idx, dtype=np.int64))
        n = idx_arr.size
    out_ref = np.empty((n, H), dtype=np.float64)
    out_bf = np.empty((n, H), dtype=np.uint16)
    ids = np.empty((n, top_k), dtype=np.int32)
    w = np.empty((n, top_k), dtype=np.float64)
    rc = lib().oracle_moe_forward(ctypes.byref(dims), _ptr(x), _ptr(wr), _ptr(wgu), _ptr(wd),
                                  _ptr(wsg) if has_shared else None, _ptr(wsd) if has_shared else None,
                                  T, _ptr(idx_arr) if idx_arr is not None else None, n,
                                  _ptr(out_ref), _ptr(out_bf), _ptr(ids), _ptr(w))
    _check(rc, "moe_forward")
    return out_ref, out_bf, ids, w


def permutation(topk_id: np.ndarray, n_experts: int, chunk: int):
    ids = np.ascontiguousarray(topk_id, dtype=np.int32)
    T, k = ids.shape
    n_chunks = (T + chunk - 1) // chunk
    offs = np.empty((n_chunks, n_experts + 1), dtype=np.int32)
    row_token = np.empty(T * k, dtype=np.int32)
    token_row = np.empty((T, k), dtype=np.int32)
    _check(lib().oracle_permutation(_ptr(ids), T, k, n_experts, chunk, _ptr(offs), _ptr(row_token),
                                    _ptr(token_row)), "permutation")
    return offs, row_token, token_row


def _combine_args(y, w, token_row, s):
    y = np.ascontiguousarray(y, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    tr = np.ascontiguousarray(token_row, dtype=np.int32)
    s = None if s is None else np.ascontiguousarray(s, dtype=np.float32)
    return y, w, tr, s


def combine_f64(y, w, token_row, s=None):
    y, w, tr, s = _combine_args(y, w, token_row, s)
    n, k = w.shape
    H = y.shape[1]
    ref = np.empty((n, H), dtype=np.float64)
    out = np.empty((n, H), dtype=np.uint16)
    _check(lib().oracle_combine_f64(_ptr(y), _ptr(w), _ptr(tr), _ptr(s) if s is not None else None, n, k, H,
                                    _ptr(ref), _ptr(out)), "combine_f64")
    return ref, out


def combine_f32_canonical(y, w, token_row, s=None):
    y, w, tr, s = _combine_args(y, w, token_row, s)
    n, k = w.shape
    H = y.shape[1]
    out = np.empty((n, H), dtype=np.uint16)
    _check(lib().oracle_combine_f32_canonical(_ptr(y), _ptr(w), _ptr(tr), _ptr(s) if s is not None else None,
                                              n, k, H, _ptr(out)), "combine_f32_canonical")
    return out


def combine_tree_partial_f64(y, w, token_row, topk_id, n_experts, n_parts=1, part=0):
    """float64 value of one aligned block of the expert-id tree (part `part` of `n_parts`); [n][H] float64."""
    y, w, tr, _ = _combine_args(y, w, token_row, None)
    ids = np.ascontiguousarray(topk_id, dtype=np.int32)
    n, k = w.shape
    H = y.shape[1]
    out = np.empty((n, H), dtype=np.float64)
    _check(lib().oracle_combine_tree_partial_f64(_ptr(y), _ptr(w), _ptr(tr), _ptr(ids), n, k, H, n_experts, n_parts,
                                                 part, _ptr(out)), "combine_tree_partial_f64")
    return out


def combine_tree_finish_f64(partials, s=None):
    """Sum the parts in the tree, add the shared expert, round once to float32, then to bf16: (f32, bf16 bits)."""
    parts = np.ascontiguousarray(np.stack(list(partials)), dtype=np.float64)
    R, n, H = parts.shape
    s = None if s is None else np.ascontiguousarray(s, dtype=np.float32)
    f32 = np.empty((n, H), dtype=np.float32)
    bf = np.empty((n, H), dtype=np.uint16)
    _check(lib().oracle_combine_tree_finish_f64(_ptr(parts), R, _ptr(s) if s is not None else None, n, H, _ptr(f32),
                                                _ptr(bf)), "combine_tree_finish_f64")
    return f32, bf


def combine_tree_f64(y, w, token_row, topk_id, n_experts, s=None):
    """The unsplit float64 tree combine: one part, then the finish."""
    return combine_tree_finish_f64([combine_tree_partial_f64(y, w, token_row, topk_id, n_experts)], s)


def dequant_mxfp8(codes, scales):
    """E4M3 codes [E][R][K] (uint8) with E8M0 scales [E][K/32][R] (uint8) -> exact bf16 bits [E][R][K]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    E, R, K = codes.shape
    assert scales.shape == (E, K // 32, R), scales.shape
    out = np.empty((E, R, K), dtype=np.uint16)
    for e in range(E):
        _check(lib().oracle_dequant_mxfp8(_ptr(codes[e]), _ptr(scales[e]), R, K, _ptr(out[e])), "dequant_mxfp8")
    return out


def dequant_nvfp4(codes, scales):
    """E2M1 codes [E][R][K/2] (two per byte, low nibble first) with E4M3 scales [E][K/16][R] -> bf16 bits [E][R][K]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    E, R, K2 = codes.shape
    K = 2 * K2
    assert scales.shape == (E, K // 16, R), scales.shape
    out = np.empty((E, R, K), dtype=np.uint16)
    for e in range(E):
        _check(lib().oracle_dequant_nvfp4(_ptr(codes[e]), _ptr(scales[e]), R, K, _ptr(out[e])), "dequant_nvfp4")
    return out
