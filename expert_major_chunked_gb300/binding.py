"""ctypes binding of libmoe_prefill.so (include/moe_prefill.h), argument marshalling only.

The functions carry the C names and take raw device pointers (ints) and sizes; `MoePrefill` below wraps them for
torch tensors (PyTorch supplies device memory and streams). Every step of the layer runs in the library's CUDA
kernels. If the library cannot be built or loaded, the import of the library raises: there is no other code path.
"""

from __future__ import annotations

import ctypes
import threading
from typing import Optional

from . import build as _build

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
                -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT", -6: "MOE_ERR_ARCH", -7: "MOE_ERR_DEVICE_BOUNDS"}
KERNEL_NAMES = ["norms", "router", "topk", "count", "scan", "permute", "gate_up", "down", "combine"]
KERNEL_KINDS = len(KERNEL_NAMES)


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class moe_dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("shared_inter", ctypes.c_int32), ("renormalize", ctypes.c_int32),
                ("max_chunk", ctypes.c_int32), ("offload_slots", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_SIGS = {
    "moe_prefill_plan": ([ctypes.POINTER(moe_dims), _P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_size_t),
                          ctypes.POINTER(_P)], ctypes.c_int),
    "moe_prefill_plan_mxfp8": ([ctypes.POINTER(moe_dims), _P, _P, _P, _P, _P, _P, _P,
                                ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(_P)], ctypes.c_int),
    "moe_prefill_plan_nvfp4": ([ctypes.POINTER(moe_dims), _P, _P, _P, _P, _P, _P, _P,
                                ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(_P)], ctypes.c_int),
    "moe_prefill_run": ([_P, _P, ctypes.c_int64, ctypes.c_int32, _P, ctypes.c_size_t, _P, _P, _P, _P, _P, _P, _P],
                        ctypes.c_int),
    "moe_prefill_run_host": ([_P, _P, ctypes.c_int64, ctypes.c_int32, _P, ctypes.c_size_t, _P, _P, _P, _P, _P, _P,
                              _P, _P, _P], ctypes.c_int),
    "moe_prefill_combine": ([_P, _P, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P], ctypes.c_int),
    "moe_prefill_combine_partial_f64": ([_P, _P, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P], ctypes.c_int),
    "moe_prefill_combine_finish_f64": ([_P, ctypes.c_int32, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P],
                                       ctypes.c_int),
    "moe_prefill_combine_f64": ([_P, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                 _P, _P, _P], ctypes.c_int),
    "moe_prefill_set_combine": ([_P, ctypes.c_int32], ctypes.c_int),
    "moe_prefill_set_cta_pairs": ([_P, ctypes.c_int32], ctypes.c_int),
    "moe_prefill_cta_pairs": ([_P], ctypes.c_int32),
    "moe_prefill_set_offload_copy": ([_P, ctypes.c_int32], ctypes.c_int),
    "moe_prefill_set_hot_experts": ([_P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "moe_prefill_prefetch": ([_P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "moe_prefill_forget_workspace": ([_P], ctypes.c_int),
    "moe_prefill_check": ([_P, _P], ctypes.c_int),
    "moe_prefill_destroy": ([_P], None),
    "moe_prefill_last_error": ([], ctypes.c_char_p),
    "moe_prefill_set_profiling": ([_P, ctypes.c_int32], ctypes.c_int),
    "moe_prefill_kernel_times": ([_P, _P, _P], ctypes.c_int),
    "moe_prefill_kernel_trace": ([_P, _P, _P, _P, ctypes.c_int32, _P], ctypes.c_int),
    "moe_prefill_launch_count": ([_P], ctypes.c_int64),
    "moe_prefill_set_wait_timeout": ([_P, ctypes.c_uint64], ctypes.c_int),
    "moe_prefill_run_stats": ([_P, _P, _P, ctypes.c_int32], ctypes.c_int),
    "moe_prefill_run_noalloc": ([_P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_prefill_debug_gemm": ([_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                ctypes.c_uint64, _P], ctypes.c_int),
    "moe_prefill_debug_gemm_pairs_scratch": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32], ctypes.c_size_t),
    "moe_prefill_debug_gemm_pairs": ([_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P,
                                      ctypes.c_size_t, _P, _P, ctypes.c_uint64, _P], ctypes.c_int),
}


def lib(build_if_needed: bool = True):
    """Load libmoe_prefill.so (building it with nvcc first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_needed else _build.LIB_PATH
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB_PATH


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, lib().moe_prefill_last_error().decode())


def moe_prefill_last_error() -> str:
    return lib().moe_prefill_last_error().decode()


def moe_prefill_plan(dims: moe_dims, w_router: int, w_gu: int, w_down: int, ws_gu: Optional[int],
                     ws_down: Optional[int]):
    """Returns (plan handle, workspace bytes)."""
    ws = ctypes.c_size_t(0)
    plan = _P(None)
    _check(lib().moe_prefill_plan(ctypes.byref(dims), w_router, w_gu, w_down, ws_gu, ws_down, ctypes.byref(ws),
                                  ctypes.byref(plan)))
    return plan.value, ws.value


def moe_prefill_plan_mxfp8(dims: moe_dims, w_router: int, gu_codes: int, gu_scales: int, down_codes: int,
                           down_scales: int, ws_gu: Optional[int], ws_down: Optional[int], fmt: str = "mxfp8"):
    """Returns (plan handle, workspace bytes) for block-scaled routed experts (fmt "mxfp8" or "nvfp4")."""
    ws = ctypes.c_size_t(0)
    plan = _P(None)
    fn = lib().moe_prefill_plan_nvfp4 if fmt == "nvfp4" else lib().moe_prefill_plan_mxfp8
    _check(fn(ctypes.byref(dims), w_router, gu_codes, gu_scales, down_codes, down_scales, ws_gu, ws_down,
              ctypes.byref(ws), ctypes.byref(plan)))
    return plan.value, ws.value


def moe_prefill_run(plan, x, T, chunk, workspace, workspace_bytes, out, topk_id=None, topk_w=None,
                    expert_offsets=None, row_token=None, compute=None, copy=None):
    _check(lib().moe_prefill_run(plan, x, T, chunk, workspace, workspace_bytes, out, topk_id, topk_w,
                                 expert_offsets, row_token, compute, copy))


def moe_prefill_run_noalloc(plan, x, T, chunk, out, topk_id=None, topk_w=None, expert_offsets=None, row_token=None,
                            device_status=None, stream=None):
    """moe_prefill_run with the library's built-in scratch array instead of a caller workspace (see the header)."""
    _check(lib().moe_prefill_run_noalloc(plan, x, T, chunk, out, topk_id, topk_w, expert_offsets, row_token,
                                         device_status, stream))


def moe_prefill_combine(y, w, token_row, s, n, k, H, out, stream=None):
    _check(lib().moe_prefill_combine(y, w, token_row, s, n, k, H, out, stream))


def moe_prefill_combine_partial_f64(y, w, token_row, topk_id, n, k, H, n_experts, n_parts, part, partial,
                                    stream=None):
    _check(lib().moe_prefill_combine_partial_f64(y, w, token_row, topk_id, n, k, H, n_experts, n_parts, part,
                                                 partial, stream))


def moe_prefill_combine_finish_f64(partials, s, n, H, out, out_f32=None, stream=None):
    """partials: list of device pointers (one per part, part 0 first)."""
    arr = (ctypes.c_void_p * len(partials))(*partials)
    _check(lib().moe_prefill_combine_finish_f64(arr, len(partials), s, n, H, out, out_f32, stream))


def moe_prefill_combine_f64(y, w, token_row, topk_id, s, n, k, H, n_experts, out, out_f32=None, stream=None):
    _check(lib().moe_prefill_combine_f64(y, w, token_row, topk_id, s, n, k, H, n_experts, out, out_f32, stream))


COMBINE_F32, COMBINE_F64_TREE = 0, 1
OFFLOAD_COPY_ALL, OFFLOAD_COPY_ROUTED = 0, 1


def moe_prefill_set_offload_copy(plan, mode: int):
    _check(lib().moe_prefill_set_offload_copy(plan, mode))


def moe_prefill_set_hot_experts(plan, hot_ids) -> int:
    """Names the offloaded experts kept resident; returns the workspace size later runs need."""
    ids = [int(e) for e in hot_ids]
    arr = (ctypes.c_int32 * max(1, len(ids)))(*ids)
    ws = ctypes.c_size_t(0)
    _check(lib().moe_prefill_set_hot_experts(plan, arr if ids else None, len(ids), ctypes.byref(ws)))
    return ws.value


def moe_prefill_forget_workspace(workspace):
    _check(lib().moe_prefill_forget_workspace(workspace))


def moe_prefill_set_combine(plan, mode: int):
    _check(lib().moe_prefill_set_combine(plan, mode))


PAIRS_GATE_UP, PAIRS_DOWN = 1, 2


def moe_prefill_set_cta_pairs(plan, which: int):
    _check(lib().moe_prefill_set_cta_pairs(plan, int(which)))


def moe_prefill_cta_pairs(plan) -> int:
    return int(lib().moe_prefill_cta_pairs(plan))


def moe_prefill_check(workspace, stream=None) -> int:
    """Returns the status (does not raise) so callers can test for device-side errors."""
    return lib().moe_prefill_check(workspace, stream)


def moe_prefill_destroy(plan):
    lib().moe_prefill_destroy(plan)


def moe_prefill_set_profiling(plan, enable: bool):
    _check(lib().moe_prefill_set_profiling(plan, 1 if enable else 0))


def moe_prefill_kernel_times(plan):
    ms = (ctypes.c_double * KERNEL_KINDS)()
    n = (ctypes.c_int64 * KERNEL_KINDS)()
    _check(lib().moe_prefill_kernel_times(plan, ms, n))
    return {KERNEL_NAMES[i]: (ms[i], n[i]) for i in range(KERNEL_KINDS)}


def moe_prefill_kernel_trace(plan, capacity: int = 4096):
    """[(kind name, start ms, end ms)] of the launches timed since the last call, in enqueue order."""
    kinds = (ctypes.c_int32 * capacity)()
    t0 = (ctypes.c_float * capacity)()
    t1 = (ctypes.c_float * capacity)()
    n = ctypes.c_int32(0)
    _check(lib().moe_prefill_kernel_trace(plan, kinds, t0, t1, capacity, ctypes.byref(n)))
    return [(KERNEL_NAMES[kinds[i]], t0[i], t1[i]) for i in range(min(n.value, capacity))]


def moe_prefill_launch_count(plan) -> int:
    return int(lib().moe_prefill_launch_count(plan))


def moe_prefill_set_wait_timeout(plan, timeout_ns: int):
    _check(lib().moe_prefill_set_wait_timeout(plan, timeout_ns))


STATS_NAMES = ["chunks", "flagged", "by_float", "by_double", "by_sequential", "by_many", "experts_copied",
               "experts_skipped", "experts_hot"]


def moe_prefill_run_stats(workspace, stream=None) -> dict:
    arr = (ctypes.c_int32 * len(STATS_NAMES))()
    _check(lib().moe_prefill_run_stats(workspace, stream, arr, len(STATS_NAMES)))
    return dict(zip(STATS_NAMES, arr))


def moe_prefill_debug_gemm(a, b, c, m, n, k_dim, epilogue, err_word, stall_flag=None, timeout_ns=0, stream=None):
    _check(lib().moe_prefill_debug_gemm(a, b, c, m, n, k_dim, epilogue, err_word, stall_flag, timeout_ns, stream))


def moe_prefill_debug_gemm_pairs_scratch(m, n, epilogue) -> int:
    return int(lib().moe_prefill_debug_gemm_pairs_scratch(m, n, epilogue))


def moe_prefill_debug_gemm_pairs(a, b, c, m, n, k_dim, epilogue, scratch, scratch_bytes, err_word, stall_flag=None,
                                 timeout_ns=0, stream=None):
    _check(lib().moe_prefill_debug_gemm_pairs(a, b, c, m, n, k_dim, epilogue, scratch, scratch_bytes, err_word,
                                              stall_flag, timeout_ns, stream))


# ---------------------------------------------------------------------------------------------------- torch helper

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


class MoePrefill:
    """One MoE layer bound to device weights (torch bf16 tensors), with its workspace.

    weights: dict with w_router [E][H], w_gu [E][2I][H], w_down [E][H][I] and optionally ws_gu [2I_s][H],
    ws_down [H][I_s], all bf16 CUDA tensors; with offload_slots > 0, w_gu and w_down are pinned CPU tensors.
    Block-scaled routed experts: instead of w_gu / w_down, uint8 tensors w_gu_q / w_gu_s / w_down_q / w_down_s —
    weight_format "mxfp8": E4M3 codes [E][2I][H], [E][H][I] with E8M0 scales [E][H/32][2I], [E][I/32][H];
    weight_format "nvfp4": E2M1 codes two per byte [E][2I][H/2], [E][H][I/2] with E4M3 scales [E][H/16][2I],
    [E][I/16][H]. Codes are CUDA tensors (pinned CPU with offload_slots), scales CUDA tensors.
    """

    def __init__(self, weights: dict, top_k: int, max_chunk: int, offload_slots: int = 0,
                 weight_format: Optional[str] = None):
        import torch
        wr = weights["w_router"]
        wsg, wsd = weights.get("ws_gu"), weights.get("ws_down")
        self.block_scaled = "w_gu_q" in weights
        self.weight_format = weight_format or ("mxfp8" if self.block_scaled else "bf16")
        if self.weight_format not in ("bf16", "mxfp8", "nvfp4") or (self.weight_format != "bf16") != self.block_scaled:
            raise ValueError("weight_format must be 'mxfp8' or 'nvfp4' with w_gu_q/... weights, 'bf16' without")
        if self.block_scaled:
            wgu, wd = weights["w_gu_q"], weights["w_down_q"]
            for t in (weights["w_gu_s"], weights["w_down_s"]) + (() if offload_slots else (wgu, wd)):
                if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
                    raise ValueError("block-scaled codes and scales must be contiguous uint8 CUDA tensors")
        else:
            wgu, wd = weights["w_gu"], weights["w_down"]
        for t in (wr, wsg, wsd) + (() if (offload_slots or self.block_scaled) else (wgu, wd)):
            if t is not None and (t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous()):
                raise ValueError("weights must be contiguous bf16 CUDA tensors")
        if offload_slots:
            want = torch.uint8 if self.block_scaled else torch.bfloat16
            for t in (wgu, wd):
                if t.dtype != want or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
                    raise ValueError("offloaded expert banks must be contiguous pinned CPU tensors")
        E, H = wr.shape
        I = wgu.shape[1] // 2  # rows of w_gu are 2I in every format
        Is = wsg.shape[0] // 2 if wsg is not None else 0
        self.dims = moe_dims(H, E, I, top_k, Is, 1, max_chunk, offload_slots)
        self.weights = weights  # keep alive: the plan points at them
        if self.block_scaled:
            self.plan, self.workspace_bytes = moe_prefill_plan_mxfp8(
                self.dims, wr.data_ptr(), wgu.data_ptr(), weights["w_gu_s"].data_ptr(), wd.data_ptr(),
                weights["w_down_s"].data_ptr(), _ptr(wsg), _ptr(wsd), fmt=self.weight_format)
        else:
            self.plan, self.workspace_bytes = moe_prefill_plan(self.dims, wr.data_ptr(), wgu.data_ptr(),
                                                               wd.data_ptr(), _ptr(wsg), _ptr(wsd))
        self._workspace = None
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=wr.device)
        self.hidden, self.n_experts, self.top_k = H, E, top_k

    @property
    def workspace(self):
        return self._workspace

    @workspace.setter
    def workspace(self, ws):
        # the library's record of the workspace being replaced is dropped before torch may reuse its memory
        old = getattr(self, "_workspace", None)
        if old is not None and old is not ws:
            moe_prefill_forget_workspace(old.data_ptr())
        self._workspace = ws

    def __del__(self):
        ws = getattr(self, "_workspace", None)
        if ws is not None and _lib is not None:
            try:
                moe_prefill_forget_workspace(ws.data_ptr())
            except Exception:
                pass
        plan = getattr(self, "plan", None)
        if plan:
            moe_prefill_destroy(plan)
            self.plan = None

    def run(self, x, chunk: int, out=None, topk_id=None, topk_w=None, expert_offsets=None, row_token=None,
            stream=None, copy_stream=None):
        import torch
        if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
            raise ValueError("x must be a contiguous bf16 CUDA tensor")
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        moe_prefill_run(self.plan, x.data_ptr(), T, chunk, self.workspace.data_ptr(), self.workspace_bytes,
                        out.data_ptr(), _ptr(topk_id), _ptr(topk_w), _ptr(expert_offsets), _ptr(row_token),
                        _stream_handle(stream), copy_stream.cuda_stream if copy_stream is not None else None)
        return out

    def set_offload_copy(self, mode: int):
        """OFFLOAD_COPY_ROUTED (stage only routed experts; default where available) or OFFLOAD_COPY_ALL."""
        moe_prefill_set_offload_copy(self.plan, mode)

    def set_hot_experts(self, hot_ids):
        """Keeps these offloaded experts resident (staged once); grows the workspace when the set needs it."""
        import torch
        need = moe_prefill_set_hot_experts(self.plan, hot_ids)
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.workspace.device)
        self.workspace_bytes = need

    def prefetch(self, copy_stream=None):
        """Stages the first window of experts of this layer's next run now (offloaded experts only)."""
        _check(lib().moe_prefill_prefetch(self.plan, self.workspace.data_ptr(), self.workspace_bytes,
                                          copy_stream.cuda_stream if copy_stream is not None else None))

    def set_combine(self, mode: int):
        """COMBINE_F32 (canonical float32, ascending expert id; default) or COMBINE_F64_TREE."""
        moe_prefill_set_combine(self.plan, mode)

    @property
    def cta_pairs(self) -> int:
        """Mask of the projections on CTA pairs (PAIRS_GATE_UP | PAIRS_DOWN; PAIRS_GATE_UP by default where the
        dimensions allow it); settable."""
        return moe_prefill_cta_pairs(self.plan)

    @cta_pairs.setter
    def cta_pairs(self, which: int):
        moe_prefill_set_cta_pairs(self.plan, which)

    def run_host(self, x_host, chunk: int, x_dev, out_dev, out_host, topk_id=None, topk_w=None,
                 expert_offsets=None, row_token=None, stream=None, copy_stream=None):
        """The layer on pinned host activations: X rows in, out rows back, overlapped with the compute.
        x_dev / out_dev are device staging tensors shaped like x_host."""
        import torch
        for t, where in ((x_host, "host"), (out_host, "host"), (x_dev, "dev"), (out_dev, "dev")):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.is_cuda != (where == "dev"):
                raise ValueError("run_host needs contiguous bf16 pinned host x/out and device staging tensors")
        T = x_host.shape[0]
        _check(lib().moe_prefill_run_host(self.plan, x_host.data_ptr(), T, chunk, self.workspace.data_ptr(),
                                          self.workspace_bytes, x_dev.data_ptr(), out_dev.data_ptr(),
                                          out_host.data_ptr(), _ptr(topk_id), _ptr(topk_w), _ptr(expert_offsets),
                                          _ptr(row_token), _stream_handle(stream),
                                          copy_stream.cuda_stream if copy_stream is not None else None))
        return out_host

    def check(self, stream=None) -> int:
        return moe_prefill_check(self.workspace.data_ptr(), _stream_handle(stream))

    def raise_on_device_error(self, stream=None):
        st = self.check(stream)
        if st != MOE_OK:
            raise MoeError(st, moe_prefill_last_error())

    def stats(self, stream=None):
        return moe_prefill_run_stats(self.workspace.data_ptr(), _stream_handle(stream))
