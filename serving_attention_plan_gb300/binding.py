"""Thin ctypes binding of the C ABI in include/fi.h (argument marshalling only).

Every step of the attention path runs inside the compiled library; this module
only converts numpy / torch arguments into pointers and sizes.  Loading fails
loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_void_p

import numpy as np

from . import build as _build

FI_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "capacity", 3: "unsupported", 4: "cuda", 5: "device", 6: "no plan"}
DEVERR_PAGE_OOB = 0x1
DEVERR_WAIT_TIMEOUT = 0x2
DEVERR_TMEM = 0x4

_LIB = None


class FiError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load the built library (raises if it is missing; run build() first)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"library not built: {path} is missing (call serving_attention_plan_gb300.build.build())")
    L = ctypes.CDLL(path)
    P32 = POINTER(c_int32)
    L.fi_workspace_create.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, c_int, POINTER(c_void_p)]
    L.fi_workspace_destroy.argtypes = [c_void_p]
    L.fi_workspace_set_cost_model.argtypes = [c_void_p, c_int64, c_int64, c_int32]
    L.fi_workspace_set_variant.argtypes = [c_void_p, c_int32, ctypes.c_float, c_int32]
    L.fi_workspace_set_kv_dtype.argtypes = [c_void_p, c_int32, ctypes.c_float, ctypes.c_float]
    L.fi_plan.argtypes = [c_void_p, P32, P32, P32, P32, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]
    L.fi_plan_composable.argtypes = [c_void_p, P32, P32, P32, P32, c_int, P32, P32, P32, P32, c_int, c_int, c_int,
                                     c_int, c_int, c_int, c_void_p]
    L.fi_run.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]
    L.fi_run_merge.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p]
    L.fi_merge_states.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                  c_void_p]
    L.fi_get_error.argtypes = [c_void_p, P32]
    L.fi_plan_info.argtypes = [c_void_p, P32]
    L.fi_plan_compute.argtypes = [P32, P32, P32, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int64, c_int64,
                                  c_int32, c_int32, P32, c_int64, POINTER(c_int64)]
    L.fi_plan_composable_compute.argtypes = [P32, P32, P32, c_int, P32, P32, P32, c_int, c_int, c_int, c_int, c_int,
                                             c_int, c_int, P32, c_int64, POINTER(c_int64)]
    L.fi_decode_noalloc.argtypes = [P32, P32, P32, P32, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                    c_void_p, c_int, c_void_p, c_void_p, c_void_p]
    L.fi_decode_noalloc_get_error.argtypes = [P32]
    L.fi_device_sm_count.argtypes = [POINTER(c_int)]
    L.fi_status_string.argtypes = [c_int]
    L.fi_status_string.restype = ctypes.c_char_p
    L.fi_last_error_message.argtypes = []
    L.fi_last_error_message.restype = ctypes.c_char_p
    for name in ("fi_workspace_create", "fi_workspace_destroy", "fi_workspace_set_cost_model",
                 "fi_workspace_set_variant", "fi_workspace_set_kv_dtype", "fi_plan", "fi_run",
                 "fi_run_merge", "fi_merge_states", "fi_get_error", "fi_plan_info", "fi_plan_compute", "fi_device_sm_count",
                 "fi_decode_noalloc", "fi_decode_noalloc_get_error", "fi_plan_composable_compute",
                 "fi_plan_composable"):
        getattr(L, name).restype = c_int
    _LIB = L
    return L


def _check(st: int, what: str):
    if st != FI_OK:
        detail = lib().fi_last_error_message().decode() if st == 4 else ""
        raise FiError(st, what, detail)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(POINTER(c_int32))


def _stream_ptr(stream) -> c_void_p:
    if stream is None:
        import torch
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return c_void_p(stream)
    return c_void_p(stream.cuda_stream)


def _dptr(t) -> c_void_p:
    return c_void_p(0 if t is None else t.data_ptr())


def plan_compute(qo_indptr, kv_indptr, last_page_len, num_qo_heads, num_kv_heads, page_size, causal, num_sms,
                 head_dim=128, alpha=1, beta=1, l_min=256, window_left=-1) -> np.ndarray:
    """The host planner alone (no GPU): returns the flat int32 plan."""
    L = lib()
    qo, kv, last = _i32(qo_indptr), _i32(kv_indptr), _i32(last_page_len)
    batch = qo.shape[0] - 1
    n = c_int64(0)
    st = L.fi_plan_compute(_p32(qo), _p32(kv), _p32(last), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                           int(causal), num_sms, alpha, beta, l_min, window_left, None, 0, ctypes.byref(n))
    if st not in (FI_OK, 2):
        _check(st, "fi_plan_compute")
    out = np.zeros(max(int(n.value), 1), dtype=np.int32)
    st = L.fi_plan_compute(_p32(qo), _p32(kv), _p32(last), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                           int(causal), num_sms, alpha, beta, l_min, window_left, _p32(out), out.shape[0],
                           ctypes.byref(n))
    _check(st, "fi_plan_compute")
    return out[: n.value]


def plan_composable_compute(shared, unique, num_qo_heads, num_kv_heads, page_size, causal, num_sms,
                            head_dim=128) -> np.ndarray:
    """The composable planner alone (no GPU): shared and unique are (qo_indptr, kv_indptr, last_page_len)."""
    L = lib()
    sq, sk, sl = (_i32(x) for x in shared)
    uq, uk, ul = (_i32(x) for x in unique)
    n = c_int64(0)
    args = [_p32(sq), _p32(sk), _p32(sl), sq.shape[0] - 1, _p32(uq), _p32(uk), _p32(ul), uq.shape[0] - 1,
            num_qo_heads, num_kv_heads, head_dim, page_size, int(causal), num_sms]
    st = L.fi_plan_composable_compute(*args, None, 0, ctypes.byref(n))
    if st not in (FI_OK, 2):
        _check(st, "fi_plan_composable_compute")
    out = np.zeros(max(int(n.value), 1), dtype=np.int32)
    _check(L.fi_plan_composable_compute(*args, _p32(out), out.shape[0], ctypes.byref(n)), "fi_plan_composable_compute")
    return out[: n.value]


def device_sm_count() -> int:
    v = c_int(0)
    _check(lib().fi_device_sm_count(ctypes.byref(v)), "fi_device_sm_count")
    return v.value


class Workspace:
    """Owns one fi_workspace (device + pinned buffers) at fixed capacity."""

    def __init__(self, max_batch, max_total_q, max_kv_pages, num_qo_heads, num_kv_heads, head_dim=128, num_sms=0):
        self._h = c_void_p(0)
        _check(lib().fi_workspace_create(max_batch, max_total_q, max_kv_pages, num_qo_heads, num_kv_heads, head_dim,
                                         num_sms, ctypes.byref(self._h)), "fi_workspace_create")
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim

    def close(self):
        if self._h:
            lib().fi_workspace_destroy(self._h)
            self._h = c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_cost_model(self, alpha=1, beta=1, l_min=256):
        _check(lib().fi_workspace_set_cost_model(self._h, alpha, beta, l_min), "fi_workspace_set_cost_model")

    def set_variant(self, window_left=-1, logits_soft_cap=0.0, kv_layout="HND"):
        """Sliding window / logit soft-cap / page layout ("HND" or "NHD") for the following plan()."""
        layout = {"HND": 0, "NHD": 1}[kv_layout]
        _check(lib().fi_workspace_set_variant(self._h, int(window_left), float(logits_soft_cap), layout),
               "fi_workspace_set_variant")

    def set_kv_dtype(self, kv_dtype="bf16", k_scale=1.0, v_scale=1.0):
        """KV page element type ("bf16" or "e4m3", with per-tensor scales) for the following plan()."""
        _check(lib().fi_workspace_set_kv_dtype(self._h, {"bf16": 0, "e4m3": 1}[kv_dtype], float(k_scale),
                                               float(v_scale)), "fi_workspace_set_kv_dtype")

    def plan(self, qo_indptr, kv_indptr, kv_indices, last_page_len, page_size, causal, stream=None):
        qo, kv, idx, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
        if idx.size == 0:
            idx = np.zeros(1, np.int32)
        _check(lib().fi_plan(self._h, _p32(qo), _p32(kv), _p32(idx), _p32(last), qo.shape[0] - 1, self.num_qo_heads,
                             self.num_kv_heads, self.head_dim, page_size, int(causal), _stream_ptr(stream)), "fi_plan")

    def plan_composable(self, shared, unique, page_size, causal, stream=None):
        """Composable plan: shared and unique are (qo_indptr, kv_indptr, kv_indices, last_page_len)."""
        sq, sk, si, sl = (_i32(x) for x in shared)
        uq, uk, ui, ul = (_i32(x) for x in unique)
        si = si if si.size else np.zeros(1, np.int32)
        ui = ui if ui.size else np.zeros(1, np.int32)
        _check(lib().fi_plan_composable(self._h, _p32(sq), _p32(sk), _p32(si), _p32(sl), sq.shape[0] - 1, _p32(uq),
                                        _p32(uk), _p32(ui), _p32(ul), uq.shape[0] - 1, self.num_qo_heads,
                                        self.num_kv_heads, self.head_dim, page_size, int(causal), _stream_ptr(stream)),
               "fi_plan_composable")

    def run(self, q, k_pages, v_pages, o, lse, stream=None):
        _check(lib().fi_run(self._h, _dptr(q), _dptr(k_pages), _dptr(v_pages), int(k_pages.shape[0]), _dptr(o),
                            _dptr(lse), _stream_ptr(stream)), "fi_run")

    def run_merge(self, q, k_pages, v_pages, o_prev, lse_prev, o, lse, stream=None):
        """fi_run with each output row merged (⊕) into the state (o_prev, lse_prev); o may be o_prev."""
        _check(lib().fi_run_merge(self._h, _dptr(q), _dptr(k_pages), _dptr(v_pages), int(k_pages.shape[0]),
                                  _dptr(o_prev), _dptr(lse_prev), _dptr(o), _dptr(lse), _stream_ptr(stream)),
               "fi_run_merge")

    def info(self) -> np.ndarray:
        h = np.zeros(16, np.int32)
        _check(lib().fi_plan_info(self._h, _p32(h)), "fi_plan_info")
        return h

    def get_error(self) -> int:
        e = np.zeros(1, np.int32)
        _check(lib().fi_get_error(self._h, _p32(e)), "fi_get_error")
        return int(e[0])

    @property
    def handle(self) -> int:
        return self._h.value


def decode_noalloc(qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads, num_kv_heads, page_size, causal,
                   q, k_pages, v_pages, o, lse, stream=None, head_dim=128):
    """Plan and run one decode batch with no workspace (the library's static scratch array)."""
    qo, kv, idx, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    if idx.size == 0:
        idx = np.zeros(1, np.int32)
    _check(lib().fi_decode_noalloc(_p32(qo), _p32(kv), _p32(idx), _p32(last), qo.shape[0] - 1, num_qo_heads,
                                   num_kv_heads, head_dim, page_size, int(causal), _dptr(q), _dptr(k_pages),
                                   _dptr(v_pages), int(k_pages.shape[0]), _dptr(o), _dptr(lse), _stream_ptr(stream)),
           "fi_decode_noalloc")


def decode_noalloc_get_error() -> int:
    """Read and clear the device-side error bits of the allocation-free entry point (synchronises)."""
    e = np.zeros(1, np.int32)
    _check(lib().fi_decode_noalloc_get_error(_p32(e)), "fi_decode_noalloc_get_error")
    return int(e[0])


def merge_states(o_a, lse_a, o_b, lse_b, o, lse, stream=None):
    rows, heads, d = o.shape
    _check(lib().fi_merge_states(_dptr(o_a), _dptr(lse_a), _dptr(o_b), _dptr(lse_b), _dptr(o), _dptr(lse), rows, heads,
                                 d, _stream_ptr(stream)), "fi_merge_states")
