"""Python binding of the ditango C ABI (include/ditango.h): argument marshalling only.

Partitioned attention with attention-state reuse (DiTango, gist.science/paper/2607.15650,
Methodology 1-2) on one GB300 (sm_103a). Every computation runs in the library's CUDA
kernels; PyTorch supplies device memory and streams. There is no fallback: if the compiled
library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build  # noqa: F401  (re-exported for users who build in place)

__all__ = [
    "DitangoError", "Plan", "attn_step", "merge", "workspace_size", "RopeTables",
    "device_status", "new_state_cache", "new_group_state", "load_library", "SYMBOLS",
    "planner_importance", "planner_snapshot", "planner_drift", "planner_select", "AnchorPlanner",
    "new_host_states", "cache_slot_map",
]

F32, BF16 = 0, 1
MAX_PARTITIONS = 64
MAX_STATES = 64

STATUS = {
    0: "OK", 1: "INVALID_ARG", 2: "INVALID_MASK", 3: "NO_CACHE", 4: "SHAPE", 5: "DTYPE",
    6: "ALIGN", 7: "WORKSPACE", 8: "CUDA", 9: "DEVICE_TIMEOUT", 10: "UNSUPPORTED",
}

# every entry point declared in include/ditango.h
SYMBOLS = [
    "ditango_plan", "ditango_plan_destroy", "ditango_plan_set_mask", "ditango_plan_check_mask",
    "ditango_plan_get_offsets", "ditango_plan_get_pairs", "ditango_plan_get_cache_state",
    "ditango_plan_set_cache_state",
    "ditango_plan_set_profile_events", "ditango_plan_inject_fault",
    "ditango_planner_importance", "ditango_planner_snapshot", "ditango_planner_drift",
    "ditango_planner_select",
    "ditango_attn_step", "ditango_attn_step_static_workspace",
    "ditango_attn_step_workspace_size", "ditango_merge",
    "ditango_rope_build_tables", "ditango_device_status", "ditango_status_string",
    "ditango_version", "ditango_cache_slot_map",
]


class DitangoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_lib().ditango_status_string(status).decode()})")


class Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class StateCache(ctypes.Structure):
    _fields_ = [("O", Tensor), ("lse", Tensor), ("group_O", Tensor), ("group_lse", Tensor),
                ("host_O", Tensor), ("host_lse", Tensor)]


def _state_cache(cache_O, cache_lse, group, host=None):
    c = StateCache(tensor_desc(cache_O), tensor_desc(cache_lse))
    if group is not None:
        c.group_O = tensor_desc(group[0])
        c.group_lse = tensor_desc(group[1])
    if host is not None:
        c.host_O = host_tensor_desc(host[0])
        c.host_lse = host_tensor_desc(host[1])
    return c


class Rope(ctypes.Structure):
    _fields_ = [("cos_t", ctypes.c_void_p), ("sin_t", ctypes.c_void_p),
                ("cos_h", ctypes.c_void_p), ("sin_h", ctypes.c_void_p),
                ("cos_w", ctypes.c_void_p), ("sin_w", ctypes.c_void_p),
                ("T_tab", ctypes.c_int64), ("Hl", ctypes.c_int64), ("Wl", ctypes.c_int64),
                ("dt", ctypes.c_int32), ("dh", ctypes.c_int32), ("dw", ctypes.c_int32),
                ("start_frame", ctypes.c_int64),
                ("cos_t_lo", ctypes.c_void_p), ("sin_t_lo", ctypes.c_void_p),
                ("cos_h_lo", ctypes.c_void_p), ("sin_h_lo", ctypes.c_void_p),
                ("cos_w_lo", ctypes.c_void_p), ("sin_w_lo", ctypes.c_void_p)]


class StateList(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("O", ctypes.POINTER(ctypes.c_void_p)), ("lse", ctypes.POINTER(ctypes.c_void_p)),
                ("shape", ctypes.c_int64 * 4), ("O_stride", ctypes.c_int64 * 3),
                ("lse_stride", ctypes.c_int64 * 3)]


_LIB = None
_LOCK = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the compiled library (raises OSError if it has not been built)."""
    if not os.path.exists(path):
        raise OSError(f"ditango library not built: {path} is missing "
                      "(run attention_state_reuse_gb300.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp, i32, i64, u8p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, P(ctypes.c_uint8)
    lib.ditango_plan.argtypes = [i64, i32, u8p, P(vp)]
    lib.ditango_plan_destroy.argtypes = [vp]
    lib.ditango_plan_destroy.restype = None
    lib.ditango_plan_set_mask.argtypes = [vp, u8p]
    lib.ditango_plan_check_mask.argtypes = [vp, u8p]
    lib.ditango_plan_get_offsets.argtypes = [vp, P(i64)]
    lib.ditango_plan_get_pairs.argtypes = [vp, u8p, P(i32), P(i32)]
    lib.ditango_plan_get_cache_state.argtypes = [vp, u8p, P(i64), P(i64)]
    lib.ditango_plan_set_cache_state.argtypes = [vp, u8p, P(i64), i64]
    lib.ditango_plan_set_profile_events.argtypes = [vp, P(vp)]
    lib.ditango_plan_inject_fault.argtypes = [vp, ctypes.c_int32]
    dp = P(ctypes.c_double)
    lib.ditango_planner_importance.argtypes = [vp, P(StateCache), vp, vp]
    lib.ditango_planner_snapshot.argtypes = [vp, P(StateCache), P(Tensor), vp]
    lib.ditango_planner_drift.argtypes = [vp, P(StateCache), P(Tensor), vp, vp]
    lib.ditango_planner_select.argtypes = [vp, dp, dp, ctypes.c_double, i32, i32, u8p]
    lib.ditango_attn_step.argtypes = [vp, P(Tensor), P(Tensor), P(Tensor), P(Rope), u8p,
                                      P(StateCache), P(Tensor), P(Tensor), ctypes.c_float, vp,
                                      ctypes.c_size_t, vp]
    lib.ditango_attn_step_static_workspace.argtypes = [vp, P(Tensor), P(Tensor), P(Tensor),
                                                       P(Rope), u8p, P(StateCache), P(Tensor),
                                                       P(Tensor), ctypes.c_float, vp]
    lib.ditango_attn_step_workspace_size.argtypes = [vp, i64, i64, i32, i32, i32]
    lib.ditango_attn_step_workspace_size.restype = ctypes.c_size_t
    lib.ditango_merge.argtypes = [P(StateList), P(Tensor), P(Tensor), vp]
    lib.ditango_rope_build_tables.argtypes = [P(Rope), ctypes.c_double, vp]
    lib.ditango_device_status.argtypes = [vp, P(i32)]
    lib.ditango_status_string.argtypes = [ctypes.c_int]
    lib.ditango_status_string.restype = ctypes.c_char_p
    lib.ditango_version.argtypes = []
    lib.ditango_cache_slot_map.argtypes = [i32, i32, P(ctypes.c_int8)]
    return lib


def _lib() -> ctypes.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = load_library()
        return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DitangoError(status, where)


def _mask_ptr(mask, P):
    """Host P*P uint8 buffer (kept alive by the returned array) or None."""
    if mask is None:
        return None, None
    import numpy as np

    arr = np.ascontiguousarray(np.asarray(mask), dtype=np.uint8)
    if arr.size != P * P:
        raise ValueError(f"reuse mask must hold {P}x{P} entries")
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def tensor_desc(t) -> Tensor:
    """ditango_tensor describing a CUDA torch tensor (no copy)."""
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must live on a CUDA device")
    d = Tensor()
    d.ptr = t.data_ptr()
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for a in range(t.dim()):
        d.shape[a] = t.shape[a]
        d.stride[a] = t.stride(a)
    return d


def host_tensor_desc(t) -> Tensor:
    """ditango_tensor describing a page-locked (pinned) CPU torch tensor (no copy)."""
    if t.is_cuda or not t.is_pinned():
        raise ValueError("host storage must be a pinned CPU tensor")
    d = Tensor()
    d.ptr = t.data_ptr()
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for a in range(t.dim()):
        d.shape[a] = t.shape[a]
        d.stride[a] = t.stride(a)
    return d


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Partition plan and per-pair cache bookkeeping (ditango_plan)."""

    def __init__(self, N: int, P: int, mask=None):
        self.N, self.P = int(N), int(P)
        h = ctypes.c_void_p()
        arr, ptr = _mask_ptr(mask, self.P)
        _check(_lib().ditango_plan(self.N, self.P, ptr, ctypes.byref(h)), "ditango_plan")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib().ditango_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def offsets(self):
        import numpy as np

        out = np.zeros(self.P + 1, dtype=np.int64)
        _check(_lib().ditango_plan_get_offsets(self._h, out.ctypes.data_as(
            ctypes.POINTER(ctypes.c_int64))), "ditango_plan_get_offsets")
        return out

    def pairs(self, mask=None):
        import numpy as np

        buf = np.zeros(2 * self.P * self.P, dtype=np.int32)
        cnt = ctypes.c_int32()
        arr, ptr = _mask_ptr(mask, self.P)
        _check(_lib().ditango_plan_get_pairs(self._h, ptr, buf.ctypes.data_as(
            ctypes.POINTER(ctypes.c_int32)), ctypes.byref(cnt)), "ditango_plan_get_pairs")
        return [tuple(x) for x in buf[: 2 * cnt.value].reshape(-1, 2).tolist()]

    def cache_state(self):
        import numpy as np

        valid = np.zeros(self.P * self.P, dtype=np.uint8)
        sc = np.zeros(self.P * self.P, dtype=np.int64)
        steps = ctypes.c_int64()
        _check(_lib().ditango_plan_get_cache_state(
            self._h, valid.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
            sc.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.byref(steps)),
            "ditango_plan_get_cache_state")
        return valid.reshape(self.P, self.P), sc.reshape(self.P, self.P), steps.value

    def set_cache_state(self, valid, step_computed, steps_run: int) -> None:
        """Restores the cache bookkeeping (e.g. with a state cache restored from a checkpoint)."""
        import numpy as np

        v = np.ascontiguousarray(np.asarray(valid), dtype=np.uint8).reshape(-1)
        sc = np.ascontiguousarray(np.asarray(step_computed), dtype=np.int64).reshape(-1)
        if v.size != self.P * self.P or sc.size != self.P * self.P:
            raise ValueError("valid and step_computed must hold P*P entries")
        _check(_lib().ditango_plan_set_cache_state(
            self._h, v.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
            sc.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(steps_run)),
            "ditango_plan_set_cache_state")

    def set_mask(self, mask):
        arr, ptr = _mask_ptr(mask, self.P)
        _check(_lib().ditango_plan_set_mask(self._h, ptr), "ditango_plan_set_mask")

    def inject_fault(self, kind=1):
        """Arms (1) or disarms (0) the one-shot device-timeout test fault of the next bf16 step."""
        _check(_lib().ditango_plan_inject_fault(self._h, int(kind)), "ditango_plan_inject_fault")

    def set_profile_events(self, events):
        """Four torch.cuda.Event(enable_timing=True) recorded around the step's kernels, or None."""
        if events is None:
            _check(_lib().ditango_plan_set_profile_events(self._h, None), "set_profile_events")
            return
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        _check(_lib().ditango_plan_set_profile_events(self._h, arr), "set_profile_events")

    def check_mask(self, mask=None) -> int:
        """Status code of a mask against the bookkeeping (0 = usable)."""
        arr, ptr = _mask_ptr(mask, self.P)
        return _lib().ditango_plan_check_mask(self._h, ptr)


def new_state_cache(B, H, P, N, d, dtype, device="cuda"):
    """Allocates an uninitialised state cache: O [B, H, P, N, d] and lse [B, H, P, N] fp32."""
    import torch

    O = torch.empty((B, H, P, N, d), dtype=dtype, device=device)
    lse = torch.empty((B, H, P, N), dtype=torch.float32, device=device)
    return O, lse


def new_host_states(B, H, P, N, d, dtype):
    """Allocates host storage for a state cache whose device part keeps S < P slots per row:
    O [B, H, P, N, d] and lse [B, H, P, N] fp32 in page-locked host memory. Pass them as
    `host=` to attn_step (and the planner calls) together with a device cache made by
    new_state_cache(B, H, S, N, d, ...)."""
    import torch

    O = torch.empty((B, H, P, N, d), dtype=dtype, pin_memory=True)
    lse = torch.empty((B, H, P, N), dtype=torch.float32, pin_memory=True)
    return O, lse


def cache_slot_map(P: int, S: int):
    """[P, P] int8 numpy array: the device slot of pair (i, j) when the device cache keeps S
    of the P states per row, -1 for a pair kept in host storage (ditango_cache_slot_map)."""
    import numpy as np

    out = np.empty(P * P, dtype=np.int8)
    _check(_lib().ditango_cache_slot_map(int(P), int(S), out.ctypes.data_as(
        ctypes.POINTER(ctypes.c_int8))), "ditango_cache_slot_map")
    return out.reshape(P, P)


def new_group_state(B, H, N, d, device="cuda"):
    """Allocates the optional group states of a cache: O [B, H, N, d] and lse [B, H, N], fp32.
    Pass them as `group=` to attn_step with the same plan every step."""
    import torch

    O = torch.empty((B, H, N, d), dtype=torch.float32, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    return O, lse


def workspace_size(plan: Plan, B: int, H: int, d: int, dtype, use_rope: bool) -> int:
    import torch

    code = BF16 if dtype == torch.bfloat16 else F32
    return _lib().ditango_attn_step_workspace_size(plan.handle, B, H, d, code, int(bool(use_rope)))


class RopeTables:
    """Device cos/sin tables of the 3D RoPE (filled by the library's table kernel)."""

    def __init__(self, T_tab, Hl, Wl, dt, dh, dw, start_frame=0, theta=10000.0, device="cuda",
                 stream=None):
        import torch

        self.T_tab, self.Hl, self.Wl = int(T_tab), int(Hl), int(Wl)
        self.dt, self.dh, self.dw = int(dt), int(dh), int(dw)
        self.start_frame = int(start_frame)
        f = dict(dtype=torch.float32, device=device)
        self.cos_t = torch.empty((self.T_tab, self.dt // 2), **f)
        self.sin_t = torch.empty_like(self.cos_t)
        self.cos_h = torch.empty((self.Hl, self.dh // 2), **f)
        self.sin_h = torch.empty_like(self.cos_h)
        self.cos_w = torch.empty((self.Wl, self.dw // 2), **f)
        self.sin_w = torch.empty_like(self.cos_w)
        # residuals: table + residual carries cos and sin to about 48 bits
        self.cos_t_lo, self.sin_t_lo = torch.empty_like(self.cos_t), torch.empty_like(self.cos_t)
        self.cos_h_lo, self.sin_h_lo = torch.empty_like(self.cos_h), torch.empty_like(self.cos_h)
        self.cos_w_lo, self.sin_w_lo = torch.empty_like(self.cos_w), torch.empty_like(self.cos_w)
        s = self.struct()
        _check(_lib().ditango_rope_build_tables(ctypes.byref(s), float(theta), _stream_ptr(stream)),
               "ditango_rope_build_tables")

    def struct(self) -> Rope:
        r = Rope()
        r.cos_t, r.sin_t = self.cos_t.data_ptr(), self.sin_t.data_ptr()
        r.cos_h, r.sin_h = self.cos_h.data_ptr(), self.sin_h.data_ptr()
        r.cos_w, r.sin_w = self.cos_w.data_ptr(), self.sin_w.data_ptr()
        r.T_tab, r.Hl, r.Wl = self.T_tab, self.Hl, self.Wl
        r.dt, r.dh, r.dw = self.dt, self.dh, self.dw
        r.start_frame = self.start_frame
        r.cos_t_lo, r.sin_t_lo = self.cos_t_lo.data_ptr(), self.sin_t_lo.data_ptr()
        r.cos_h_lo, r.sin_h_lo = self.cos_h_lo.data_ptr(), self.sin_h_lo.data_ptr()
        r.cos_w_lo, r.sin_w_lo = self.cos_w_lo.data_ptr(), self.sin_w_lo.data_ptr()
        return r


def attn_step(plan: Plan, q, k, v, cache_O, cache_lse, out, out_lse=None, reuse_mask=None,
              rope: RopeTables | None = None, softmax_scale: float | None = None, workspace=None,
              stream=None, group=None, host=None) -> None:
    """One attention-layer step (ditango_attn_step), asynchronous on `stream`. `group`: the
    cache's optional group states (new_group_state), or None. `host`: the cache's optional host
    storage (new_host_states) when cache_O keeps fewer than P slots per row, or None."""
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** -0.5
    qd, kd, vd, od = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out)
    cache = _state_cache(cache_O, cache_lse, group, host)
    ld = tensor_desc(out_lse) if out_lse is not None else None
    rs = rope.struct() if rope is not None else None
    arr, mptr = _mask_ptr(reuse_mask, plan.P)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib().ditango_attn_step(
        plan.handle, ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd),
        ctypes.byref(rs) if rs is not None else None, mptr, ctypes.byref(cache), ctypes.byref(od),
        ctypes.byref(ld) if ld is not None else None, ctypes.c_float(softmax_scale), ws_ptr,
        ws_bytes, _stream_ptr(stream))
    _check(st, "ditango_attn_step")


def attn_step_static_workspace(plan: Plan, q, k, v, cache_O, cache_lse, out, out_lse=None,
                               reuse_mask=None, rope: RopeTables | None = None,
                               softmax_scale: float | None = None, stream=None,
                               group=None, host=None) -> None:
    """ditango_attn_step_static_workspace: the step without a caller workspace, for callers
    that cannot allocate device memory; its scratch lives in a 64 MiB array inside the
    library (steps needing more are refused with WORKSPACE). Concurrent calls race on it."""
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** -0.5
    qd, kd, vd, od = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out)
    cache = _state_cache(cache_O, cache_lse, group, host)
    ld = tensor_desc(out_lse) if out_lse is not None else None
    rs = rope.struct() if rope is not None else None
    arr, mptr = _mask_ptr(reuse_mask, plan.P)
    st = _lib().ditango_attn_step_static_workspace(
        plan.handle, ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd),
        ctypes.byref(rs) if rs is not None else None, mptr, ctypes.byref(cache), ctypes.byref(od),
        ctypes.byref(ld) if ld is not None else None, ctypes.c_float(softmax_scale),
        _stream_ptr(stream))
    _check(st, "ditango_attn_step_static_workspace")


def merge(O_states, lse_states, out, out_lse=None, stream=None) -> None:
    """Merges states O_s [G1, G2, R, d] / lse_s [G1, G2, R] (common strides) into out."""
    n = len(O_states)
    if n != len(lse_states) or n < 1:
        raise ValueError("need matching, non-empty lists of O and lse")
    sl = StateList()
    sl.n = n
    sl.dtype = _dtype_code(O_states[0])
    optrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in O_states])
    lptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_states])
    sl.O = ctypes.cast(optrs, ctypes.POINTER(ctypes.c_void_p))
    sl.lse = ctypes.cast(lptrs, ctypes.POINTER(ctypes.c_void_p))
    O0, L0 = O_states[0], lse_states[0]
    for t in O_states:
        if t.shape != O0.shape or t.stride() != O0.stride() or t.dtype != O0.dtype or not t.is_cuda:
            raise ValueError("all O states must share shape, strides, dtype and live on CUDA")
    for t in lse_states:
        if t.shape != L0.shape or t.stride() != L0.stride() or not t.is_cuda:
            raise ValueError("all lse states must share shape and strides and live on CUDA")
    for a in range(4):
        sl.shape[a] = O0.shape[a]
    for a in range(3):
        sl.O_stride[a] = O0.stride(a)
        sl.lse_stride[a] = L0.stride(a)
    od = tensor_desc(out)
    ld = tensor_desc(out_lse) if out_lse is not None else None
    _check(_lib().ditango_merge(ctypes.byref(sl), ctypes.byref(od),
                                ctypes.byref(ld) if ld is not None else None, _stream_ptr(stream)),
           "ditango_merge")


# ---------------------------------------------------------------- anchor-guided planner
def planner_importance(plan: Plan, cache_O, cache_lse, stream=None, host=None):
    """w [P, P] float64 (device): partition j's mean share of partition i's attention mass
    in the cache as it stands (ditango_planner_importance; call after an anchor step)."""
    import torch

    w = torch.empty((plan.P, plan.P), dtype=torch.float64, device=cache_O.device)
    cache = _state_cache(cache_O, cache_lse, None, host)
    _check(_lib().ditango_planner_importance(plan.handle, ctypes.byref(cache),
                                             ctypes.c_void_p(w.data_ptr()), _stream_ptr(stream)),
           "ditango_planner_importance")
    return w


def planner_snapshot(plan: Plan, cache_O, cache_lse, snapshot, stream=None, host=None) -> None:
    """Copies every partition's local states into `snapshot` [B, H, N, d] (cache dtype)."""
    cache = _state_cache(cache_O, cache_lse, None, host)
    sd = tensor_desc(snapshot)
    _check(_lib().ditango_planner_snapshot(plan.handle, ctypes.byref(cache), ctypes.byref(sd),
                                           _stream_ptr(stream)), "ditango_planner_snapshot")


def planner_drift(plan: Plan, cache_O, cache_lse, snapshot, stream=None, host=None):
    """delta [P] float64 (device): relative change of each partition's local states since
    the snapshot."""
    import torch

    buf = torch.empty(2 * plan.P, dtype=torch.float64, device=cache_O.device)
    cache = _state_cache(cache_O, cache_lse, None, host)
    sd = tensor_desc(snapshot)
    _check(_lib().ditango_planner_drift(plan.handle, ctypes.byref(cache), ctypes.byref(sd),
                                        ctypes.c_void_p(buf.data_ptr()), _stream_ptr(stream)),
           "ditango_planner_drift")
    return buf[:plan.P]


def planner_select(plan: Plan, w, delta, tau: float, group: int = 1, budget: int = -1):
    """Reuse mask (numpy uint8 [P, P]) for the next step (ditango_planner_select, host)."""
    import numpy as np

    wa = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    da = np.ascontiguousarray(np.asarray(delta, dtype=np.float64))
    if wa.shape != (plan.P, plan.P) or da.shape != (plan.P,):
        raise ValueError("w must be [P, P] and delta [P]")
    mask = np.empty((plan.P, plan.P), dtype=np.uint8)
    dp = ctypes.POINTER(ctypes.c_double)
    _check(_lib().ditango_planner_select(plan.handle, wa.ctypes.data_as(dp), da.ctypes.data_as(dp),
                                         float(tau), int(group), int(budget),
                                         mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))),
           "ditango_planner_select")
    return mask


class AnchorPlanner:
    """Drives the reuse masks of one layer: every `anchor_every` steps an anchor step computes
    every pair, after which the importance weights are refreshed and the local states are
    snapshotted; on the other steps the drift since the anchor and the weights choose the mask
    (planner_select with tau, group and budget). `host`: the cache's host storage, if any.

    build_ahead: before each anchor after the first, the plan's default mask is set to the
    mask chosen right after the previous anchor, so that the anchor's merge builds those group
    states (ditango_attn_step does so for an all-compute step); when the next choice is the same
    mask, its step finds them current. The masks this class returns are always explicit."""

    def __init__(self, plan: Plan, cache_O, cache_lse, anchor_every: int, tau: float,
                 group: int = 1, budget: int = -1, host=None, build_ahead: bool = True):
        import torch

        self.plan, self.cO, self.cL, self.host = plan, cache_O, cache_lse, host
        self.anchor_every, self.tau, self.group, self.budget = anchor_every, tau, group, budget
        self.build_ahead = build_ahead
        B, H, P, N, d = cache_O.shape
        self.snapshot = torch.empty((B, H, N, d), dtype=cache_O.dtype, device=cache_O.device)
        self.w = None
        self.t = 0
        self._last_anchor = False  # the previous step was an anchor
        self.predicted = None      # the mask chosen right after the last anchor

    def mask(self):
        """Reuse mask for the next step."""
        import numpy as np

        if self.w is None or self.t % self.anchor_every == 0:
            if self.build_ahead and self.predicted is not None:
                self.plan.set_mask(self.predicted)
            return np.zeros((self.plan.P, self.plan.P), np.uint8)
        delta = planner_drift(self.plan, self.cO, self.cL, self.snapshot,
                              host=self.host).cpu().numpy()
        return planner_select(self.plan, self.w, delta, self.tau, self.group, self.budget)

    def after_step(self, mask) -> None:
        """Call after the step that used `mask`: an all-compute step becomes the anchor."""
        import numpy as np

        m = np.asarray(mask)
        if not m.any():
            self.w = planner_importance(self.plan, self.cO, self.cL, host=self.host).cpu().numpy()
            planner_snapshot(self.plan, self.cO, self.cL, self.snapshot, host=self.host)
            self._last_anchor = True
        else:
            if self._last_anchor:
                self.predicted = np.array(m, dtype=np.uint8, copy=True)
            self._last_anchor = False
        self.t += 1


def device_status(stream=None):
    """(status, code): synchronises the stream and reads/clears the kernel timeout word."""
    code = ctypes.c_int32()
    st = _lib().ditango_device_status(_stream_ptr(stream), ctypes.byref(code))
    return st, code.value
