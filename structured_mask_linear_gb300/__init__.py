"""Python binding of libloglinear.so, the C ABI declared in include/loglinear.h.

Argument marshalling only: every step of the forward and of the decode step runs in
the library's CUDA kernels.  Torch tensors supply device memory and the current CUDA
stream.  There is no fallback: if the library cannot be loaded, the calls raise.

Functions mirror the C names:

* ``loglinear_fwd(q, k, v, a, lam, chunk, ...)``  -> o (and optionally the Fenwick
  bucket states at position T)
* ``loglinear_decode_step(pos, q_t, k_t, v_t, a_t, lam_t, states, state_logscale)`` -> o_t
* ``loglinear_fwd_host(...)`` end-to-end from host (pinned) tensors
* ``loglinear_fwd_continue``, ``loglinear_segment_total``, ``loglinear_prefix_states``:
  a forward that starts from the bucket memories at a position T0, and the pieces that
  build those memories from whole earlier segments (see ``sharded`` for a sequence split
  over ranks)
* ``loglinear_fwd_workspace_bytes``, ``loglinear_fwd_path``, ``loglinear_check_status``,
  ``loglinear_selftest_wait_timeout``, ``loglinear_status_string``
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as _LIB_PATH

LL_OK = 0
STATUS_NAMES = {0: "LL_OK", 1: "LL_ERR_NULL", 2: "LL_ERR_SHAPE", 3: "LL_ERR_DTYPE",
                4: "LL_ERR_ALIGN", 5: "LL_ERR_WORKSPACE", 6: "LL_ERR_CUDA", 7: "LL_ERR_TIMEOUT",
                8: "LL_ERR_UNIMPLEMENTED"}
LL_F32, LL_BF16 = 0, 1


class LogLinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({loglinear_status_string(status)})")


class LLShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("T", ctypes.c_int), ("heads", ctypes.c_int),
                ("heads_per_group", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("chunk", ctypes.c_int), ("levels", ctypes.c_int), ("dtype", ctypes.c_int)]


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_SP = ctypes.POINTER(LLShape)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: run __graft_entry__.build() "
                                   "(or python -m structured_mask_linear_gb300._build)")
            L = ctypes.CDLL(_LIB_PATH)
            L.loglinear_status_string.restype = ctypes.c_char_p
            L.loglinear_status_string.argtypes = [ctypes.c_int]
            L.loglinear_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_fwd_workspace_bytes.argtypes = [_SP]
            L.loglinear_fwd_path.restype = ctypes.c_int
            L.loglinear_fwd_path.argtypes = [_SP]
            L.loglinear_fwd.restype = ctypes.c_int
            L.loglinear_fwd.argtypes = [_SP] + [_vp] * 7 + [ctypes.c_size_t, _vp, _vp,
                                                           ctypes.c_int, _vp]
            L.loglinear_decode_step.restype = ctypes.c_int
            L.loglinear_decode_step.argtypes = [_SP, ctypes.c_longlong] + [_vp] * 9
            L.loglinear_fwd_host_arena_bytes.restype = ctypes.c_size_t
            L.loglinear_fwd_host_arena_bytes.argtypes = [_SP]
            L.loglinear_fwd_host.restype = ctypes.c_int
            L.loglinear_fwd_host.argtypes = [_SP] + [_vp] * 7 + [ctypes.c_size_t, _vp]
            L.loglinear_check_status.restype = ctypes.c_int
            L.loglinear_check_status.argtypes = [_vp]
            L.loglinear_selftest_wait_timeout.restype = ctypes.c_int
            L.loglinear_selftest_wait_timeout.argtypes = [ctypes.c_longlong, _vp]
            L.loglinear_fwd_profiled.restype = ctypes.c_int
            L.loglinear_fwd_profiled.argtypes = ([_SP] + [_vp] * 7 + [ctypes.c_size_t, _vp, _vp,
                                                  ctypes.c_int, _vp, ctypes.POINTER(_vp),
                                                  ctypes.c_int])
            L.loglinear_fwd_kernel_names.restype = ctypes.c_char_p
            L.loglinear_fwd_kernel_names.argtypes = [_SP, ctypes.c_int]
            L.loglinear_fwd_static_workspace.restype = ctypes.c_int
            L.loglinear_fwd_static_workspace.argtypes = [_SP] + [_vp] * 8 + [ctypes.c_int, _vp]
            L.loglinear_launch_count.restype = ctypes.c_ulonglong
            L.loglinear_launch_count.argtypes = []
            L.loglinear_fwd_naive_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_fwd_naive_workspace_bytes.argtypes = [_SP]
            L.loglinear_fwd_naive.restype = ctypes.c_int
            L.loglinear_fwd_naive.argtypes = [_SP] + [_vp] * 7 + [ctypes.c_size_t, _vp]
            L.ssd_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.ssd_fwd_workspace_bytes.argtypes = [_SP]
            L.loglinear_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_bwd_workspace_bytes.argtypes = [_SP]
            L.loglinear_bwd.restype = ctypes.c_int
            L.loglinear_bwd.argtypes = [_SP] + [_vp] * 12 + [ctypes.c_size_t, _vp]
            L.loglinear_gdn_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_gdn_fwd_workspace_bytes.argtypes = [_SP]
            L.loglinear_gdn_fwd.restype = ctypes.c_int
            L.loglinear_gdn_fwd.argtypes = [_SP] + [_vp] * 8 + [ctypes.c_size_t, _vp]
            L.ssd_fwd.restype = ctypes.c_int
            L.ssd_fwd.argtypes = [_SP] + [_vp] * 6 + [ctypes.c_size_t, _vp]
            L.loglinear_fwd_continue_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_fwd_continue_workspace_bytes.argtypes = [_SP, ctypes.c_longlong]
            L.loglinear_fwd_continue.restype = ctypes.c_int
            L.loglinear_fwd_continue.argtypes = ([_SP, ctypes.c_longlong] + [_vp] * 7 + [ctypes.c_int] +
                                                 [_vp, _vp, ctypes.c_size_t, _vp, _vp, ctypes.c_int, _vp])
            L.loglinear_segment_total_workspace_bytes.restype = ctypes.c_size_t
            L.loglinear_segment_total_workspace_bytes.argtypes = [_SP]
            L.loglinear_segment_total.restype = ctypes.c_int
            L.loglinear_segment_total.argtypes = [_SP] + [_vp] * 4 + [ctypes.c_size_t, _vp, _vp, _vp]
            L.loglinear_prefix_states.restype = ctypes.c_int
            L.loglinear_prefix_states.argtypes = [_SP, ctypes.c_int] + [_vp] * 4 + [ctypes.c_int, _vp]
            _lib = L
    return _lib


def loglinear_status_string(status: int) -> str:
    return lib().loglinear_status_string(int(status)).decode()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return LL_BF16
    if dt == torch.float32:
        return LL_F32
    raise TypeError(f"unsupported dtype {dt}")


def make_shape(batch, T, heads, heads_per_group, d_k, d_v, chunk, levels, dtype) -> LLShape:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return LLShape(batch, T, heads, heads_per_group, d_k, d_v, chunk, levels, code)


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _ptr(x):
    return None if x is None else x.data_ptr()


def _check(status: int, where: str):
    if status != LL_OK:
        raise LogLinearError(status, where)


def _on_device(*tensors):
    """Context that makes the tensors' CUDA device current for the call.  The library
    works on the current device (its status word, its stream lookups, the static
    workspace) and the default stream is the current device's, so every tensor of a call
    must live on one device and that device must be current while the call enqueues."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors of a call must be on one CUDA device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if dev.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {dev}")
    return torch.cuda.device(dev)


def loglinear_fwd_workspace_bytes(shape: LLShape) -> int:
    return int(lib().loglinear_fwd_workspace_bytes(ctypes.byref(shape)))


def loglinear_fwd_path(shape: LLShape) -> int:
    return int(lib().loglinear_fwd_path(ctypes.byref(shape)))


def fwd_shape(q, v, lam, chunk) -> LLShape:
    B, T, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    return make_shape(B, T, H, H // G, dk, dv, chunk, lam.shape[3], q.dtype)


def loglinear_fwd(q, k, v, a, lam, chunk: int = 64, o=None, workspace=None, states_out=None,
                  state_logscale_out=None, state_levels: int = 0, stream=None):
    """o = log-linear Mamba-2 forward.  q, k: (B, T, G, d_k); v: (B, T, H, d_v);
    a: (B, T, H) fp32; lam: (B, T, H, L) fp32; all contiguous CUDA tensors."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    if workspace is None:
        nb = loglinear_fwd_workspace_bytes(shape)
        if nb == 0:
            raise LogLinearError(2, "loglinear_fwd_workspace_bytes")
        workspace = torch.empty(nb, dtype=torch.uint8, device=q.device)
    for x in (q, k, v, a, lam, o):
        if not x.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    with _on_device(q, k, v, a, lam, o, workspace, states_out, state_logscale_out):
        st = lib().loglinear_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(lam),
                                 _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(states_out), _ptr(state_logscale_out), int(state_levels),
                                 _stream_ptr(stream))
    _check(st, "loglinear_fwd")
    return o


def loglinear_fwd_profiled(q, k, v, a, lam, events, chunk: int = 64, o=None, workspace=None,
                           states_out=None, state_logscale_out=None, state_levels: int = 0,
                           stream=None):
    """loglinear_fwd that also records torch.cuda.Event objects around its kernels:
    events[0] before the first kernel, events[i + 1] after kernel i."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(loglinear_fwd_workspace_bytes(shape), dtype=torch.uint8,
                                device=q.device)
    arr = (_vp * len(events))(*[e.cuda_event for e in events])
    with _on_device(q, k, v, a, lam, o, workspace, states_out, state_logscale_out):
        st = lib().loglinear_fwd_profiled(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                          _ptr(lam), _ptr(o), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _ptr(states_out), _ptr(state_logscale_out),
                                          int(state_levels), _stream_ptr(stream), arr, len(events))
    _check(st, "loglinear_fwd_profiled")
    return o


STATIC_WORKSPACE_BYTES = 32 << 20


def loglinear_fwd_static_workspace(q, k, v, a, lam, chunk: int = 64, o=None, states_out=None,
                                   state_logscale_out=None, state_levels: int = 0, stream=None):
    """loglinear_fwd without a workspace argument, for callers that cannot allocate device
    memory: the library's own fixed 32 MiB device array is used instead (shapes needing
    more are rejected).  Only `o` is allocated here, and only when it is not given."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    with _on_device(q, k, v, a, lam, o, states_out, state_logscale_out):
        st = lib().loglinear_fwd_static_workspace(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                                  _ptr(a), _ptr(lam), _ptr(o), _ptr(states_out),
                                                  _ptr(state_logscale_out), int(state_levels),
                                                  _stream_ptr(stream))
    _check(st, "loglinear_fwd_static_workspace")
    return o


def loglinear_gdn_fwd(q, k, v, a, beta, lam, chunk: int = 64, o=None, workspace=None, stream=None):
    """Log-linear Gated DeltaNet forward: beta (B, T, H) fp32, the rest as loglinear_fwd."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    nb = int(lib().loglinear_gdn_fwd_workspace_bytes(ctypes.byref(shape)))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    with _on_device(q, k, v, a, beta, lam, o, workspace):
        st = lib().loglinear_gdn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta),
                                     _ptr(lam), _ptr(o), _ptr(workspace), workspace.numel(),
                                     _stream_ptr(stream))
    _check(st, "loglinear_gdn_fwd")
    return o


def loglinear_bwd(q, k, v, a, lam, dO, chunk: int = 64, workspace=None, stream=None):
    """Gradients of sum(dO * loglinear_fwd(q, k, v, a, lam)): returns dq, dk (B, T, G, d_k)
    and dv (B, T, H, d_v) in the input dtype, dlog_a (B, T, H; with respect to log a) and
    dlam (B, T, H, L) in fp32."""
    shape = fwd_shape(q, v, lam, chunk)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dloga, dlam = torch.empty_like(a), torch.empty_like(lam)
    nb = int(lib().loglinear_bwd_workspace_bytes(ctypes.byref(shape)))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    with _on_device(q, k, v, a, lam, dO, dq, dk, dv, dloga, dlam, workspace):
        st = lib().loglinear_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(lam),
                                 _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dloga), _ptr(dlam),
                                 _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(st, "loglinear_bwd")
    return dq, dk, dv, dloga, dlam


def loglinear_fwd_naive(q, k, v, a, lam, chunk: int = 64, o=None, workspace=None, stream=None):
    """Comparator: the same output as loglinear_fwd, one output pass per level (no level
    fusion).  Tensor-core shape only."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    nb = int(lib().loglinear_fwd_naive_workspace_bytes(ctypes.byref(shape)))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    with _on_device(q, k, v, a, lam, o, workspace):
        st = lib().loglinear_fwd_naive(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                       _ptr(lam), _ptr(o), _ptr(workspace), workspace.numel(),
                                       _stream_ptr(stream))
    _check(st, "loglinear_fwd_naive")
    return o


def ssd_fwd(q, k, v, a, chunk: int = 64, o=None, workspace=None, stream=None):
    """Comparator: the lambda-constant special case (Mamba-2 SSD) with a sequential state
    pass over tiles.  Tensor-core shape only."""
    B, T, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    shape = make_shape(B, T, H, H // G, dk, dv, chunk, max(1, (T - 1).bit_length() + 1), q.dtype)
    if o is None:
        o = torch.empty_like(v)
    nb = int(lib().ssd_fwd_workspace_bytes(ctypes.byref(shape)))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    with _on_device(q, k, v, a, o, workspace):
        st = lib().ssd_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o),
                           _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(st, "ssd_fwd")
    return o


def loglinear_fwd_continue(q, k, v, a, lam, T0: int, prefix_states=None, prefix_logscale=None,
                           chunk: int = 64, o=None, workspace=None, states_out=None,
                           state_logscale_out=None, state_levels: int = 0, stream=None):
    """Forward over the positions T0 .. T0+T-1 (the segment's tensors, laid out as for
    loglinear_fwd, lambda with absolute levels) from the bucket memories at T0:
    prefix_states (B, H, Lp, d_k, d_v) fp32 and prefix_logscale (B, H, Lp) fp32.  T0 must
    be a multiple of the smallest power of two >= T.  states_out (may be prefix_states)
    receives the memories at T0 + T."""
    shape = fwd_shape(q, v, lam, chunk)
    if o is None:
        o = torch.empty_like(v)
    nb = int(lib().loglinear_fwd_continue_workspace_bytes(ctypes.byref(shape), int(T0)))
    if nb == 0:
        raise LogLinearError(2, "loglinear_fwd_continue_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nb, dtype=torch.uint8, device=q.device)
    Lp = 0 if prefix_states is None else prefix_states.shape[2]
    with _on_device(q, k, v, a, lam, o, workspace, prefix_states, prefix_logscale, states_out,
                    state_logscale_out):
        st = lib().loglinear_fwd_continue(ctypes.byref(shape), int(T0), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                          _ptr(lam), _ptr(prefix_states), _ptr(prefix_logscale), int(Lp),
                                          _ptr(o), _ptr(workspace), workspace.numel(), _ptr(states_out),
                                          _ptr(state_logscale_out), int(state_levels), _stream_ptr(stream))
    _check(st, "loglinear_fwd_continue")
    return o


def loglinear_segment_total(k, v, a, chunk: int = 64, workspace=None, stream=None):
    """The memory of the whole segment held by k, v, a ((B, T, G, d_k), (B, T, H, d_v),
    (B, T, H)): returns total_state (B, H, d_k, d_v) fp32 and total_logdecay (B, H) fp32."""
    B, T, G, dk = k.shape
    H, dv = v.shape[2], v.shape[3]
    shape = make_shape(B, T, H, H // G, dk, dv, chunk, max(1, (T - 1).bit_length() + 1), k.dtype)
    nb = int(lib().loglinear_segment_total_workspace_bytes(ctypes.byref(shape)))
    if nb == 0:
        raise LogLinearError(2, "loglinear_segment_total_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nb, dtype=torch.uint8, device=k.device)
    total = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    logdecay = torch.empty((B, H), dtype=torch.float32, device=k.device)
    with _on_device(k, v, a, workspace, total, logdecay):
        st = lib().loglinear_segment_total(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(a), _ptr(workspace),
                                           workspace.numel(), _ptr(total), _ptr(logdecay), _stream_ptr(stream))
    _check(st, "loglinear_segment_total")
    return total, logdecay


def loglinear_prefix_states(seg_states, seg_logdecay, seg_len: int, state_levels: int, states_out=None,
                            state_logscale_out=None, stream=None):
    """Bucket memories at T0 = n * seg_len from the memories of the n segments before it:
    seg_states (n, B, H, d_k, d_v) and seg_logdecay (n, B, H), fp32.  Returns states
    (B, H, state_levels, d_k, d_v) and log-scales (B, H, state_levels); only the levels
    live at T0 are written (zero log-scales there)."""
    n, B, H, dk, dv = seg_states.shape
    dev = seg_states.device
    if states_out is None:
        states_out = torch.zeros((B, H, state_levels, dk, dv), dtype=torch.float32, device=dev)
    if state_logscale_out is None:
        state_logscale_out = torch.zeros((B, H, state_levels), dtype=torch.float32, device=dev)
    shape = make_shape(B, seg_len, H, 1, dk, dv, 16, 1, LL_F32)
    with _on_device(seg_states, seg_logdecay, states_out, state_logscale_out):
        st = lib().loglinear_prefix_states(ctypes.byref(shape), int(n), _ptr(seg_states), _ptr(seg_logdecay),
                                           _ptr(states_out), _ptr(state_logscale_out), int(state_levels),
                                           _stream_ptr(stream))
    _check(st, "loglinear_prefix_states")
    return states_out, state_logscale_out


def loglinear_fwd_kernel_names(shape: LLShape, with_export: bool = False):
    raw = lib().loglinear_fwd_kernel_names(ctypes.byref(shape), int(bool(with_export))).decode()
    return [n for n in raw.split(",") if n]


def loglinear_launch_count() -> int:
    return int(lib().loglinear_launch_count())


def loglinear_decode_step(pos: int, q_t, k_t, v_t, a_t, lam_t, states, state_logscale, o_t=None,
                          stream=None):
    """One decode step at position pos.  q_t, k_t: (B, G, d_k); v_t: (B, H, d_v);
    a_t: (B, H); lam_t: (B, H, L); states: (B, H, L, d_k, d_v) fp32 and
    state_logscale: (B, H, L) fp32, both updated in place."""
    B, G, dk = q_t.shape
    H, dv = v_t.shape[1], v_t.shape[2]
    L = states.shape[2]
    shape = make_shape(B, 1, H, H // G, dk, dv, 16, L, q_t.dtype)
    if o_t is None:
        o_t = torch.empty_like(v_t)
    with _on_device(q_t, k_t, v_t, a_t, lam_t, o_t, states, state_logscale):
        st = lib().loglinear_decode_step(ctypes.byref(shape), int(pos), _ptr(q_t), _ptr(k_t),
                                         _ptr(v_t), _ptr(a_t), _ptr(lam_t), _ptr(o_t), _ptr(states),
                                         _ptr(state_logscale), _stream_ptr(stream))
    _check(st, "loglinear_decode_step")
    return o_t


def loglinear_fwd_host_arena_bytes(shape: LLShape) -> int:
    return int(lib().loglinear_fwd_host_arena_bytes(ctypes.byref(shape)))


def loglinear_fwd_host(q, k, v, a, lam, o, arena, chunk: int = 64, stream=None):
    """End-to-end forward from host tensors (pinned for async copies) into host o,
    using the device buffer `arena`; enqueued on `stream`, the caller synchronises."""
    shape = fwd_shape(q, v, lam, chunk)
    with _on_device(arena):
        st = lib().loglinear_fwd_host(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                      _ptr(lam), _ptr(o), _ptr(arena),
                                      arena.numel() * arena.element_size(), _stream_ptr(stream))
    _check(st, "loglinear_fwd_host")
    return o


def loglinear_check_status(stream=None) -> int:
    return int(lib().loglinear_check_status(_stream_ptr(stream)))


def loglinear_selftest_wait_timeout(spins: int, stream=None) -> None:
    _check(lib().loglinear_selftest_wait_timeout(int(spins), _stream_ptr(stream)),
           "loglinear_selftest_wait_timeout")
