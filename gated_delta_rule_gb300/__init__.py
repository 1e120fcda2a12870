"""Python binding of libkda, the GB300 KDA core (C ABI in include/kda.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libkda.so``.  PyTorch supplies device memory and streams.  There is
no fallback: if the library is missing, importing the binding's entry points
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB, build, up_to_date  # noqa: F401

__all__ = ["kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_fused_recurrent_fwd", "kda_recurrent_step",
           "kda_recurrent_multi_step", "kda_chunk_fwd_gated", "kda_chunk_fwd_checkpointed",
           "kda_decode_step_fused", "kda_backward", "kda_chunk_bwd",
           "kda_get_device_error", "kda_set_launch_events", "kda_last_launch_count",
           "kda_test_stall_next_prefill", "KdaError",
           "load_library", "build", "STATUS"]

STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
          4: "KDA_ERR_DEVICE", 5: "KDA_ERR_TIMEOUT", 6: "KDA_ERR_DOMAIN"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.int32: 2}

EXPORTED = ["kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_fused_recurrent_fwd", "kda_recurrent_step",
            "kda_recurrent_multi_step", "kda_chunk_fwd_gated", "kda_chunk_fwd_checkpointed",
            "kda_decode_step_fused", "kda_backward", "kda_chunk_bwd",
            "kda_get_device_error", "kda_status_string", "kda_last_error_message",
            "kda_set_launch_events", "kda_last_launch_count", "kda_test_stall_next_prefill"]


class KdaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


_lib = None
_P = ctypes.POINTER(KdaTensor)


def load_library(path: str | None = None):
    """Load libkda.so (built in-tree by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise ImportError(f"libkda.so not built ({path}); run gated_delta_rule_gb300.build()")
    lib = ctypes.CDLL(path)
    fwd = [_P] * 6 + [ctypes.c_float, _P, _P, _P, ctypes.c_void_p]
    for name in ("kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_fused_recurrent_fwd"):
        f = getattr(lib, name)
        f.restype, f.argtypes = ctypes.c_int, fwd
    lib.kda_recurrent_step.restype = ctypes.c_int
    lib.kda_recurrent_step.argtypes = [_P] * 6 + [ctypes.c_float, _P, ctypes.c_void_p]
    lib.kda_backward.restype = ctypes.c_int
    lib.kda_backward.argtypes = [_P] * 6 + [ctypes.c_float] + [_P] * 9 + [ctypes.c_void_p]
    lib.kda_chunk_bwd.restype = ctypes.c_int
    lib.kda_chunk_bwd.argtypes = [_P] * 6 + [ctypes.c_float] + [_P] * 9 + [ctypes.c_void_p]
    lib.kda_decode_step_fused.restype = ctypes.c_int
    lib.kda_decode_step_fused.argtypes = [_P] * 14 + [ctypes.c_float, ctypes.c_float, _P, ctypes.c_void_p]
    lib.kda_chunk_fwd_checkpointed.restype = ctypes.c_int
    lib.kda_chunk_fwd_checkpointed.argtypes = [_P] * 6 + [ctypes.c_float, _P, ctypes.c_int64, _P, _P, _P,
                                                   ctypes.c_void_p]
    lib.kda_chunk_fwd_gated.restype = ctypes.c_int
    lib.kda_chunk_fwd_gated.argtypes = [_P] * 7 + [ctypes.c_float, _P, _P, _P, ctypes.c_void_p]
    lib.kda_recurrent_multi_step.restype = ctypes.c_int
    lib.kda_recurrent_multi_step.argtypes = [_P] * 6 + [ctypes.c_float, _P, _P, ctypes.c_void_p]
    lib.kda_get_device_error.restype = ctypes.c_int
    lib.kda_get_device_error.argtypes = [ctypes.c_void_p]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_last_error_message.restype = ctypes.c_char_p
    lib.kda_last_error_message.argtypes = []
    lib.kda_set_launch_events.restype = ctypes.c_int
    lib.kda_set_launch_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    lib.kda_last_launch_count.restype = ctypes.c_int
    lib.kda_last_launch_count.argtypes = []
    lib.kda_test_stall_next_prefill.restype = ctypes.c_int
    lib.kda_test_stall_next_prefill.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def desc(t: torch.Tensor | None):
    """kda_tensor descriptor of a torch tensor (no copy); None stays NULL."""
    if t is None:
        return None
    if t.dim() > 4:
        raise ValueError("at most 4 dimensions")
    d = KdaTensor()
    d.data = t.data_ptr() if t.numel() else None
    d.dtype = DTYPES.get(t.dtype, -1)
    d.ndim = t.dim()
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = s
        d.stride[i] = st
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _check(lib, status: int):
    if status != 0:
        raise KdaError(status, lib.kda_last_error_message().decode())


def kda_chunk_fwd(q, k, v, g, beta, initial_state=None, scale=None, cu_seqlens=None, out=None,
                  final_state=None, output_final_state=True, stream=None, _entry="kda_chunk_fwd"):
    """Chunked KDA prefill.  Shapes as in include/kda.h; returns (out, final_state)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.shape[0] - 1
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    ds = [desc(x) for x in (q, k, v, g, beta, initial_state, cu_seqlens, out, final_state)]
    st = getattr(lib, _entry)(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), _ref(ds[4]),
                              _ref(ds[5]), float(scale), _ref(ds[6]), _ref(ds[7]), _ref(ds[8]),
                              _stream(stream))
    _check(lib, st)
    return out, final_state


def kda_chunk_fwd_gated(q, k, v, gate, gate_scale, beta, initial_state=None, scale=None,
                        cu_seqlens=None, out=None, final_state=None, output_final_state=True,
                        stream=None):
    """Chunked prefill with the log-decay formed in the kernel: g = -5 sigmoid(A_h z),
    ``gate`` = z [B, T, H, dk] in q's dtype, ``gate_scale`` = A [H] fp32 (device).
    Returns (out, final_state)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.shape[0] - 1
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    ds = [desc(x) for x in (q, k, v, gate, gate_scale, beta, initial_state, cu_seqlens, out, final_state)]
    st = lib.kda_chunk_fwd_gated(*[_ref(x) for x in ds[:7]], float(scale), _ref(ds[7]), _ref(ds[8]),
                                 _ref(ds[9]), _stream(stream))
    _check(lib, st)
    return out, final_state


def kda_chunk_fwd_checkpointed(q, k, v, g, beta, initial_state=None, scale=None, cu_seqlens=None,
                               checkpoint_tokens=512, checkpoints=None, num_checkpoints=None, out=None,
                               final_state=None, output_final_state=True, stream=None):
    """kda_chunk_fwd plus the state after every ``checkpoint_tokens`` tokens of each
    sequence.  ``checkpoints`` [N * C, H, dk, dv] fp32 (allocated with C =
    ``num_checkpoints``, default T // checkpoint_tokens, when None); row n * C + j
    is checkpoint j of sequence n.  Returns (out, final_state, checkpoints)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.shape[0] - 1
    if scale is None:
        scale = dk ** -0.5
    if checkpoints is None:
        C = T // checkpoint_tokens if num_checkpoints is None else int(num_checkpoints)
        checkpoints = torch.zeros((N * C, H, dk, dv), dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    ds = [desc(x) for x in (q, k, v, g, beta, initial_state, cu_seqlens, checkpoints, out, final_state)]
    st = lib.kda_chunk_fwd_checkpointed(*[_ref(x) for x in ds[:6]], float(scale), _ref(ds[6]),
                                        int(checkpoint_tokens), _ref(ds[7]), _ref(ds[8]), _ref(ds[9]),
                                        _stream(stream))
    _check(lib, st)
    return out, final_state, checkpoints


def kda_fused_recurrent_fwd(*args, **kw):
    """Token-by-token KDA prefill with on-chip fp32 state; same contract as kda_chunk_fwd."""
    kw["_entry"] = "kda_fused_recurrent_fwd"
    return kda_chunk_fwd(*args, **kw)


def kda_chunk_fwd_noalloc(*args, **kw):
    """kda_chunk_fwd without any device allocation inside the library call: the
    chunk records live in the library's fixed 64 MiB device workspace (see
    include/kda.h).  Outputs not passed in are still allocated here, by torch,
    before the call; pass ``out`` and ``final_state`` to avoid that too."""
    kw["_entry"] = "kda_chunk_fwd_noalloc"
    return kda_chunk_fwd(*args, **kw)


def kda_recurrent_step(state, q, k, v, g, beta, scale=None, out=None, stream=None):
    """One decode step per (request, head); updates ``state`` in place, returns out."""
    lib = load_library()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    ds = [desc(x) for x in (state, q, k, v, g, beta, out)]
    st = lib.kda_recurrent_step(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), _ref(ds[4]),
                                _ref(ds[5]), float(scale), _ref(ds[6]), _stream(stream))
    _check(lib, st)
    return out


def kda_recurrent_multi_step(state, q, k, v, g, beta, scale=None, num_accepted=None, out=None,
                             stream=None):
    """n decode tokens per request: q, k, g [N, n, H, d_k], v [N, n, H, d_v], beta
    [N, n, H].  Keeps the state after the first ``num_accepted[i]`` tokens (int32
    [N] on the device; None = all n), written once in place.  With ``q=None`` no
    outputs are made (a commit); otherwise returns out [N, n, H, d_v]."""
    lib = load_library()
    N, n, H, dk = k.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    if q is not None and out is None:
        out = torch.empty((N, n, H, dv), dtype=k.dtype, device=k.device)
    if q is None:
        out = None
    ds = [desc(x) for x in (state, q, k, v, g, beta, num_accepted, out)]
    st = lib.kda_recurrent_multi_step(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), _ref(ds[4]),
                                      _ref(ds[5]), float(scale), _ref(ds[6]), _ref(ds[7]), _stream(stream))
    _check(lib, st)
    return out


def kda_decode_step_fused(state, conv_q, conv_k, conv_v, q, k, v, w_q, w_k, w_v, g, beta, out_gate,
                          norm_weight=None, scale=None, eps=1e-6, out=None, stream=None):
    """Decode step with the layer's front end (short convolutions over the caches,
    SiLU, L2 norm of q and k) and back end (RMSNorm, sigmoid output gate).  The
    state and the three conv caches are updated in place; returns out [N, H, dv]."""
    lib = load_library()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    ds = [desc(x) for x in (state, conv_q, conv_k, conv_v, q, k, v, w_q, w_k, w_v, g, beta, out_gate,
                            norm_weight, out)]
    st = lib.kda_decode_step_fused(*[_ref(x) for x in ds[:14]], float(scale), float(eps), _ref(ds[14]),
                                   _stream(stream))
    _check(lib, st)
    return out


def _backward(entry, q, k, v, g, beta, initial_state, scale, d_out, d_final_state, cu_seqlens,
              need_initial_state_grad, stream):
    lib = load_library()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.shape[0] - 1
    if scale is None:
        scale = dk ** -0.5
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
               dv=torch.empty((B, T, H, dv), **f32), dg=torch.empty((B, T, H, dk), **f32),
               dbeta=torch.empty((B, T, H), **f32),
               d_initial_state=torch.empty((N, H, dk, dv), **f32) if need_initial_state_grad else None)
    ds = [desc(x) for x in (q, k, v, g, beta, initial_state)]
    dr = [desc(x) for x in (cu_seqlens, d_out, d_final_state, out["dq"], out["dk"], out["dv"], out["dg"],
                            out["dbeta"], out["d_initial_state"])]
    st = getattr(lib, entry)(*[_ref(x) for x in ds], float(scale), *[_ref(x) for x in dr], _stream(stream))
    _check(lib, st)
    return out


def kda_backward(q, k, v, g, beta, initial_state, scale, d_out, d_final_state=None, cu_seqlens=None,
                 need_initial_state_grad=True, stream=None):
    """Gradients of the KDA core (kda_chunk_fwd's forward) given d_out [B, T, H, dv]
    and d_final_state [N, H, dk, dv] (or None), by the token loop.  Returns a dict of
    fp32 tensors dq, dk, dv, dg, dbeta and d_initial_state (None unless requested)."""
    return _backward("kda_backward", q, k, v, g, beta, initial_state, scale, d_out, d_final_state, cu_seqlens,
                     need_initial_state_grad, stream)


def kda_chunk_bwd(q, k, v, g, beta, initial_state, scale, d_out, d_final_state=None, cu_seqlens=None,
                  need_initial_state_grad=True, stream=None):
    """The gradients of kda_backward by the chunked form (g in [-5, 0]); same
    arguments and result."""
    return _backward("kda_chunk_bwd", q, k, v, g, beta, initial_state, scale, d_out, d_final_state, cu_seqlens,
                     need_initial_state_grad, stream)


def kda_get_device_error(stream=None) -> int:
    """Synchronise ``stream`` and raise KdaError if the device recorded an error."""
    lib = load_library()
    _check(lib, lib.kda_get_device_error(_stream(stream)))
    return 0


_armed = None  # keeps the handle array alive until the armed call has returned


def kda_set_launch_events(events) -> None:
    """Arm this thread's next compute call to record ``events[0]`` before its first
    kernel and ``events[i]`` after its i-th (``torch.cuda.Event(enable_timing=True)``
    objects that have been recorded once, so that their CUDA handles exist).  An
    empty list or None disarms."""
    global _armed
    lib = load_library()
    events = list(events or [])
    handles = [e.cuda_event for e in events]
    if any(h == 0 for h in handles):
        raise ValueError("record each event once before arming it (its handle is created lazily)")
    _armed = (ctypes.c_void_p * max(1, len(handles)))(*handles)
    _check(lib, lib.kda_set_launch_events(_armed if handles else None, len(handles)))


def kda_last_launch_count() -> int:
    """Kernels enqueued by this thread's last compute call."""
    return load_library().kda_last_launch_count()


def kda_test_stall_next_prefill(on: bool = True) -> None:
    """Testing hook: this thread's next prefill call runs its serial kernel with the
    chunk-record copies suppressed and short bounded waits, so the waits give up and
    kda_get_device_error reports KDA_ERR_TIMEOUT (see include/kda.h)."""
    _check(load_library(), load_library().kda_test_stall_next_prefill(1 if on else 0))
