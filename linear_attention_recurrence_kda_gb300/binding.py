"""ctypes binding of libkda.so (the C ABI in include/kda.h), with the same entry-point names.

Argument marshalling only: tensors are checked for device/dtype/shape/contiguity, their data
pointers and the current CUDA stream are passed to the C ABI, and any non-OK status raises
``KdaError``.  Every step of the computation runs in the library's CUDA kernels; there is no
fallback path, and loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4
KDA_ERR_WORKSPACE = 5
KDA_ERR_DEVICE_CHECK = 6

KDA_F32 = 0
KDA_BF16 = 1

G_MIN = -5.0

# Every symbol include/kda.h declares.
EXPORTS = ("kda_forward_workspace_bytes", "kda_forward", "kda_decode_step", "kda_workspace_status",
           "kda_status_string", "kda_profile_enable", "kda_profile_read", "kda_abi_version",
           "kda_forward_static_scratch", "kda_forward_plan", "kda_decode_replay", "kda_prologue",
           "kda_epilogue", "kda_static_scratch_status", "kda_backward_workspace_bytes", "kda_backward",
           "kda_forward_summary_workspace_bytes", "kda_forward_summary", "kda_state_scan")

# Size of the library's own scratch array used by kda_forward_static_scratch.
KDA_STATIC_SCRATCH_BYTES = 8 << 20


class KdaPlan(ctypes.Structure):
    """Mirror of kda_plan_t."""
    _fields_ = [("split", ctypes.c_int32), ("seg_chunks", ctypes.c_int32), ("num_segments", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class KdaProblem(ctypes.Structure):
    """Mirror of kda_problem_t."""
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64), ("max_seqlen", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("io_dtype", ctypes.c_int), ("g_min", ctypes.c_float)]


class KdaKernelTime(ctypes.Structure):
    """Mirror of kda_kernel_time_t."""
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def lib():
    """The loaded libkda.so with argument types declared (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libkda.so is not built ({LIB_PATH} missing); run "
                                   "`python -m linear_attention_recurrence_kda_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER(KdaProblem)
            L.kda_forward_workspace_bytes.restype = ctypes.c_size_t
            L.kda_forward_workspace_bytes.argtypes = [P]
            L.kda_forward.restype = ctypes.c_int
            L.kda_forward.argtypes = [_vp] * 10 + [P, _vp, ctypes.c_size_t, _vp]
            L.kda_decode_step.restype = ctypes.c_int
            L.kda_decode_step.argtypes = [_vp] * 8 + [P, _vp]
            L.kda_decode_replay.restype = ctypes.c_int
            L.kda_decode_replay.argtypes = [_vp] * 10 + [P, _vp]
            L.kda_prologue.restype = ctypes.c_int
            L.kda_prologue.argtypes = [_vp] * 6 + [ctypes.c_int32] + [_vp] * 4 + [P, _vp]
            L.kda_epilogue.restype = ctypes.c_int
            L.kda_epilogue.argtypes = [_vp, _vp, _vp, ctypes.c_float, _vp, P, _vp]
            L.kda_workspace_status.restype = ctypes.c_int
            L.kda_workspace_status.argtypes = [_vp, ctypes.c_size_t, _vp]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_profile_enable.restype = ctypes.c_int
            L.kda_profile_enable.argtypes = [ctypes.c_int]
            L.kda_profile_read.restype = ctypes.c_int32
            L.kda_profile_read.argtypes = [ctypes.POINTER(KdaKernelTime), ctypes.c_int32]
            L.kda_forward_static_scratch.restype = ctypes.c_int
            L.kda_forward_static_scratch.argtypes = [_vp] * 10 + [P, _vp]
            L.kda_backward_workspace_bytes.restype = ctypes.c_size_t
            L.kda_backward_workspace_bytes.argtypes = [P]
            L.kda_backward.restype = ctypes.c_int
            L.kda_backward.argtypes = [_vp] * 17 + [P, _vp, ctypes.c_size_t, _vp]
            L.kda_forward_summary_workspace_bytes.restype = ctypes.c_size_t
            L.kda_forward_summary_workspace_bytes.argtypes = [P]
            L.kda_forward_summary.restype = ctypes.c_int
            L.kda_forward_summary.argtypes = [_vp] * 9 + [P, _vp, ctypes.c_size_t, _vp]
            L.kda_state_scan.restype = ctypes.c_int
            L.kda_state_scan.argtypes = [_vp, _vp, _vp, ctypes.c_int32, _vp, P, _vp]
            L.kda_static_scratch_status.restype = ctypes.c_int
            L.kda_static_scratch_status.argtypes = [_vp]
            L.kda_forward_plan.restype = ctypes.c_int
            L.kda_forward_plan.argtypes = [P, ctypes.c_size_t, ctypes.POINTER(KdaPlan)]
            L.kda_abi_version.restype = ctypes.c_uint32
            L.kda_abi_version.argtypes = []
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def make_problem(num_seqs: int, total_tokens: int, max_seqlen: int, num_heads: int, d_k: int, d_v: int,
                 io_dtype, g_min: float = G_MIN) -> KdaProblem:
    dt = io_dtype
    if isinstance(dt, torch.dtype):
        dt = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}[dt]
    return KdaProblem(int(num_seqs), int(total_tokens), int(max_seqlen), int(num_heads), int(d_k), int(d_v),
                      int(dt), float(g_min))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kda_forward_workspace_bytes(problem: KdaProblem) -> int:
    return int(lib().kda_forward_workspace_bytes(ctypes.byref(problem)))


def kda_forward_plan(problem: KdaProblem, workspace_bytes: Optional[int] = None) -> dict:
    """The plan kda_forward picks for ``problem`` with ``workspace_bytes`` (None: the fastest)."""
    plan = KdaPlan()
    wb = ctypes.c_size_t(-1).value if workspace_bytes is None else int(workspace_bytes)
    st = lib().kda_forward_plan(ctypes.byref(problem), wb, ctypes.byref(plan))
    if st != KDA_OK:
        raise KdaError(st, "kda_forward_plan")
    return {"split": bool(plan.split), "seg_chunks": int(plan.seg_chunks), "num_segments": int(plan.num_segments)}


def kda_forward(q, k, v, z, A, beta, initial_state=None, cu_seqlens=None, out=None, final_state=None,
                max_seqlen: Optional[int] = None, workspace=None, g_min: float = G_MIN, stream=None,
                want_final: bool = True):
    """Chunkwise KDA prefill (see include/kda.h).  Shapes: q, k, z [T, H, d_k]; v [T, H, d_v];
    A [H] fp32; beta [T, H] fp32; initial_state [N, H, d_k, d_v] fp32 or None; cu_seqlens [N+1]
    int32 on the device or None (one sequence, or N = initial_state.shape[0] equal lengths).

    ``max_seqlen`` must bound every sequence length when cu_seqlens is given (it is only used for
    grid sizing; pass it to avoid a device->host read of cu_seqlens).  Returns (out, final_state).
    """
    T, H, dk = k.shape
    dv = v.shape[2]
    dev = k.device
    dt = k.dtype
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    else:
        N = initial_state.shape[0] if initial_state is not None else 1
        max_seqlen = T // N
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("z", z, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=dt, device=dev)
    _need(out, "out", dt, (T, H, dv), dev)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, dk, dv), dev)
    prob = make_problem(N, T, max_seqlen, H, dk, dv, dt, g_min)
    wsb = kda_forward_workspace_bytes(prob)
    if wsb == 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_forward_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = lib().kda_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(initial_state),
                           _ptr(cu_seqlens), _ptr(out), _ptr(final_state), ctypes.byref(prob), _ptr(workspace),
                           ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_forward")
    return out, final_state


def kda_forward_static_scratch(q, k, v, z, A, beta, initial_state=None, cu_seqlens=None, out=None,
                               final_state=None, max_seqlen: Optional[int] = None, g_min: float = G_MIN,
                               stream=None, want_final: bool = True):
    """kda_forward without a workspace argument, for callers that cannot allocate device scratch
    (see include/kda.h): the library's own fixed-size device array is used instead.  Arguments and
    results as in :func:`kda_forward`; problems needing more than KDA_STATIC_SCRATCH_BYTES of
    scratch raise KdaError(KDA_ERR_WORKSPACE).  Calls that overlap on the GPU race on the array."""
    T, H, dk = k.shape
    dv = v.shape[2]
    dev = k.device
    dt = k.dtype
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    else:
        N = initial_state.shape[0] if initial_state is not None else 1
        max_seqlen = T // N
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("z", z, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=dt, device=dev)
    _need(out, "out", dt, (T, H, dv), dev)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, dk, dv), dev)
    prob = make_problem(N, T, max_seqlen, H, dk, dv, dt, g_min)
    st = lib().kda_forward_static_scratch(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta),
                                          _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                          ctypes.byref(prob), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_forward_static_scratch")
    return out, final_state


def kda_backward_workspace_bytes(problem: KdaProblem) -> int:
    return int(lib().kda_backward_workspace_bytes(ctypes.byref(problem)))


def kda_backward(q, k, v, z, A, beta, d_out, d_final_state=None, initial_state=None, cu_seqlens=None,
                 max_seqlen: Optional[int] = None, want_d_initial: bool = True, workspace=None,
                 g_min: float = G_MIN, stream=None):
    """Gradients of kda_forward (see include/kda.h): for L = <d_out, out> + <d_final_state,
    final_state>, returns (dq, dk, dv, dz, dA, dbeta, d_initial_state or None).  Shapes and dtypes
    as for :func:`kda_forward`; d_out [T, H, d_v] in the io dtype, d_final_state [N, H, d_k, d_v]
    fp32 or None (zero)."""
    T, H, dk = k.shape
    dv = v.shape[2]
    dev = k.device
    dt = k.dtype
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    else:
        N = (initial_state.shape[0] if initial_state is not None else
             d_final_state.shape[0] if d_final_state is not None else 1)
        max_seqlen = T // N
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("z", z, (T, H, dk)), ("v", v, (T, H, dv)),
                         ("d_out", d_out, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _need(t, name, torch.float32, (N, H, dk, dv), dev)
    dq, dk_, dz = (torch.empty((T, H, dk), dtype=dt, device=dev) for _ in range(3))
    dv_ = torch.empty((T, H, dv), dtype=dt, device=dev)
    dA = torch.empty((H,), dtype=torch.float32, device=dev)
    dbeta = torch.empty((T, H), dtype=torch.float32, device=dev)
    dS0 = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev) if want_d_initial else None
    prob = make_problem(N, T, max_seqlen, H, dk, dv, dt, g_min)
    wsb = kda_backward_workspace_bytes(prob)
    if wsb == 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_backward_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = lib().kda_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(initial_state),
                            _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk_), _ptr(dv_),
                            _ptr(dz), _ptr(dA), _ptr(dbeta), _ptr(dS0), ctypes.byref(prob), _ptr(workspace),
                            ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_backward")
    return dq, dk_, dv_, dz, dA, dbeta, dS0


def kda_forward_summary(q, k, v, z, A, beta, cu_seqlens=None, num_seqs: int = 1, max_seqlen: Optional[int] = None,
                        workspace=None, g_min: float = G_MIN, stream=None):
    """The affine summary (M, S~) of every sequence's token range (see include/kda.h): M
    [N, H, d_k, d_k] and S~ [N, H, d_k, d_v] fp32, with S_end = M S_in + S~.  Inputs as for
    :func:`kda_forward` (cu_seqlens, or ``num_seqs`` equal lengths)."""
    T, H, dk = k.shape
    dv = v.shape[2]
    dev = k.device
    dt = k.dtype
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
        if max_seqlen is None:
            max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    else:
        N = int(num_seqs)
        max_seqlen = T // N
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("z", z, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    M = torch.empty((N, H, dk, dk), dtype=torch.float32, device=dev)
    St = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    prob = make_problem(N, T, max_seqlen, H, dk, dv, dt, g_min)
    if workspace is None:
        wsb = int(lib().kda_forward_summary_workspace_bytes(ctypes.byref(prob)))
        if wsb == 0:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_forward_summary_workspace_bytes")
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = lib().kda_forward_summary(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(cu_seqlens), _ptr(M),
                                   _ptr(St), ctypes.byref(prob), _ptr(workspace),
                                   ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_forward_summary")
    return M, St


def kda_state_scan(transition, state_from_zero, initial_state=None, count: Optional[int] = None, state_out=None,
                   stream=None):
    """Apply S <- M_i S + S~_i for i < count (default: all) to ``initial_state`` (None: zeros).
    transition [R, N, H, d_k, d_k], state_from_zero [R, N, H, d_k, d_v] fp32 on one device."""
    R, N, H, dk, dv = state_from_zero.shape
    dev = state_from_zero.device
    count = R if count is None else int(count)
    if not 0 <= count <= R:
        raise ValueError("count out of range")
    _need(transition, "transition", torch.float32, (R, N, H, dk, dk), dev)
    _need(state_from_zero, "state_from_zero", torch.float32, (R, N, H, dk, dv), dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, dk, dv), dev)
    if state_out is None:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _need(state_out, "state_out", torch.float32, (N, H, dk, dv), dev)
    prob = make_problem(N, N, 1, H, dk, dv, torch.float32)
    st = lib().kda_state_scan(_ptr(transition), _ptr(state_from_zero), _ptr(initial_state), ctypes.c_int32(count),
                              _ptr(state_out), ctypes.byref(prob), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_state_scan")
    return state_out


def kda_decode_step(q, k, v, z, A, beta, state, out=None, g_min: float = G_MIN, stream=None):
    """One decode token per sequence: q, k, z [N, H, d_k]; v [N, H, d_v]; beta [N, H] fp32;
    state [N, H, d_k, d_v] fp32 (updated in place).  Returns out [N, H, d_v]."""
    N, H, dk = k.shape
    dv = v.shape[2]
    dev = k.device
    dt = k.dtype
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("z", z, (N, H, dk)), ("v", v, (N, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (N, H), dev)
    _need(state, "state", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=dt, device=dev)
    _need(out, "out", dt, (N, H, dv), dev)
    prob = make_problem(N, N, 1, H, dk, dv, dt, g_min)
    st = lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(state), _ptr(out),
                               ctypes.byref(prob), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step")
    return out


def kda_decode_replay(q, k, v, z, A, beta, state_in, accepted=None, state_out=None, out=None,
                      want_out: bool = True, want_state: bool = True, g_min: float = G_MIN, stream=None):
    """A window of L drafted tokens per sequence from the snapshot ``state_in`` (speculative-decode
    state replay; see include/kda.h): q, k, z [N*L, H, d_k] with token t of sequence n at row
    n*L + t; v [N*L, H, d_v]; beta [N*L, H] fp32; state_in [N, H, d_k, d_v] fp32; accepted [N]
    int32 or None (all L).  ``out`` receives o_t of every window token (allocated when
    ``want_out`` and not given); ``state_out`` the state after each accepted prefix (allocated when
    ``want_state`` and not given; pass ``state_in`` to advance the snapshot in place).
    Returns (out or None, state_out or None)."""
    N, H, dk, dv = state_in.shape
    T = k.shape[0]
    dev = k.device
    dt = k.dtype
    if N < 1 or T < N or T % N:
        raise ValueError("the token count must be a positive multiple of the number of sequences")
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("z", z, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(beta, "beta", torch.float32, (T, H), dev)
    _need(state_in, "state_in", torch.float32, (N, H, dk, dv), dev)
    if accepted is not None:
        _need(accepted, "accepted", torch.int32, (N,), dev)
    if out is None and want_out:
        out = torch.empty((T, H, dv), dtype=dt, device=dev)
    if out is not None:
        _need(out, "out", dt, (T, H, dv), dev)
    if state_out is None and want_state:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if state_out is not None:
        _need(state_out, "state_out", torch.float32, (N, H, dk, dv), dev)
    prob = make_problem(N, T, T // N, H, dk, dv, dt, g_min)
    st = lib().kda_decode_replay(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(state_in),
                                 _ptr(accepted), _ptr(state_out), _ptr(out), ctypes.byref(prob), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_replay")
    return out, state_out


def kda_prologue(xq, xk, xv, wq, wk, wv, cu_seqlens=None, num_seqs: Optional[int] = None, q=None, k=None, v=None,
                 stream=None):
    """Layer prologue (see include/kda.h): short causal convolution, Swish and (q, k) regularised
    L2 normalisation of the projections xq, xk [T, H, d_k] and xv [T, H, d_v]; conv weights
    w* [H, d, K] fp32 with K = 1..4; cu_seqlens [N+1] int32 or None (``num_seqs`` equal lengths,
    default 1).  Returns (q, k, v)."""
    T, H, dk = xk.shape
    dv = xv.shape[2]
    dev = xk.device
    dt = xk.dtype
    K = wq.shape[2]
    for name, t, shp in (("xq", xq, (T, H, dk)), ("xk", xk, (T, H, dk)), ("xv", xv, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    for name, t, shp in (("wq", wq, (H, dk, K)), ("wk", wk, (H, dk, K)), ("wv", wv, (H, dv, K))):
        _need(t, name, torch.float32, shp, dev)
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    else:
        N = 1 if num_seqs is None else int(num_seqs)
    q = torch.empty_like(xq) if q is None else q
    k = torch.empty_like(xk) if k is None else k
    v = torch.empty_like(xv) if v is None else v
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp, dev)
    prob = make_problem(N, T, 0, H, dk, dv, dt)
    st = lib().kda_prologue(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv), ctypes.c_int32(K),
                            _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), ctypes.byref(prob), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prologue")
    return q, k, v


def kda_epilogue(o, gate, weight, eps: float = 1e-5, y=None, stream=None):
    """Layer epilogue (see include/kda.h): head-wise RMSNorm of o [T, H, d_v] with weight [d_v]
    fp32, times sigmoid(gate) [T, H, d_v].  ``y`` may be ``o`` (in place).  Returns y."""
    T, H, dv = o.shape
    dev = o.device
    dt = o.dtype
    _need(gate, "gate", dt, (T, H, dv), dev)
    _need(weight, "weight", torch.float32, (dv,), dev)
    y = torch.empty_like(o) if y is None else y
    _need(y, "y", dt, (T, H, dv), dev)
    prob = make_problem(1, T, 0, H, dv, dv, dt)
    st = lib().kda_epilogue(_ptr(o), _ptr(gate), _ptr(weight), ctypes.c_float(eps), _ptr(y), ctypes.byref(prob),
                            _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_epilogue")
    return y


def kda_workspace_status(workspace, stream=None) -> int:
    """Synchronise and return the device-side check status of a forward workspace."""
    return int(lib().kda_workspace_status(_ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream)))


def kda_static_scratch_status(stream=None) -> int:
    """Synchronise and return the device-side check status of the last kda_forward_static_scratch
    call in the current context."""
    return int(lib().kda_static_scratch_status(_stream(stream)))


def kda_abi_version() -> int:
    return int(lib().kda_abi_version())


def kda_profile_enable(enable: bool = True) -> None:
    """Start (or stop) recording per-kernel device time for launches made through the C ABI."""
    lib().kda_profile_enable(1 if enable else 0)


def kda_profile_read() -> dict:
    """{kernel name: (launches, total device ms)} since the last kda_profile_enable."""
    buf = (KdaKernelTime * 64)()
    n = lib().kda_profile_read(buf, 64)
    if n < 0:
        raise KdaError(KDA_ERR_CUDA, "kda_profile_read")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(min(n, 64))}
