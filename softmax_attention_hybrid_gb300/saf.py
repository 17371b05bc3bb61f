"""Thin Python binding of the C ABI in include/saf.h (ctypes).

The functions here have the C names and only marshal arguments: torch CUDA
tensors become device pointers, the current torch stream becomes the
cudaStream_t, and a nonzero status becomes SafError. Every step of the layer
runs in the CUDA library; if libsaf.so is missing, importing this module
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsaf.so")

SAF_BF16 = 0
SAF_FP32 = 1

SAF_OK = 0
SAF_EINVAL = -1
SAF_EALIGN = -2
SAF_EUNSUPPORTED = -3
SAF_ELAUNCH = -4
SAF_EWORKSPACE = -5
SAF_ETIMEOUT = -6
SAF_ECUDA = -8
SAF_ESCRATCH = -9

# Every symbol that include/saf.h declares.
EXPORTED = ("saf_attn_workspace_bytes", "saf_attn_fwd", "saf_attn_bwd", "saf_device_status",
            "saf_error_string", "saf_version", "saf_set_trace_events", "saf_launch_count",
            "saf_attn_fwd_noalloc", "saf_fit_workspace_bytes", "saf_fit_compact",
            "saf_pattern_grad", "saf_attn_fwd_gqa", "saf_attn_bwd_gqa", "saf_fit_stats_workspace_bytes",
            "saf_fit_target_stats", "saf_fit_from_target_workspace_bytes", "saf_fit_from_target",
            "saf_attn_fwd_diag", "saf_frozen_state_bytes", "saf_frozen_prepare", "saf_attn_fwd_prepared",
            "saf_attn_bwd_prepared", "saf_pattern_grad_tc_workspace_bytes", "saf_pattern_grad_tc")

SAF_KERNEL_NONE = 0
SAF_KERNEL_LOGNORM = 1
SAF_KERNEL_FWD = 2
SAF_KERNEL_BWD_DELTA = 3
SAF_KERNEL_BWD_KV = 4
SAF_KERNEL_BWD_Q = 5
SAF_KERNEL_BWD = 6
SAF_KERNEL_DQ_FINISH = 7
SAF_KERNEL_PATTERN_PREP = 8
SAF_KERNEL_PATTERN_GRAD = 9


class SafError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status} ({_lib.saf_error_string(status).decode()})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m softmax_attention_hybrid_gb300.build_lib`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.saf_attn_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.saf_attn_workspace_bytes.restype = sz
    lib.saf_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.saf_attn_fwd.restype = i
    lib.saf_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, vp, vp, vp]
    lib.saf_attn_fwd_noalloc.restype = i
    lib.saf_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
    lib.saf_fit_stats_workspace_bytes.restype = sz
    lib.saf_fit_stats_workspace_bytes.argtypes = [i, i]
    lib.saf_fit_target_stats.restype = i
    lib.saf_fit_target_stats.argtypes = [vp, i, i, vp, vp, vp, vp, sz, vp]
    lib.saf_fit_from_target_workspace_bytes.restype = sz
    lib.saf_fit_from_target_workspace_bytes.argtypes = [i, i]
    lib.saf_fit_from_target.restype = i
    lib.saf_fit_from_target.argtypes = [vp, i, i, i, ctypes.c_float, ctypes.c_float, vp, vp, vp, vp, vp, sz, vp]
    lib.saf_frozen_state_bytes.restype = sz
    lib.saf_frozen_state_bytes.argtypes = [i, i, i]
    lib.saf_frozen_prepare.restype = i
    lib.saf_frozen_prepare.argtypes = [vp, vp, i, vp, i, i, i, vp, sz, vp]
    lib.saf_attn_fwd_prepared.restype = i
    lib.saf_attn_fwd_prepared.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.saf_attn_bwd_prepared.restype = i
    lib.saf_attn_bwd_prepared.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, vp, vp, vp,
                                          vp, sz, vp]
    lib.saf_attn_fwd_diag.restype = i
    lib.saf_attn_fwd_diag.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, vp, vp, vp, sz, vp, i,
                                      ctypes.c_uint]
    lib.saf_attn_fwd_gqa.restype = i
    lib.saf_attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.saf_attn_bwd_gqa.restype = i
    lib.saf_attn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
    lib.saf_attn_bwd.restype = i
    lib.saf_device_status.argtypes = [vp, vp]
    lib.saf_device_status.restype = i
    lib.saf_error_string.argtypes = [i]
    lib.saf_error_string.restype = ctypes.c_char_p
    lib.saf_version.argtypes = []
    lib.saf_version.restype = i
    lib.saf_set_trace_events.argtypes = [i, vp, vp]
    lib.saf_set_trace_events.restype = i
    lib.saf_launch_count.argtypes = []
    lib.saf_launch_count.restype = ctypes.c_ulonglong
    lib.saf_fit_workspace_bytes.argtypes = [i, i]
    lib.saf_fit_workspace_bytes.restype = sz
    lib.saf_fit_compact.argtypes = [vp, vp, i, i, i, ctypes.c_float, vp, vp, vp, vp, sz, vp]
    lib.saf_fit_compact.restype = i
    lib.saf_pattern_grad.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, vp, vp, vp]
    lib.saf_pattern_grad.restype = i
    lib.saf_pattern_grad_tc_workspace_bytes.argtypes = [i, i, i, i]
    lib.saf_pattern_grad_tc_workspace_bytes.restype = sz
    lib.saf_pattern_grad_tc.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, vp, vp, vp, sz, vp]
    lib.saf_pattern_grad_tc.restype = i
    return lib


_lib = _load()


def library():
    """The loaded ctypes handle of libsaf.so."""
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SAF_BF16
    if t.dtype == torch.float32:
        return SAF_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _frozen_bytes(frozen, H):
    if frozen is None:
        return None
    vals = [1 if int(x) else 0 for x in (frozen.tolist() if torch.is_tensor(frozen) else frozen)]
    if len(vals) != H:
        raise ValueError("frozen mask must have H entries")
    return (ctypes.c_uint8 * H)(*vals)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def saf_error_string(status: int) -> str:
    return _lib.saf_error_string(int(status)).decode()


def saf_version() -> int:
    return _lib.saf_version()


def saf_attn_workspace_bytes(B, H, T, d, dtype, backward) -> int:
    dt = SAF_BF16 if dtype in (torch.bfloat16, SAF_BF16, "bf16") else SAF_FP32
    return int(_lib.saf_attn_workspace_bytes(int(B), int(H), int(T), int(d), dt, 1 if backward else 0))


def alloc_workspace(B, H, T, d, dtype, backward, device="cuda"):
    """A workspace buffer for saf_attn_fwd / saf_attn_bwd (256-byte aligned by torch)."""
    n = saf_attn_workspace_bytes(B, H, T, d, dtype, backward)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def saf_attn_fwd(q, k, v, a, r, frozen, o=None, lse=None, workspace=None, stream=None):
    """Forward pass; returns (o, lse). q, k, v: [B, H, T, d] CUDA tensors;
    a, r: [H, ld_prior] fp32 CUDA tensors (or None when nothing is frozen);
    frozen: H flags (list or tensor, read on the host)."""
    B, H, T, d = v.shape
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, False, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(r), int(ld), _frozen_bytes(frozen, H),
                           B, H, T, d, _dt(v), _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_fwd")
    return o, lse


def saf_attn_fwd_diag(q, k, v, a, r, frozen, withhold, wait_limit_us, o=None, lse=None, workspace=None,
                      stream=None):
    """Diagnostic forward for testing failure detection: with withhold=1 the
    kernel's producer publishes no work item and every bounded wait expires
    after wait_limit_us; returns (o, lse, workspace). Read the result with
    saf_device_status(workspace)."""
    B, H, T, d = v.shape
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, False, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_fwd_diag(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(r), int(ld), _frozen_bytes(frozen, H),
                                B, H, T, d, _dt(v), _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                _stream(stream), int(withhold), int(wait_limit_us))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_fwd_diag")
    return o, lse, workspace


def saf_attn_fwd_noalloc(q, k, v, a, r, frozen, o=None, lse=None, stream=None):
    """Forward pass without a workspace, for callers that cannot allocate
    device memory: the library uses its fixed 8 MiB device scratch instead.
    Same outputs as saf_attn_fwd; raises SafError (SAF_ESCRATCH) when the
    problem does not fit. Calls on one device share that scratch, so they
    must be ordered on one stream."""
    B, H, T, d = v.shape
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(r), int(ld), _frozen_bytes(frozen, H),
                                   B, H, T, d, _dt(v), _ptr(o), _ptr(lse), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_fwd_noalloc")
    return o, lse


def saf_attn_bwd(q, k, v, o, do, lse, a, r, frozen, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward pass; returns (dq, dk, dv)."""
    B, H, T, d = v.shape
    dq = torch.empty_like(v) if dq is None else dq
    dk = torch.empty_like(v) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, True, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(a), _ptr(r), int(ld),
                           _frozen_bytes(frozen, H), B, H, T, d, _dt(v), _ptr(dq), _ptr(dk), _ptr(dv),
                           _ptr(workspace), workspace.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_bwd")
    return dq, dk, dv


def _gqa_shape(q, v, frozen):
    B, Hkv, T, d = v.shape
    if q is not None:
        H = q.shape[1]
    elif frozen is not None:
        H = len(frozen)
    else:
        raise ValueError("q is needed unless the frozen mask gives H")
    return B, H, Hkv, T, d


def saf_attn_fwd_gqa(q, k, v, a, r, frozen, o=None, lse=None, workspace=None, stream=None):
    """Grouped-query forward; returns (o, lse). q: [B, H, T, d]; k, v:
    [B, Hkv, T, d] with H a multiple of Hkv (query head h reads key/value head
    h // (H // Hkv)); a, r, frozen per query head, as for saf_attn_fwd."""
    B, H, Hkv, T, d = _gqa_shape(q, v, frozen)
    if o is None:
        o = torch.empty((B, H, T, d), dtype=v.dtype, device=v.device)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, False, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(r), int(ld), _frozen_bytes(frozen, H),
                               B, H, Hkv, T, d, _dt(v), _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                               _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_fwd_gqa")
    return o, lse


def saf_attn_bwd_gqa(q, k, v, o, do, lse, a, r, frozen, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Grouped-query backward; returns dq [B, H, T, d] and dk, dv [B, Hkv, T, d]
    (a shared head's gradient is the sum over its query heads)."""
    B, H, Hkv, T, d = _gqa_shape(q, v, frozen)
    dq = torch.empty((B, H, T, d), dtype=v.dtype, device=v.device) if dq is None else dq
    dk = torch.empty_like(v) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, True, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(a), _ptr(r), int(ld),
                               _frozen_bytes(frozen, H), B, H, Hkv, T, d, _dt(v), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_bwd_gqa")
    return dq, dk, dv


def saf_frozen_prepare(a, r, frozen, T, dtype, state=None, stream=None):
    """Fill (and return) the prepared frozen-pattern state of a, r ([H, ld_prior]
    fp32 CUDA tensors) for sequences of length T in `dtype`."""
    H = a.shape[0]
    dt = SAF_BF16 if dtype in (torch.bfloat16, SAF_BF16, "bf16") else SAF_FP32
    n = int(_lib.saf_frozen_state_bytes(H, int(T), dt))
    if state is None:
        state = torch.empty(max(n, 256), dtype=torch.uint8, device=a.device)
    st = _lib.saf_frozen_prepare(_ptr(a), _ptr(r), int(a.shape[1]), _frozen_bytes(frozen, H), H, int(T), dt,
                                 _ptr(state), state.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_frozen_prepare")
    return state


def saf_attn_fwd_prepared(q, k, v, a, r, frozen, state, o=None, lse=None, workspace=None, stream=None):
    """Forward with the frozen-pattern data from a prepared state (grouped-query
    shapes allowed: k, v [B, Hkv, T, d]); returns (o, lse)."""
    B, H, Hkv, T, d = _gqa_shape(q, v, frozen)
    if o is None:
        o = torch.empty((B, H, T, d), dtype=v.dtype, device=v.device)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, False, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_fwd_prepared(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(r), int(ld), _frozen_bytes(frozen, H),
                                    _ptr(state), B, H, Hkv, T, d, _dt(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                    workspace.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_fwd_prepared")
    return o, lse


def saf_attn_bwd_prepared(q, k, v, o, do, lse, a, r, frozen, state, dq=None, dk=None, dv=None, workspace=None,
                          stream=None):
    """Backward with the frozen-pattern data from a prepared state; returns (dq, dk, dv)."""
    B, H, Hkv, T, d = _gqa_shape(q, v, frozen)
    dq = torch.empty((B, H, T, d), dtype=v.dtype, device=v.device) if dq is None else dq
    dk = torch.empty_like(v) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = alloc_workspace(B, H, T, d, v.dtype, True, v.device)
    ld = a.shape[1] if a is not None else T
    st = _lib.saf_attn_bwd_prepared(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(a), _ptr(r),
                                    int(ld), _frozen_bytes(frozen, H), _ptr(state), B, H, Hkv, T, d, _dt(v),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                                    _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_attn_bwd_prepared")
    return dq, dk, dv


def saf_set_trace_events(kernel: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event `start`/`stop` around every launch of `kernel`
    (a SAF_KERNEL_* id) from now on; kernel 0 or None events switch it off."""
    sp = ctypes.c_void_p(start.cuda_event) if start is not None else None
    ep = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    st = _lib.saf_set_trace_events(int(kernel), sp, ep)
    if st != SAF_OK:
        raise SafError(st, "saf_set_trace_events")


def saf_launch_count() -> int:
    return int(_lib.saf_launch_count())


def saf_device_status(workspace, stream=None) -> int:
    return int(_lib.saf_device_status(_ptr(workspace), _stream(stream)))


def saf_fit_workspace_bytes(H, T) -> int:
    return int(_lib.saf_fit_workspace_bytes(int(H), int(T)))


def saf_fit_compact(eta_abs, eta_rel, steps=400, lr=0.05, a=None, r=None, loss=None, workspace=None, stream=None):
    """Fit a, r of Eq. 3 to target marginals eta_abs, eta_rel (fp32 CUDA tensors
    [H, T]); returns (a, r, loss) as fp32 CUDA tensors [H, T], [H, T], [H]."""
    H, T = eta_abs.shape
    dev = eta_abs.device
    a = torch.empty((H, T), dtype=torch.float32, device=dev) if a is None else a
    r = torch.empty((H, T), dtype=torch.float32, device=dev) if r is None else r
    loss = torch.empty((H,), dtype=torch.float32, device=dev) if loss is None else loss
    if workspace is None:
        workspace = torch.empty(max(saf_fit_workspace_bytes(H, T), 256), dtype=torch.uint8, device=dev)
    st = _lib.saf_fit_compact(_ptr(eta_abs), _ptr(eta_rel), H, T, int(steps), float(lr), _ptr(a), _ptr(r),
                              _ptr(loss), _ptr(workspace), workspace.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_fit_compact")
    return a, r, loss


def saf_fit_target_stats(A, stream=None):
    """eta_abs, eta_rel [H, T] and negent [H] of the floored, row-normalised
    targets of A (fp32 CUDA tensor [H, T, T])."""
    H, T, _ = A.shape
    dev = A.device
    ea = torch.empty((H, T), dtype=torch.float32, device=dev)
    er = torch.empty((H, T), dtype=torch.float32, device=dev)
    ng = torch.empty((H,), dtype=torch.float32, device=dev)
    ws = torch.empty(max(int(_lib.saf_fit_stats_workspace_bytes(H, T)), 256), dtype=torch.uint8, device=dev)
    st = _lib.saf_fit_target_stats(_ptr(A), H, T, _ptr(ea), _ptr(er), _ptr(ng), _ptr(ws), ws.numel(),
                                   _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_fit_target_stats")
    return ea, er, ng


def saf_fit_from_target(A, steps=400, lr=0.05, tol=0.2, stream=None):
    """Fit every head of A (fp32 CUDA tensor [H, T, T]) from its measured
    pattern to accept / reject on the device; returns a, r [H, T], kappa [H]
    and accept [H] (uint8)."""
    H, T, _ = A.shape
    dev = A.device
    a = torch.empty((H, T), dtype=torch.float32, device=dev)
    r = torch.empty((H, T), dtype=torch.float32, device=dev)
    kappa = torch.empty((H,), dtype=torch.float32, device=dev)
    accept = torch.empty((H,), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(int(_lib.saf_fit_from_target_workspace_bytes(H, T)), 256), dtype=torch.uint8, device=dev)
    st = _lib.saf_fit_from_target(_ptr(A), H, T, int(steps), float(lr), float(tol), _ptr(a), _ptr(r), _ptr(kappa),
                                  _ptr(accept), _ptr(ws), ws.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_fit_from_target")
    return a, r, kappa, accept


def saf_pattern_grad(v, do, o, lse, a, r, frozen, da=None, dr=None, stream=None):
    """Gradients of a and r of the frozen heads (fp32 CUDA tensors [H, T])."""
    B, H, T, d = v.shape
    da = torch.empty((H, T), dtype=torch.float32, device=v.device) if da is None else da
    dr = torch.empty((H, T), dtype=torch.float32, device=v.device) if dr is None else dr
    st = _lib.saf_pattern_grad(_ptr(v), _ptr(do), _ptr(o), _ptr(lse), _ptr(a), _ptr(r), a.shape[-1],
                               _frozen_bytes(frozen, H), B, H, T, d, _dt(v), _ptr(da), _ptr(dr), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_pattern_grad")
    return da, dr


def saf_pattern_grad_tc_workspace_bytes(B, H, T, n_frozen):
    return int(_lib.saf_pattern_grad_tc_workspace_bytes(B, H, T, n_frozen))


def saf_pattern_grad_tc(v, do, o, lse, a, r, frozen, da=None, dr=None, workspace=None, stream=None):
    """Gradients of a and r of the frozen heads on the tensor cores (bf16 v, do, o
    [B, H, T, d], d = 64, 96 or 128); fp32 CUDA tensors [H, T], the same bits on
    every run.
    `workspace` (uint8 CUDA tensor) is allocated when not given."""
    B, H, T, d = v.shape
    fz = _frozen_bytes(frozen, H)
    nf = sum(fz) if fz is not None else 0
    da = torch.empty((H, T), dtype=torch.float32, device=v.device) if da is None else da
    dr = torch.empty((H, T), dtype=torch.float32, device=v.device) if dr is None else dr
    if workspace is None:
        n = max(saf_pattern_grad_tc_workspace_bytes(B, H, T, nf), 256)
        workspace = torch.empty(n, dtype=torch.uint8, device=v.device)
    st = _lib.saf_pattern_grad_tc(_ptr(v), _ptr(do), _ptr(o), _ptr(lse), _ptr(a), _ptr(r), a.shape[-1], fz, B, H,
                                  T, d, _ptr(da), _ptr(dr), _ptr(workspace), workspace.numel(), _stream(stream))
    if st != SAF_OK:
        raise SafError(st, "saf_pattern_grad_tc")
    return da, dr
