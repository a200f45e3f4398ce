"""Kimi Delta Attention (KDA) prefill and decode on one GB300 (sm_103a).

This package is a thin binding over ``libkda.so`` (C ABI in include/kda.h):
the Python functions below carry the same names as the C entry points and do
argument marshalling only -- every step of the computation runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There is
no CPU fallback: if ``libkda.so`` has not been built, importing the binding's
entry points raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from ._build import LIB_PATH, build  # noqa: F401

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_DEVICE_CHECK, \
    KDA_ERR_TIMEOUT = range(6)
KDA_F32, KDA_BF16 = 0, 1
KDA_ALGO_AUTO, KDA_ALGO_RECURRENT, KDA_ALGO_CHUNKED, KDA_ALGO_CHUNKED_PER_STATE, \
    KDA_ALGO_CHUNKED_COOP, KDA_ALGO_CHUNKED_COOP_HALVES = range(6)

EXPORTS = ("kda_prefill_varlen", "kda_prefill_varlen_retain", "kda_decode", "kda_decode_spec",
           "kda_prefill_varlen_fused", "kda_decode_fused", "kda_fused_scratch_bytes",
           "kda_workspace_bytes",
           "kda_snapshot_count", "kda_device_status", "kda_status_string",
           "kda_last_launch_count")


class KdaArgs(ctypes.Structure):
    """Mirror of ``kda_args`` in include/kda.h."""
    _fields_ = [("B", ctypes.c_int32), ("T_total", ctypes.c_int32), ("H", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("algo", ctypes.c_int32),
                ("snaps_capacity", ctypes.c_int64), ("stream", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("ev_begin", ctypes.c_void_p), ("ev_end", ctypes.c_void_p)]


class KdaFusedArgs(ctypes.Structure):
    """Mirror of ``kda_fused_args`` in include/kda.h."""
    _fields_ = [("gate", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p), ("conv_pool", ctypes.c_void_p),
                ("conv_width", ctypes.c_int32), ("conv_act", ctypes.c_int32),
                ("norm_eps", ctypes.c_float), ("reserved", ctypes.c_int32)]


CONV_ACT = {"none": 0, "silu": 1}


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def lib(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is None or path:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(p)
        V, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        A = ctypes.POINTER(KdaArgs)
        L.kda_prefill_varlen.argtypes = [V, V, V, V, V, V, V, V, V, I32, V, A]
        L.kda_prefill_varlen.restype = ctypes.c_int
        L.kda_prefill_varlen_retain.argtypes = [V, V, V, V, V, V, V, V, V, I32, V, A]
        L.kda_prefill_varlen_retain.restype = ctypes.c_int
        L.kda_decode.argtypes = [V, V, V, V, V, V, V, V, I32, V, A]
        L.kda_decode.restype = ctypes.c_int
        L.kda_workspace_bytes.argtypes = [A]
        L.kda_workspace_bytes.restype = ctypes.c_size_t
        L.kda_snapshot_count.argtypes = [V, I32, I32]
        L.kda_snapshot_count.restype = I64
        L.kda_device_status.argtypes = [A, ctypes.POINTER(ctypes.c_uint32)]
        L.kda_device_status.restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_last_launch_count.argtypes = []
        L.kda_last_launch_count.restype = I32
        L.kda_decode_noalloc.argtypes = [V, V, V, V, V, V, V, V, I32, V, V, A]
        L.kda_decode_noalloc.restype = ctypes.c_int
        L.kda_decode_spec.argtypes = [V, V, V, V, V, V, V, V, I32, V, V, V, V, V, I32, A]
        L.kda_decode_spec.restype = ctypes.c_int
        F = ctypes.POINTER(KdaFusedArgs)
        L.kda_prefill_varlen_fused.argtypes = [V, V, V, V, V, V, V, V, V, I32, V, F, V,
                                               ctypes.c_size_t, A]
        L.kda_prefill_varlen_fused.restype = ctypes.c_int
        L.kda_decode_fused.argtypes = [V, V, V, V, V, V, V, V, I32, V, F, A]
        L.kda_decode_fused.restype = ctypes.c_int
        L.kda_fused_scratch_bytes.argtypes = [A]
        L.kda_fused_scratch_bytes.restype = ctypes.c_size_t
        if path:
            return L
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


# ---------------------------------------------------------------- marshalling

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkda must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_args(*, B, T_total, H, dk, dv, n_slots, dtype, algo=KDA_ALGO_AUTO, snaps_capacity=0,
              stream=None, workspace=None, events=None) -> KdaArgs:
    a = KdaArgs(B=B, T_total=T_total, H=H, dk=dk, dv=dv, n_slots=n_slots, dtype=dtype,
                algo=algo, snaps_capacity=snaps_capacity)
    a.stream = _stream_ptr(stream)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    if events is not None:
        a.ev_begin = events[0].cuda_event
        a.ev_end = events[1].cuda_event
    return a


def workspace_for(B: int, H: int, n_slots: int, device="cuda"):
    """A zero-filled workspace tensor large enough for (B, H, n_slots)."""
    import torch
    a = KdaArgs(B=B, H=H, n_slots=n_slots)
    n = lib().kda_workspace_bytes(ctypes.byref(a))
    return torch.zeros(max(int(n), 256), dtype=torch.uint8, device=device)


def kda_workspace_bytes(B: int, H: int, n_slots: int) -> int:
    a = KdaArgs(B=B, H=H, n_slots=n_slots)
    return int(lib().kda_workspace_bytes(ctypes.byref(a)))


def kda_snapshot_count(cu_seqlens_host, snap_interval: int) -> int:
    import torch
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous().cpu()
    n = lib().kda_snapshot_count(cu.data_ptr(), cu.numel() - 1, int(snap_interval))
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_snapshot_count")
    return int(n)


def kda_prefill_varlen(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, out,
                       snap_interval: int = 0, snaps=None, *, workspace, stream=None,
                       algo: int = KDA_ALGO_AUTO, events=None) -> None:
    """Varlen chunked prefill (see kda_prefill_varlen in include/kda.h).
    All tensors are CUDA tensors; raises KdaError on a nonzero status."""
    a = make_args(B=cu_seqlens.numel() - 1, T_total=q.shape[0], H=q.shape[1], dk=q.shape[2],
                  dv=v.shape[2], n_slots=state_pool.shape[0], dtype=_dtype_code(q), algo=algo,
                  snaps_capacity=0 if snaps is None else snaps.shape[0], stream=stream,
                  workspace=workspace, events=events)
    st = lib().kda_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(cu_seqlens), _ptr(init_slots), _ptr(state_pool), _ptr(out),
                                  int(snap_interval), _ptr(snaps), ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_varlen")


def kda_prefill_varlen_retain(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, out,
                              snap_interval: int, snap_slots, *, workspace, stream=None,
                              algo: int = KDA_ALGO_AUTO, events=None) -> None:
    """kda_prefill_varlen with a retention map (see kda_prefill_varlen_retain
    in include/kda.h): snap_slots[s] is the pool slot of snapshot s, or -1."""
    a = make_args(B=cu_seqlens.numel() - 1, T_total=q.shape[0], H=q.shape[1], dk=q.shape[2],
                  dv=v.shape[2], n_slots=state_pool.shape[0], dtype=_dtype_code(q), algo=algo,
                  snaps_capacity=0 if snap_slots is None else snap_slots.numel(), stream=stream,
                  workspace=workspace, events=events)
    st = lib().kda_prefill_varlen_retain(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         _ptr(cu_seqlens), _ptr(init_slots), _ptr(state_pool),
                                         _ptr(out), int(snap_interval), _ptr(snap_slots),
                                         ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_varlen_retain")


def kda_decode(q, k, v, g, beta, slot_ids, state_pool, out, n_tok: int = 1,
               per_tok_states=None, *, workspace, stream=None, events=None) -> None:
    """In-place decode of n_tok tokens per sequence (see kda_decode in include/kda.h)."""
    a = make_args(B=slot_ids.numel(), T_total=q.shape[0], H=q.shape[1], dk=q.shape[2],
                  dv=v.shape[2], n_slots=state_pool.shape[0], dtype=_dtype_code(q),
                  stream=stream, workspace=workspace, events=events)
    st = lib().kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(slot_ids),
                          _ptr(state_pool), _ptr(out), int(n_tok), _ptr(per_tok_states),
                          ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")


def kda_decode_spec(q, k, v, g, beta, slot_ids, state_pool, out, n_tok: int, k_prev=None,
                    v_prev=None, g_prev=None, beta_prev=None, accepted_prev=None,
                    n_prev: int = 0, *, workspace, stream=None, events=None,
                    H: Optional[int] = None, dk: Optional[int] = None,
                    dv: Optional[int] = None, dtype: Optional[int] = None) -> None:
    """Speculative verify with the commit of the previous step folded in (see
    kda_decode_spec in include/kda.h): replays accepted_prev[n] tokens of the
    previous step onto slot_ids[n], writes that state, then writes the outputs
    of this step's n_tok tokens without advancing the slot.  With n_tok == 0
    (commit only) q, k, v, g, beta and out may be None and the shape keywords
    H / dk / dv / dtype describe the call instead."""
    ref = q if q is not None else k_prev
    vref = v if v is not None else v_prev
    a = make_args(B=slot_ids.numel(), T_total=slot_ids.numel() * int(n_tok),
                  H=H or ref.shape[1], dk=dk or ref.shape[2], dv=dv or vref.shape[2],
                  n_slots=state_pool.shape[0],
                  dtype=dtype if dtype is not None else _dtype_code(ref),
                  stream=stream, workspace=workspace, events=events)
    st = lib().kda_decode_spec(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(slot_ids),
                               _ptr(state_pool), _ptr(out), int(n_tok), _ptr(k_prev),
                               _ptr(v_prev), _ptr(g_prev), _ptr(beta_prev), _ptr(accepted_prev),
                               int(n_prev), ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_spec")


def kda_decode_noalloc(q, k, v, g, beta, slot_ids, state_pool, out, n_tok: int = 1,
                       per_tok_states=None, err_bits=None, *, stream=None):
    """kda_decode for dk = dv = 128 without a workspace: for callers that may
    not allocate device memory (see kda_decode_noalloc in include/kda.h).
    err_bits: int32/uint32 CUDA tensor of one element that collects the
    device-side check bits (the caller clears it).  When it is not given, a
    zeroed one is created on the device of ``out`` (the only allocation here,
    from torch's cache, in Python, not in the library), so that a bad or
    duplicate slot is never silently dropped.  Returns err_bits."""
    if err_bits is None:
        import torch
        err_bits = torch.zeros(1, dtype=torch.int32, device=out.device)
    a = make_args(B=slot_ids.numel(), T_total=q.shape[0], H=q.shape[1], dk=q.shape[2],
                  dv=v.shape[2], n_slots=state_pool.shape[0], dtype=_dtype_code(q),
                  stream=stream)
    st = lib().kda_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(slot_ids), _ptr(state_pool), _ptr(out), int(n_tok),
                                  _ptr(per_tok_states), _ptr(err_bits), ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_noalloc")
    return err_bits


def _fused_args(gate, conv_w, norm_w, conv_pool, conv_act="none", norm_eps=1e-6):
    for t in (conv_w, norm_w):
        if t is not None and t.dtype.is_floating_point and t.element_size() != 4:
            raise TypeError("conv_w and norm_w are fp32")
    return KdaFusedArgs(gate=_ptr(gate), conv_w=_ptr(conv_w), norm_w=_ptr(norm_w),
                        conv_pool=_ptr(conv_pool), conv_width=conv_w.shape[-1],
                        conv_act=CONV_ACT[conv_act], norm_eps=float(norm_eps), reserved=0)


def kda_fused_scratch_bytes(T_total: int, H: int, dk: int, dv: int, dtype: int) -> int:
    a = KdaArgs(T_total=T_total, H=H, dk=dk, dv=dv, dtype=dtype)
    return int(lib().kda_fused_scratch_bytes(ctypes.byref(a)))


def kda_prefill_varlen_fused(xq, xk, xv, g, beta, gate, conv_w, norm_w, cu_seqlens, init_slots,
                             state_pool, conv_pool, out, snap_interval: int = 0, snaps=None, *,
                             workspace, scratch=None, conv_act="none", norm_eps=1e-6,
                             stream=None, algo: int = KDA_ALGO_AUTO, events=None):
    """The prefill with the short convolution before it and the gated RMSNorm
    after it (see kda_prefill_varlen_fused in include/kda.h).  xq, xk, xv are
    the raw inputs; conv_w [H, 2dk+dv, 4] and norm_w [dv] fp32; conv_pool
    [n_slots, H, 2dk+dv, 3] in the input dtype.  scratch: a uint8 CUDA tensor
    of kda_fused_scratch_bytes(...) bytes (made here when not given).
    Returns the scratch tensor."""
    import torch
    dt = _dtype_code(xq)
    T, H, dk = xq.shape
    dv = xv.shape[2]
    if scratch is None:
        n = kda_fused_scratch_bytes(T, H, dk, dv, dt)
        scratch = torch.empty(max(n, 16), dtype=torch.uint8, device=xq.device)
    a = make_args(B=cu_seqlens.numel() - 1, T_total=T, H=H, dk=dk, dv=dv,
                  n_slots=state_pool.shape[0], dtype=dt, algo=algo,
                  snaps_capacity=0 if snaps is None else snaps.shape[0], stream=stream,
                  workspace=workspace, events=events)
    f = _fused_args(gate, conv_w, norm_w, conv_pool, conv_act, norm_eps)
    st = lib().kda_prefill_varlen_fused(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta),
                                        _ptr(cu_seqlens), _ptr(init_slots), _ptr(state_pool),
                                        _ptr(out), int(snap_interval), _ptr(snaps),
                                        ctypes.byref(f), _ptr(scratch),
                                        scratch.numel() * scratch.element_size(),
                                        ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_varlen_fused")
    return scratch


def kda_decode_fused(xq, xk, xv, g, beta, gate, conv_w, norm_w, slot_ids, state_pool, conv_pool,
                     out, n_tok: int = 1, per_tok_states=None, *, workspace, conv_act="none",
                     norm_eps=1e-6, stream=None, events=None) -> None:
    """Decode with the short convolution and the gated RMSNorm in one launch
    (see kda_decode_fused in include/kda.h); dk = dv = 128."""
    a = make_args(B=slot_ids.numel(), T_total=xq.shape[0], H=xq.shape[1], dk=xq.shape[2],
                  dv=xv.shape[2], n_slots=state_pool.shape[0], dtype=_dtype_code(xq),
                  stream=stream, workspace=workspace, events=events)
    f = _fused_args(gate, conv_w, norm_w, conv_pool, conv_act, norm_eps)
    st = lib().kda_decode_fused(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(g), _ptr(beta), _ptr(slot_ids),
                                _ptr(state_pool), _ptr(out), int(n_tok), _ptr(per_tok_states),
                                ctypes.byref(f), ctypes.byref(a))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_fused")


def kda_device_status(workspace, stream=None):
    """(status, error bits) of device-side checks since the last query; clears them."""
    a = make_args(B=0, T_total=0, H=1, dk=128, dv=128, n_slots=1, dtype=KDA_BF16,
                  stream=stream, workspace=workspace)
    bits = ctypes.c_uint32(0)
    st = lib().kda_device_status(ctypes.byref(a), ctypes.byref(bits))
    return int(st), int(bits.value)


def kda_last_launch_count() -> int:
    return int(lib().kda_last_launch_count())
