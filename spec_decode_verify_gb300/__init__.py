"""Batched speculative-verify causal depthwise conv1d update on GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/convverify.h`` (library built in-tree by
``spec_decode_verify_gb300.build``).  This module only marshals torch tensors into pointers and
element strides; every step of the computation runs in the library's CUDA kernels.  There is no
CPU path: CPU tensors are rejected and a missing library raises.

    conv_verify(x, conv_state, weight, bias, out, window, layout=..., qk_channels=..., head_dim=...)
    conv_commit(conv_state, window, accept_len, layout=..., T=..., width=..., x=...)
    conv_prefill(x, conv_state, weight, bias, out, cu_seqlens, max_seqlen=..., qk_channels=..., head_dim=...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = ["conv_verify", "conv_commit", "conv_prefill", "verify_plan", "status_string", "load_library", "library_path",
           "CvError", "DENSE", "DEDUP", "HISTORY", "RECOMPUTE", "SEQ_BAD_SLOT", "SEQ_BAD_OFFSET", "SEQ_BAD_ACCEPT",
           "SEQ_TIMEOUT", "SEQ_BAD_SPAN", "SEQ_BAD_TREE"]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "_build", "libconvverify.so")

DENSE, DEDUP, HISTORY, RECOMPUTE = 1, 2, 3, 4
F32, BF16 = 0, 1
SEQ_BAD_SLOT, SEQ_BAD_OFFSET, SEQ_BAD_ACCEPT, SEQ_TIMEOUT, SEQ_BAD_SPAN, SEQ_BAD_TREE = 1, 2, 4, 8, 16, 32
MAX_T = 128

c_i32, c_i64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p


class VerifyArgs(ctypes.Structure):
    """Mirror of cv_verify_args."""
    _fields_ = [
        ("n_seq", c_i32), ("T", c_i32), ("dim", c_i32), ("width", c_i32), ("qk_channels", c_i32),
        ("head_dim", c_i32), ("dtype", c_i32), ("l2_eps", ctypes.c_float),
        ("x", c_vp), ("x_seq_stride", c_i64), ("x_tok_stride", c_i64),
        ("out", c_vp), ("out_seq_stride", c_i64), ("out_tok_stride", c_i64),
        ("conv_state", c_vp), ("n_slots", c_i32), ("state_cols", c_i32),
        ("state_slot_stride", c_i64), ("state_ch_stride", c_i64),
        ("cache_idx", c_vp), ("state_off", c_vp), ("weight", c_vp), ("bias", c_vp),
        ("window", c_vp), ("window_layout", c_i32), ("wait_polls", c_i32),
        ("win_seq_stride", c_i64), ("win_step_stride", c_i64), ("win_ch_stride", c_i64), ("win_col_stride", c_i64),
        ("err", c_vp), ("state_dtype", c_i32), ("parent", c_vp), ("cu_draft", c_vp), ("total_tokens", c_i32),
        ("state_col_stride", c_i64),
    ]


class CommitArgs(ctypes.Structure):
    """Mirror of cv_commit_args."""
    _fields_ = [
        ("n_seq", c_i32), ("T", c_i32), ("dim", c_i32), ("width", c_i32), ("dtype", c_i32), ("n_slots", c_i32),
        ("conv_state", c_vp), ("state_slot_stride", c_i64), ("state_ch_stride", c_i64),
        ("state_cols", c_i32), ("window_layout", c_i32), ("cache_idx", c_vp), ("window", c_vp),
        ("win_seq_stride", c_i64), ("win_step_stride", c_i64), ("win_ch_stride", c_i64), ("win_col_stride", c_i64),
        ("accept_len", c_vp), ("err", c_vp), ("x", c_vp), ("x_seq_stride", c_i64), ("x_tok_stride", c_i64),
        ("cu_draft", c_vp), ("total_tokens", c_i32), ("wait_polls", c_i32),
    ]


class PrefillArgs(ctypes.Structure):
    """Mirror of cv_prefill_args."""
    _fields_ = [
        ("n_seq", c_i32), ("dim", c_i32), ("width", c_i32), ("qk_channels", c_i32), ("head_dim", c_i32),
        ("dtype", c_i32), ("l2_eps", ctypes.c_float), ("total_tokens", c_i32), ("max_seqlen", c_i32),
        ("x", c_vp), ("x_tok_stride", c_i64), ("out", c_vp), ("out_tok_stride", c_i64), ("cu_seqlens", c_vp),
        ("conv_state", c_vp), ("n_slots", c_i32), ("state_cols", c_i32), ("state_slot_stride", c_i64),
        ("state_ch_stride", c_i64), ("cache_idx", c_vp), ("has_initial_state", c_vp), ("weight", c_vp),
        ("bias", c_vp), ("err", c_vp),
    ]


class LaunchPlan(ctypes.Structure):
    """Mirror of cv_launch_plan."""
    _fields_ = [("grid_x", c_i32), ("grid_y", c_i32), ("threads", c_i32), ("smem_bytes", c_i32),
                ("channels_per_block", c_i32), ("path", c_i32), ("stages", c_i32), ("token_groups", c_i32)]


class CvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load_library(path: Optional[str] = None):
    """Load the CUDA library (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (python -m spec_decode_verify_gb300.build)")
    lib = ctypes.CDLL(p)
    lib.cv_conv_verify.argtypes = [ctypes.POINTER(VerifyArgs), c_vp]
    lib.cv_conv_verify.restype = c_i32
    lib.cv_conv_commit.argtypes = [ctypes.POINTER(CommitArgs), c_vp]
    lib.cv_conv_commit.restype = c_i32
    lib.cv_conv_prefill.argtypes = [ctypes.POINTER(PrefillArgs), c_vp]
    lib.cv_conv_prefill.restype = c_i32
    lib.cv_verify_plan.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.POINTER(LaunchPlan)]
    lib.cv_verify_plan.restype = c_i32
    lib.cv_status_string.argtypes = [c_i32]
    lib.cv_status_string.restype = ctypes.c_char_p
    lib.cv_abi_version.argtypes = []
    lib.cv_abi_version.restype = c_i32
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().cv_status_string(int(status)).decode()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: expected bfloat16 or float32")


def _dev_ptr(t, name, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    return t.data_ptr()


def _need_shape(t, name, shape):
    """Shapes are checked here because the library sees only pointers: a buffer smaller than the
    sizes describe would be read or written past its end."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_int32(t, name, n=None, shape=None):
    """An int32 device array: contiguous, of the given shape, or holding at least n elements."""
    if t is None:
        return
    import torch
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 tensor")
    if shape is not None:
        _need_shape(t, name, shape)
    if n is not None and t.numel() < n:
        raise ValueError(f"{name} needs at least {n} elements, got {t.numel()}")


def _layout_code(layout) -> int:
    if layout in (DENSE, "dense"):
        return DENSE
    if layout in (DEDUP, "dedup"):
        return DEDUP
    if layout in (HISTORY, "history"):
        return HISTORY
    if layout in (RECOMPUTE, "recompute"):
        return RECOMPUTE
    raise ValueError(f"unknown window layout {layout!r}")


def _window_strides(window, layout: int):
    if layout in (HISTORY, RECOMPUTE) or window is None:  # no window buffer
        return 0, 0, 0, 0
    s = window.stride()
    if layout == DENSE:  # [n_seq, T, dim, W-1]
        return s[0], s[1], s[2], s[3]
    return s[0], s[2], s[1], s[2]  # dedup row [n_seq, dim, T+W-2]: step stride = column stride


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_verify_args(x, conv_state, weight, bias, out, window, *, layout, qk_channels, head_dim,
                     l2_eps=1e-6, cache_idx=None, state_off=None, err=None, parent=None, wait_polls=0,
                     cu_draft=None, T=None, check_device=True) -> VerifyArgs:
    """Build cv_verify_args from tensors.

    x [n_seq, T, dim] (channel stride 1, any seq/token strides), conv_state [n_slots, dim, S]
    (column stride 1; it may have the other dtype than x: mixed dtypes), weight [dim, W] contiguous,
    bias [dim] or None, out [n_seq, T, dim] (channel stride 1), window dense [n_seq, T, dim, W-1] or
    dedup [n_seq, dim, T+W-2] (any strides, the dtype of conv_state), or
    None with layout "history" (conv_state [n_slots, dim, S >= T+W-2] then receives the snapshot
    row and the next call reads at state_off = accept_len - 1) or "recompute" (outputs only; the
    commit rebuilds the state from x), cache_idx / state_off / err int32 [n_seq] or None, parent int32
    [n_seq, T] contiguous (tree verify, dense layout) or None.  wait_polls: the limit of the
    pipelined kernel's bounded waits (0 = the default; see cv_verify_args).

    Packed ragged drafts: cu_draft int32 [n_seq + 1]; x and out are then [total_tokens, dim] (token
    stride free, channel stride 1), sequence s owning rows cu_draft[s] .. cu_draft[s+1]-1, and T
    (required) is the largest draft count, the T of the window buffer."""
    lay = _layout_code(layout)
    ptr = _dev_ptr if check_device else (lambda t, n, required=True: None if t is None else t.data_ptr())
    varlen = cu_draft is not None
    if x.dim() != (2 if varlen else 3) or conv_state.dim() != 3 or weight.dim() != 2:
        raise ValueError("x must be [n_seq, T, dim] ([total_tokens, dim] with cu_draft), conv_state "
                         "[n_slots, dim, S] and weight [dim, W]")
    if varlen:
        if T is None:
            raise ValueError("packed drafts need T, the largest draft count")
        _need_int32(cu_draft, "cu_draft")
        if cu_draft.dim() != 1 or cu_draft.shape[0] < 1:
            raise ValueError("cu_draft must be [n_seq + 1]")
        n_seq, (total, dim) = cu_draft.shape[0] - 1, x.shape
        T = int(T)
    else:
        n_seq, T, dim = x.shape
        total = 0
    W = weight.shape[1]
    _need_shape(out, "out", x.shape)
    _need_shape(weight, "weight", (dim, W))
    _need_shape(bias, "bias", (dim,))
    if conv_state.shape[1] != dim:
        raise ValueError(f"conv_state must have dim = {dim} channels, got {conv_state.shape[1]}")
    if lay == DENSE:
        _need_shape(window, "window", (n_seq, T, dim, W - 1))
    elif lay == DEDUP:
        _need_shape(window, "window", (n_seq, dim, T + W - 2))
    for t, name in ((cache_idx, "cache_idx"), (state_off, "state_off"), (err, "err")):
        _need_int32(t, name, n=n_seq)
    _need_int32(parent, "parent", shape=(n_seq, T))
    if x.stride(-1) != 1 or out.stride(-1) != 1:
        raise ValueError("x and out need a unit innermost stride")
    # conv_state: columns contiguous, or (history layout) column-major rows [n_slots, S, dim] seen
    # as [n_slots, dim, S]; the library checks which strides it accepts
    st_col = 1 if conv_state.shape[2] == 1 else conv_state.stride(2)
    if not weight.is_contiguous() or (bias is not None and not bias.is_contiguous()):
        raise ValueError("weight and bias must be contiguous")
    ws = _window_strides(window, lay)
    return VerifyArgs(
        n_seq=n_seq, T=T, dim=dim, width=W, qk_channels=qk_channels, head_dim=head_dim, dtype=_dtype_code(x),
        l2_eps=l2_eps, x=ptr(x, "x", total > 0 or not varlen), x_seq_stride=0 if varlen else x.stride(0),
        x_tok_stride=x.stride(-2), out=ptr(out, "out", total > 0 or not varlen),
        out_seq_stride=0 if varlen else out.stride(0), out_tok_stride=out.stride(-2),
        conv_state=ptr(conv_state, "conv_state"), n_slots=conv_state.shape[0], state_cols=conv_state.shape[2],
        state_slot_stride=conv_state.stride(0), state_ch_stride=conv_state.stride(1),
        cache_idx=ptr(cache_idx, "cache_idx", False), state_off=ptr(state_off, "state_off", False),
        weight=ptr(weight, "weight"), bias=ptr(bias, "bias", False),
        window=ptr(window, "window", lay not in (HISTORY, RECOMPUTE)),
        window_layout=lay, wait_polls=int(wait_polls), win_seq_stride=ws[0], win_step_stride=ws[1], win_ch_stride=ws[2],
        win_col_stride=ws[3], err=ptr(err, "err", False),
        state_dtype=0 if conv_state.dtype == x.dtype else _dtype_code(conv_state) + 1,
        parent=ptr(parent, "parent", False), cu_draft=ptr(cu_draft, "cu_draft", False), total_tokens=total,
        state_col_stride=st_col)


def conv_verify(x, conv_state, weight, bias, out, window, *, layout, qk_channels, head_dim, l2_eps=1e-6,
                cache_idx=None, state_off=None, err=None, parent=None, wait_polls=0, cu_draft=None, T=None,
                stream=None) -> None:
    """Queue one batched verify on ``stream`` (default: torch's current stream).

    Writes out, window, conv_state (and err); raises CvError on an invalid argument.  With layout
    "history" pass window=None: the snapshots go into the state rows."""
    for t in (weight, out):
        if t.dtype != x.dtype:
            raise TypeError("x, weight and out must share one dtype")
    if window is not None and window.dtype != conv_state.dtype:
        raise TypeError("window must have the dtype of conv_state")
    _dtype_code(conv_state)
    if bias is not None and bias.dtype != x.dtype:
        raise TypeError("bias must have the dtype of x")
    a = make_verify_args(x, conv_state, weight, bias, out, window, layout=layout, qk_channels=qk_channels,
                         head_dim=head_dim, l2_eps=l2_eps, cache_idx=cache_idx, state_off=state_off, err=err,
                         parent=parent, wait_polls=wait_polls, cu_draft=cu_draft, T=T)
    rc = load_library().cv_conv_verify(ctypes.byref(a), _stream_ptr(stream))
    if rc != 0:
        raise CvError(rc, "cv_conv_verify")


def verify_plan(x, conv_state, weight, bias, out, window, *, layout, qk_channels, head_dim, l2_eps=1e-6,
                cache_idx=None, state_off=None, err=None, parent=None, cu_draft=None, T=None) -> LaunchPlan:
    """The launch cv_conv_verify would make (validates without touching the GPU)."""
    a = make_verify_args(x, conv_state, weight, bias, out, window, layout=layout, qk_channels=qk_channels,
                         head_dim=head_dim, l2_eps=l2_eps, cache_idx=cache_idx, state_off=state_off, err=err,
                         parent=parent, cu_draft=cu_draft, T=T, check_device=False)
    pl = LaunchPlan()
    rc = load_library().cv_verify_plan(ctypes.byref(a), ctypes.byref(pl))
    if rc != 0:
        raise CvError(rc, "cv_verify_plan")
    return pl


def make_commit_args(conv_state, window, accept_len, *, layout, T, width, cache_idx=None, err=None,
                     x=None, cu_draft=None, total_tokens=None, wait_polls=0, check_device=True) -> CommitArgs:
    """Build cv_commit_args.  Layout "recompute": window is None and x is the verify's input
    [n_seq, T, dim] (channel stride 1).  cu_draft: the matching verify's packed draft spans (x is
    then [total_tokens, dim]); accept_len[s] must lie in 1..T_s."""
    lay = _layout_code(layout)
    if x is not None and x.stride(-1) != 1:
        raise ValueError("x needs a unit channel stride")
    varlen = cu_draft is not None
    if varlen:
        _need_int32(cu_draft, "cu_draft", n=accept_len.shape[0] + 1)
        if total_tokens is None:
            total_tokens = x.shape[0] if x is not None else 0
    ptr = _dev_ptr if check_device else (lambda t, n, required=True: None if t is None else t.data_ptr())
    ws = _window_strides(window, lay)
    if conv_state.dim() != 3 or conv_state.stride(2) != 1:
        raise ValueError("conv_state must be [n_slots, dim, S] with a unit column stride")
    _need_int32(accept_len, "accept_len")
    if accept_len.dim() != 1:
        raise ValueError("accept_len must be [n_seq]")
    n_seq, dim = accept_len.shape[0], conv_state.shape[1]
    for t, name in ((cache_idx, "cache_idx"), (err, "err")):
        _need_int32(t, name, n=n_seq)
    if lay == DENSE:
        _need_shape(window, "window", (n_seq, T, dim, width - 1))
    elif lay == DEDUP:
        _need_shape(window, "window", (n_seq, dim, T + width - 2))
    elif varlen:
        if x is None or x.dim() != 2 or x.shape[1] != dim or x.shape[0] != total_tokens:
            raise ValueError(f"x must be [total_tokens, {dim}] with packed drafts")
    else:
        _need_shape(x, "x", (n_seq, T, dim))
    return CommitArgs(
        n_seq=accept_len.shape[0], T=T, dim=conv_state.shape[1], width=width, dtype=_dtype_code(conv_state),
        n_slots=conv_state.shape[0], conv_state=ptr(conv_state, "conv_state"),
        state_slot_stride=conv_state.stride(0), state_ch_stride=conv_state.stride(1),
        state_cols=conv_state.shape[2], window_layout=lay, cache_idx=ptr(cache_idx, "cache_idx", False),
        window=ptr(window, "window", lay != RECOMPUTE), win_seq_stride=ws[0], win_step_stride=ws[1],
        win_ch_stride=ws[2], win_col_stride=ws[3], accept_len=ptr(accept_len, "accept_len"),
        err=ptr(err, "err", False), x=ptr(x, "x", lay == RECOMPUTE and not (varlen and total_tokens == 0)),
        x_seq_stride=x.stride(0) if x is not None and not varlen else 0,
        x_tok_stride=x.stride(-2) if x is not None else 0,
        cu_draft=ptr(cu_draft, "cu_draft", False), total_tokens=int(total_tokens or 0), wait_polls=int(wait_polls))


def conv_commit(conv_state, window, accept_len, *, layout, T, width, cache_idx=None, err=None, x=None,
                cu_draft=None, total_tokens=None, wait_polls=0, stream=None) -> None:
    """Queue the commit: conv_state[slot] <- snapshot accept_len[s]-1 of sequence s (rebuilt from the
    kept window and x with layout "recompute")."""
    for t in (window, x):
        if t is not None and t.dtype != conv_state.dtype:
            raise TypeError("window / x and conv_state must share one dtype")
    a = make_commit_args(conv_state, window, accept_len, layout=layout, T=T, width=width, cache_idx=cache_idx,
                         err=err, x=x, cu_draft=cu_draft, total_tokens=total_tokens, wait_polls=wait_polls)
    rc = load_library().cv_conv_commit(ctypes.byref(a), _stream_ptr(stream))
    if rc != 0:
        raise CvError(rc, "cv_conv_commit")


def make_prefill_args(x, conv_state, weight, bias, out, cu_seqlens, *, max_seqlen, qk_channels, head_dim,
                      l2_eps=1e-6, cache_idx=None, has_initial_state=None, err=None, check_device=True) -> PrefillArgs:
    """Build cv_prefill_args from tensors.

    x, out [total_tokens, dim] (channel stride 1, any token stride), conv_state [n_slots, dim, S]
    (column stride 1), weight [dim, W] contiguous, bias [dim] or None, cu_seqlens int32
    [n_seq + 1], cache_idx / has_initial_state / err int32 [n_seq] or None; max_seqlen bounds
    every sequence's length (host int)."""
    ptr = _dev_ptr if check_device else (lambda t, n, required=True: None if t is None else t.data_ptr())
    if x.dim() != 2 or conv_state.dim() != 3 or weight.dim() != 2:
        raise ValueError("x must be [total_tokens, dim], conv_state [n_slots, dim, S] and weight [dim, W]")
    total, dim = x.shape
    _need_shape(out, "out", x.shape)
    _need_shape(weight, "weight", (dim, weight.shape[1]))
    _need_shape(bias, "bias", (dim,))
    if conv_state.shape[1] != dim:
        raise ValueError(f"conv_state must have dim = {dim} channels, got {conv_state.shape[1]}")
    _need_int32(cu_seqlens, "cu_seqlens")
    if cu_seqlens.dim() != 1 or cu_seqlens.shape[0] < 1:
        raise ValueError("cu_seqlens must be [n_seq + 1]")
    for t, name in ((cache_idx, "cache_idx"), (has_initial_state, "has_initial_state"), (err, "err")):
        _need_int32(t, name, n=cu_seqlens.shape[0] - 1)
    if x.stride(1) != 1 or out.stride(1) != 1 or conv_state.stride(2) != 1:
        raise ValueError("x, out and conv_state need a unit innermost stride")
    if not weight.is_contiguous() or (bias is not None and not bias.is_contiguous()):
        raise ValueError("weight and bias must be contiguous")
    return PrefillArgs(
        n_seq=cu_seqlens.shape[0] - 1, dim=dim, width=weight.shape[1], qk_channels=qk_channels, head_dim=head_dim,
        dtype=_dtype_code(x), l2_eps=l2_eps, total_tokens=total, max_seqlen=int(max_seqlen),
        x=ptr(x, "x", total > 0), x_tok_stride=x.stride(0), out=ptr(out, "out", total > 0),
        out_tok_stride=out.stride(0), cu_seqlens=ptr(cu_seqlens, "cu_seqlens"),
        conv_state=ptr(conv_state, "conv_state"), n_slots=conv_state.shape[0], state_cols=conv_state.shape[2],
        state_slot_stride=conv_state.stride(0), state_ch_stride=conv_state.stride(1),
        cache_idx=ptr(cache_idx, "cache_idx", False), has_initial_state=ptr(has_initial_state, "has_initial_state", False),
        weight=ptr(weight, "weight"), bias=ptr(bias, "bias", False), err=ptr(err, "err", False))


def conv_prefill(x, conv_state, weight, bias, out, cu_seqlens, *, max_seqlen, qk_channels, head_dim, l2_eps=1e-6,
                 cache_idx=None, has_initial_state=None, err=None, stream=None) -> None:
    """Queue one packed variable-length prefill on ``stream`` (default: torch's current stream).

    Writes out, conv_state (and err); raises CvError on an invalid argument."""
    for t in (x, conv_state, weight, out):
        if t.dtype != x.dtype:
            raise TypeError("x, conv_state, weight and out must share one dtype")
    if bias is not None and bias.dtype != x.dtype:
        raise TypeError("bias must have the dtype of x")
    a = make_prefill_args(x, conv_state, weight, bias, out, cu_seqlens, max_seqlen=max_seqlen, qk_channels=qk_channels,
                          head_dim=head_dim, l2_eps=l2_eps, cache_idx=cache_idx, has_initial_state=has_initial_state,
                          err=err)
    rc = load_library().cv_conv_prefill(ctypes.byref(a), _stream_ptr(stream))
    if rc != 0:
        raise CvError(rc, "cv_conv_prefill")
