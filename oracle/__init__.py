"""CPU oracle for the batched speculative-verify causal depthwise conv1d update.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the bench's CPU-baseline
leg may import this module.  It loads ``oracle.c`` (built with gcc, -ffp-contract=off) through
ctypes and marshals CPU torch tensors into plain pointers and element strides.  It shares no code
with the CUDA library.

The arithmetic and the passages it follows are stated in the header comment of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p


class _VerifyArgs(ctypes.Structure):
    _fields_ = [
        ("n_seq", c_i32), ("T", c_i32), ("dim", c_i32), ("width", c_i32), ("qk_channels", c_i32),
        ("head_dim", c_i32), ("is_bf16", c_i32), ("l2_eps", ctypes.c_float),
        ("x", c_vp), ("x_seq", c_i64), ("x_tok", c_i64),
        ("out", c_vp), ("out_seq", c_i64), ("out_tok", c_i64),
        ("state", c_vp), ("n_slots", c_i32), ("state_cols", c_i32), ("st_slot", c_i64), ("st_ch", c_i64),
        ("cache_idx", c_vp), ("state_off", c_vp), ("weight", c_vp), ("bias", c_vp),
        ("window", c_vp), ("dedup", c_i32), ("w_seq", c_i64), ("w_step", c_i64), ("w_ch", c_i64),
        ("w_col", c_i64), ("status", c_vp), ("history", c_i32), ("recompute", c_i32), ("state_is_bf16", c_i32),
        ("parent", c_vp), ("cu_draft", c_vp), ("total_tokens", c_i32),
    ]


class _CommitArgs(ctypes.Structure):
    _fields_ = [
        ("n_seq", c_i32), ("T", c_i32), ("dim", c_i32), ("width", c_i32), ("is_bf16", c_i32),
        ("state", c_vp), ("n_slots", c_i32), ("st_slot", c_i64), ("st_ch", c_i64), ("cache_idx", c_vp),
        ("window", c_vp), ("dedup", c_i32), ("w_seq", c_i64), ("w_step", c_i64), ("w_ch", c_i64),
        ("w_col", c_i64), ("accept_len", c_vp), ("status", c_vp), ("recompute", c_i32), ("x", c_vp),
        ("x_seq", c_i64), ("x_tok", c_i64), ("cu_draft", c_vp), ("total_tokens", c_i32),
    ]


class _PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("n_seq", c_i32), ("dim", c_i32), ("width", c_i32), ("qk_channels", c_i32), ("head_dim", c_i32),
        ("is_bf16", c_i32), ("l2_eps", ctypes.c_float), ("total_tokens", c_i32),
        ("x", c_vp), ("x_tok", c_i64), ("out", c_vp), ("out_tok", c_i64), ("cu_seqlens", c_vp),
        ("state", c_vp), ("n_slots", c_i32), ("state_cols", c_i32), ("st_slot", c_i64), ("st_ch", c_i64),
        ("cache_idx", c_vp), ("has_initial_state", c_vp), ("weight", c_vp), ("bias", c_vp), ("status", c_vp),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (plain C, no vector intrinsics, no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-shared",
                        "-fPIC", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _open(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_conv_verify.argtypes = [ctypes.POINTER(_VerifyArgs)]
    lib.oracle_conv_verify.restype = c_i32
    lib.oracle_conv_commit.argtypes = [ctypes.POINTER(_CommitArgs)]
    lib.oracle_conv_commit.restype = c_i32
    lib.oracle_conv_prefill.argtypes = [ctypes.POINTER(_PrefillArgs)]
    lib.oracle_conv_prefill.restype = c_i32
    lib.oracle_round_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_round_f32_to_bf16.restype = ctypes.c_uint32
    return lib


def swap_library(path):
    """Use the oracle built at ``path`` (None: the in-tree build) and return the previous handle.

    Only the mutation tests use this, to check that the pins reject a planted mistake."""
    global _lib
    prev = _lib
    _lib = _open(path) if isinstance(path, str) else path
    return prev


def _load():
    global _lib
    if _lib is None:
        build()
        lib = _open(_SO)
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu", "the oracle takes CPU tensors"
    return t.data_ptr()


def _is_bf16(t) -> int:
    if t.dtype == torch.bfloat16:
        return 1
    if t.dtype == torch.float32:
        return 0
    raise TypeError(f"unsupported dtype {t.dtype}")


def window_strides(window: torch.Tensor, layout: str):
    """(seq, step, ch, col) element strides of a window buffer.

    dense: window is [n_seq, T, dim, W-1].  dedup: window is the [n_seq, dim, T+W-2] row buffer and
    the step stride equals the column stride.  history, recompute: there is no window buffer."""
    if layout in ("history", "recompute"):
        return 0, 0, 0, 0
    if layout == "dense":
        s = window.stride()
        return s[0], s[1], s[2], s[3]
    s = window.stride()
    return s[0], s[2], s[1], s[2]


def conv_verify(x, conv_state, weight, bias, out, window, *, layout, qk_channels, head_dim, l2_eps,
                cache_idx=None, state_off=None, status=None, parent=None, cu_draft=None, T=None):
    """Run the oracle verify in place on CPU tensors (conv_state, out, window, status are written).

    x [n_seq, T, dim] (channel stride 1), conv_state [n_slots, dim, S] (any strides: a state whose
    columns are not contiguous is run on a contiguous copy, written back afterwards), weight
    [dim, W] contiguous, bias [dim] or None, out [n_seq, T, dim] (channel stride 1),
    window dense [n_seq, T, dim, W-1] / dedup [n_seq, dim, T+W-2] / None for the history layout
    (the state row, S >= T+W-2 columns, receives the snapshot row) and the recompute layout
    (outputs only, state untouched); cache_idx, state_off, status int32 [n_seq] or None; parent
    int32 [n_seq, T] contiguous (tree verify, dense layout only) or None (a chain).

    Packed ragged drafts: cu_draft int32 [n_seq + 1]; x and out are then [total_tokens, dim]
    (sequence s owns rows cu_draft[s] .. cu_draft[s+1]-1) and T (required) is the largest draft
    count, the T of the window buffer."""
    if parent is not None:
        assert layout == "dense" and parent.is_contiguous() and parent.dtype == torch.int32
    if layout not in ("dense", "dedup", "history", "recompute"):
        raise ValueError(f"unknown layout {layout!r}")
    if (layout in ("history", "recompute")) != (window is None):
        raise ValueError("the history and recompute layouts take no window buffer; the others need one")
    if cu_draft is not None:
        assert cu_draft.dtype == torch.int32 and cu_draft.is_contiguous() and T is not None
        assert parent is None, "packed ragged drafts are chains"
        total, dim = x.shape
        n_seq = cu_draft.shape[0] - 1
        assert x.stride(1) == 1 and out.stride(1) == 1 and tuple(out.shape) == (total, dim)
        x_seq, x_tok, o_seq, o_tok = 0, x.stride(0), 0, out.stride(0)
    else:
        n_seq, T, dim = x.shape
        total = 0
        assert x.stride(2) == 1 and out.stride(2) == 1
        x_seq, x_tok, o_seq, o_tok = x.stride(0), x.stride(1), out.stride(0), out.stride(1)
    W = weight.shape[1]
    state_arg = conv_state  # (the storage order of the state rows is not part of the arithmetic)
    if conv_state.stride(2) != 1:
        conv_state = conv_state.contiguous()
    assert weight.is_contiguous()
    ws = window_strides(window, layout)
    a = _VerifyArgs(
        n_seq=n_seq, T=T, dim=dim, width=W, qk_channels=qk_channels, head_dim=head_dim, is_bf16=_is_bf16(x),
        l2_eps=l2_eps, x=_ptr(x), x_seq=x_seq, x_tok=x_tok, out=_ptr(out),
        out_seq=o_seq, out_tok=o_tok, state=_ptr(conv_state), n_slots=conv_state.shape[0],
        state_cols=conv_state.shape[2], st_slot=conv_state.stride(0), st_ch=conv_state.stride(1),
        cache_idx=_ptr(cache_idx), state_off=_ptr(state_off), weight=_ptr(weight), bias=_ptr(bias),
        window=_ptr(window), dedup=1 if layout == "dedup" else 0, w_seq=ws[0], w_step=ws[1], w_ch=ws[2],
        w_col=ws[3], status=_ptr(status), history=1 if layout == "history" else 0,
        recompute=1 if layout == "recompute" else 0, state_is_bf16=_is_bf16(conv_state), parent=_ptr(parent),
        cu_draft=_ptr(cu_draft), total_tokens=total)
    if window is not None and window.dtype != conv_state.dtype:
        raise TypeError("the window has the state's dtype")
    rc = _load().oracle_conv_verify(ctypes.byref(a))
    if rc != 0:
        raise RuntimeError(f"oracle_conv_verify returned {rc}")
    if conv_state is not state_arg:
        state_arg.copy_(conv_state)


def conv_commit(conv_state, window, accept_len, *, layout, T, width, cache_idx=None, status=None, x=None,
                cu_draft=None, total_tokens=0):
    """Run the oracle commit in place: state slot of seq s <- snapshot accept_len[s]-1.

    layout "recompute": window is None and x [n_seq, T, dim] (channel stride 1) is the verify's
    input; the snapshot is rebuilt from the state's window and x.  cu_draft int32 [n_seq + 1]: the
    verify's packed ragged spans (accept_len then lies in 1..T_s, and x is [total_tokens, dim])."""
    if (layout == "recompute") != (x is not None and window is None):
        raise ValueError("the recompute commit takes x and no window; the others take a window")
    x_seq = x_tok = 0
    if x is not None and cu_draft is not None:
        assert x.stride(1) == 1
        x_tok, total_tokens = x.stride(0), x.shape[0]
    elif x is not None:
        assert x.stride(2) == 1
        x_seq, x_tok = x.stride(0), x.stride(1)
    ws = window_strides(window, layout)
    n_seq = accept_len.shape[0]
    a = _CommitArgs(
        n_seq=n_seq, T=T, dim=conv_state.shape[1], width=width, is_bf16=_is_bf16(conv_state),
        state=_ptr(conv_state), n_slots=conv_state.shape[0], st_slot=conv_state.stride(0),
        st_ch=conv_state.stride(1), cache_idx=_ptr(cache_idx), window=_ptr(window),
        dedup=1 if layout == "dedup" else 0, w_seq=ws[0], w_step=ws[1], w_ch=ws[2], w_col=ws[3],
        accept_len=_ptr(accept_len), status=_ptr(status), recompute=1 if layout == "recompute" else 0,
        x=_ptr(x), x_seq=x_seq, x_tok=x_tok, cu_draft=_ptr(cu_draft), total_tokens=int(total_tokens))
    rc = _load().oracle_conv_commit(ctypes.byref(a))
    if rc != 0:
        raise RuntimeError(f"oracle_conv_commit returned {rc}")


def conv_prefill(x, conv_state, weight, bias, out, cu_seqlens, *, qk_channels, head_dim, l2_eps, cache_idx=None,
                 has_initial_state=None, status=None):
    """Run the oracle prefill in place on CPU tensors (conv_state, out, status are written).

    x, out [total_tokens, dim] (channel stride 1, any token stride), conv_state [n_slots, dim, S]
    (column stride 1), weight [dim, W] contiguous, bias [dim] or None, cu_seqlens int32
    [n_seq + 1], cache_idx / has_initial_state / status int32 [n_seq] or None."""
    total, dim = x.shape
    n_seq = cu_seqlens.shape[0] - 1
    assert x.stride(1) == 1 and out.stride(1) == 1 and conv_state.stride(2) == 1 and weight.is_contiguous()
    a = _PrefillArgs(
        n_seq=n_seq, dim=dim, width=weight.shape[1], qk_channels=qk_channels, head_dim=head_dim,
        is_bf16=_is_bf16(x), l2_eps=l2_eps, total_tokens=total, x=_ptr(x), x_tok=x.stride(0), out=_ptr(out),
        out_tok=out.stride(0), cu_seqlens=_ptr(cu_seqlens), state=_ptr(conv_state), n_slots=conv_state.shape[0],
        state_cols=conv_state.shape[2], st_slot=conv_state.stride(0), st_ch=conv_state.stride(1),
        cache_idx=_ptr(cache_idx), has_initial_state=_ptr(has_initial_state), weight=_ptr(weight),
        bias=_ptr(bias), status=_ptr(status))
    rc = _load().oracle_conv_prefill(ctypes.byref(a))
    if rc != 0:
        raise RuntimeError(f"oracle_conv_prefill returned {rc}")


def round_f32_to_bf16_bits(v: float) -> int:
    return int(_load().oracle_round_f32_to_bf16(v))
