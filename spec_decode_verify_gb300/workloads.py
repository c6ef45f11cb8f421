"""Seeded synthetic inputs for the batched speculative-verify conv1d update.

This module only draws random inputs and allocates output buffers filled with a sentinel bit
pattern.  It holds none of the method's arithmetic, so both the CUDA library's tests and the CPU
oracle's tests can take their inputs from it.

The five named workloads follow the shapes the pages describe:
  * the sglang PR #46184 benchmark ("Benchmarking and Profiling": GB300, dim 10240, conv width 4,
    bf16, T 8, batch 128) with the deduplicated window layout of MambaPool ("Motivation");
  * the Atlas batched verify (fn gdn_verify_fused_conv_kn_batched: K draft positions, strided
    input/output rows, dense intermediates) with the q|k|v conv weights bound as
    concat([q, k, v]) (glm5next_kda mod.rs: the checkpoint stores the q, k and v conv weights
    as separate tensors);
  * a width-3 conv without L2 groups and with a per-sequence accepted-token state offset (PR
    #46184's tests cover an offset of the accepted-token count into the state; its "Scope" names
    width-3 deduplicated windows);
  * the benchmark shape with an fp32 state and fp32 snapshots under bf16 inputs (PR #46184's
    extra check covers mixed input and state dtypes);
  * the benchmark shape with the draft tokens forming a random tree (PR #46184 "Scope": tree
    verify keeps dense windows);
  * the benchmark shape again with the recompute rollback (memra-engine ssm_conv_ring_rebuild_dc:
    no snapshots; the commit rebuilds the state from the kept window and the accepted inputs) and
    with the history-row state: the state row of each slot is the deduplicated [dim, T+W-2] row
    itself and the committed window is read at accept_len - 1.
Values: x, state ~ N(0, 1), weights ~ U(-0.5, 0.5), bias ~ N(0, 0.1); bf16 values are drawn in
fp32 and converted by torch (round to nearest even).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# Sentinel bit patterns for buffers that must stay untouched (bf16: a finite negative number;
# fp32: a finite negative number), so an untouched region compares bitwise.
SENTINEL_BF16 = 0xDEAD
SENTINEL_F32 = 0xDEADBEEF


@dataclasses.dataclass(frozen=True)
class VerifyWorkload:
    name: str
    n_seq: int
    T: int
    dim: int
    width: int
    qk_channels: int
    head_dim: int
    dtype: str  # "f32" or "bf16"
    # "dense", "dedup", "history" (the state row is the dedup row; no window buffer) or "recompute"
    # (no snapshots; the commit rebuilds the state from the pre-verify window and x)
    layout: str
    bias: bool = False
    l2_eps: float = 1e-6
    n_pad: int = 0  # sequences whose cache index is -1
    extra_slots: int = 0  # pool slots no sequence uses (must stay untouched)
    x_row_stride: Optional[int] = None  # token stride of x when it is a slice of a wider buffer
    qkv_split: Optional[tuple] = None  # (q, k, v) channel counts of separately drawn conv weights
    state_offset: bool = False  # per-sequence offset = accept_len - 1 into a wider state row
    state_dtype: Optional[str] = None  # dtype of state and window when it differs from x ("f32"/"bf16")
    tree: bool = False  # draft tokens form a tree: a random earlier parent (or -1) per token
    # dedup rows stored column by column ([n_seq, T+W-2, dim] seen as [n_seq, dim, T+W-2]: MambaPool's
    # axis-0 window layout seen transposed, sglang PR #46184 "Modifications", test coverage)
    window_transposed: bool = False
    # state rows stored column by column ([n_slots, state_cols, dim] seen as [n_slots, dim, state_cols]);
    # the history layout only: the commit-free step then reads W-1 and writes T+W-2 channel runs
    state_transposed: bool = False
    seed: int = 0

    @property
    def n_slots(self) -> int:
        return self.n_seq + self.extra_slots

    @property
    def state_cols(self) -> int:
        if self.layout == "history":
            return self.T + self.width - 2
        return self.width - 1 + (self.T - 1 if self.state_offset else 0)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def state_torch_dtype(self):
        sd = self.state_dtype or self.dtype
        return torch.float32 if sd == "f32" else torch.bfloat16

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def state_esize(self) -> int:
        return 4 if (self.state_dtype or self.dtype) == "f32" else 2

    def replace(self, **kw) -> "VerifyWorkload":
        return dataclasses.replace(self, **kw)


# The five workloads.  The first finishes in the oracle in milliseconds; the third is the
# benchmark configuration of the PR's table.
WORKLOADS = {
    w.name: w
    for w in [
        VerifyWorkload("n1_t2_dim512_w4_f32_dense", n_seq=1, T=2, dim=512, width=4, qk_channels=256,
                       head_dim=64, dtype="f32", layout="dense", seed=0),
        VerifyWorkload("n4_t4_dim4096_w4_bf16_dedup_bias", n_seq=4, T=4, dim=4096, width=4,
                       qk_channels=2048, head_dim=128, dtype="bf16", layout="dedup", bias=True, seed=1),
        VerifyWorkload("n128_t8_dim10240_w4_bf16_dedup_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup", n_pad=13,
                       extra_slots=16, seed=2),
        VerifyWorkload("n8_t17_dim8192_w4_bf16_dense_qkvsplit_xstride12288", n_seq=8, T=17, dim=8192,
                       width=4, qk_channels=4096, head_dim=128, dtype="bf16", layout="dense",
                       x_row_stride=12288, qkv_split=(2048, 2048, 4096), seed=3),
        VerifyWorkload("n64_t8_dim6144_w3_bf16_dense_nol2_stateoff", n_seq=64, T=8, dim=6144, width=3,
                       qk_channels=0, head_dim=128, dtype="bf16", layout="dense", state_offset=True,
                       seed=4),
        VerifyWorkload("n128_t8_dim10240_w4_bf16_recompute_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="recompute", n_pad=13,
                       extra_slots=16, seed=6),
        VerifyWorkload("n128_t8_dim10240_w4_bf16x_f32state_dedup_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", state_dtype="f32", layout="dedup", n_pad=13,
                       extra_slots=16, seed=7),
        VerifyWorkload("n128_t8_dim10240_w4_bf16_tree_dense_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="dense", n_pad=13, extra_slots=16,
                       tree=True, seed=8),
        VerifyWorkload("n128_t8_dim10240_w4_bf16_history_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="history", n_pad=13,
                       extra_slots=16, state_offset=True, seed=5),
        # the rows of the pages' kernel-time table (bs 128, T 8 and T 16, dim 10240, width 4, bf16,
        # deduplicated rows), with no padded rows, as that table has none
        VerifyWorkload("n128_t8_dim10240_w4_bf16_dedup_nopad", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup", seed=10),
        VerifyWorkload("n128_t16_dim10240_w4_bf16_dedup_nopad", n_seq=128, T=16, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup", seed=11),
        VerifyWorkload("n128_t8_dim10240_w4_bf16_dedupT_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup", n_pad=13,
                       extra_slots=16, window_transposed=True, seed=9),
        # the commit-free step with the state rows stored column by column
        VerifyWorkload("n128_t8_dim10240_w4_bf16_historyT_pad13", n_seq=128, T=8, dim=10240, width=4,
                       qk_channels=4096, head_dim=128, dtype="bf16", layout="history", n_pad=13,
                       extra_slots=16, state_offset=True, state_transposed=True, seed=12),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)
BENCH_WORKLOAD = "n128_t8_dim10240_w4_bf16_dedup_pad13"


def _to_dtype(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype)


def sentinel_tensor(shape, dtype) -> torch.Tensor:
    """A CPU tensor whose every element holds the sentinel bit pattern."""
    if dtype == torch.bfloat16:
        return torch.full(shape, SENTINEL_BF16 - 65536, dtype=torch.int16).view(torch.bfloat16)
    return torch.full(shape, SENTINEL_F32 - 2**32, dtype=torch.int32).view(torch.float32)


def window_shape(w: VerifyWorkload):
    if w.layout in ("history", "recompute"):
        return None
    if w.layout == "dense":
        return (w.n_seq, w.T, w.dim, w.width - 1)
    return (w.n_seq, w.dim, w.T + w.width - 2)


def make_inputs(w: VerifyWorkload, seed: Optional[int] = None) -> dict:
    """CPU tensors for one verify + commit of workload ``w``.

    Returns x [n_seq, T, dim] (a view with token stride ``x_row_stride`` when set), conv_state
    [n_slots, dim, state_cols] (column-major when ``state_transposed``), weight [dim, W], bias [dim] or None, cache_idx int32 [n_seq]
    (-1 = padded), state_off int32 [n_seq] or None, accept_len int32 [n_seq] in 1..T, and
    sentinel-filled out [n_seq, T, dim] and window buffers (dense [n_seq, T, dim, W-1], dedup
    [n_seq, dim, T+W-2], None for the history and recompute layouts).
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    dt = w.torch_dtype
    row = w.x_row_stride or w.dim
    xw = rng.standard_normal((w.n_seq * w.T, row), dtype=np.float32)
    x_wide = _to_dtype(xw, dt)
    x = x_wide.view(w.n_seq, w.T, row)[:, :, : w.dim]
    state = _to_dtype(rng.standard_normal((w.n_slots, w.dim, w.state_cols), dtype=np.float32), w.state_torch_dtype)
    if w.state_transposed:  # the same values, stored column-major
        st = torch.empty((w.n_slots, w.state_cols, w.dim), dtype=state.dtype).transpose(1, 2)
        st.copy_(state)
        state = st
    if w.qkv_split:
        parts = [rng.uniform(-0.5, 0.5, size=(n, 1, w.width)).astype(np.float32) for n in w.qkv_split]
        weight = _to_dtype(np.concatenate(parts, axis=0), dt).squeeze(1)
        assert weight.shape == (w.dim, w.width)
    else:
        weight = _to_dtype(rng.uniform(-0.5, 0.5, size=(w.dim, w.width)).astype(np.float32), dt)
    bias = _to_dtype(rng.normal(0.0, 0.1, size=(w.dim,)).astype(np.float32), dt) if w.bias else None
    perm = rng.permutation(w.n_slots)[: w.n_seq].astype(np.int32)
    if w.n_pad:
        pad = rng.permutation(w.n_seq)[: w.n_pad]
        perm[pad] = -1
    cache_idx = torch.from_numpy(perm.copy())
    accept = torch.from_numpy(rng.integers(1, w.T + 1, size=w.n_seq).astype(np.int32))
    state_off = (accept - 1).to(torch.int32) if w.state_offset else None
    out = sentinel_tensor((w.n_seq, w.T, w.dim), dt)
    window = None if w.layout in ("history", "recompute") else sentinel_tensor(window_shape(w), w.state_torch_dtype)
    if window is not None and w.window_transposed:
        window = sentinel_tensor((w.n_seq, w.T + w.width - 2, w.dim), w.state_torch_dtype).transpose(1, 2)
    r = dict(x=x, x_base=x_wide, conv_state=state, weight=weight, bias=bias, cache_idx=cache_idx,
             state_off=state_off, accept_len=accept, out=out, window=window)
    if w.tree:
        par = np.full((w.n_seq, w.T), -1, dtype=np.int32)
        for t in range(1, w.T):
            par[:, t] = rng.integers(-1, t, size=w.n_seq)
        r["parent"] = torch.from_numpy(par)
    return r


def random_case(rng: np.random.Generator, **over) -> VerifyWorkload:
    """A small random workload for sweeps (shapes drawn from the ranges the pages test)."""
    W = int(over.pop("width", rng.integers(2, 5)))
    T = int(over.pop("T", rng.choice([1, 2, 3, 4, 8, 9, 16, 17])))
    hd = int(over.pop("head_dim", rng.choice([8, 16, 32, 64, 128])))
    groups = int(rng.integers(0, 5))
    qk = over.pop("qk_channels", groups * hd)
    dim = int(over.pop("dim", qk + int(rng.integers(1, 300))))
    return VerifyWorkload(
        name=over.pop("name", "random"), n_seq=int(over.pop("n_seq", rng.integers(1, 6))), T=T, dim=dim,
        width=W, qk_channels=int(qk), head_dim=hd, dtype=over.pop("dtype", str(rng.choice(["f32", "bf16"]))),
        layout=over.pop("layout", str(rng.choice(["dense", "dedup"]))), bias=bool(over.pop("bias", rng.integers(0, 2))),
        seed=int(over.pop("seed", rng.integers(0, 2**31))), **over)


def algorithmic_bytes(w: VerifyWorkload, n_active: Optional[int] = None) -> dict:
    """Bytes the verify and the commit must move (each element once), per the data movement of
    the method: x read, committed window read, outputs written, snapshots written, state written;
    weights and bias read once; the int32 index arrays once."""
    e, se = w.esize, w.state_esize  # x/out/taps element size; state/window element size
    n = (w.n_seq - w.n_pad) if n_active is None else n_active
    shared = (w.dim * w.width + (w.dim if w.bias else 0)) * e + 4 * w.n_seq * (1 + (1 if w.state_offset else 0))
    R = w.width - 1
    if w.layout == "history":
        # committed window read; the snapshot row written into the state row; nothing to commit
        per_seq = 2 * w.T * w.dim * e + (R + w.T + w.width - 2) * w.dim * se
        return dict(verify=n * per_seq + shared, commit=0, per_seq=per_seq)
    if w.layout == "recompute":
        # verify: x and committed window read, outputs written; commit: the window and the accepted
        # x rows (at most W-1 of them, counted as W-1) read, the window written
        per_seq = 2 * w.T * w.dim * e + R * w.dim * se
        commit = n * (2 * R * w.dim * se + R * w.dim * e) + 8 * w.n_seq
        return dict(verify=n * per_seq + shared, commit=commit, per_seq=per_seq)
    win_cols = (w.T + w.width - 2) if w.layout == "dedup" else w.T * R
    per_seq = 2 * w.T * w.dim * e + (R + win_cols + R) * w.dim * se
    commit = n * 2 * R * w.dim * se + 8 * w.n_seq
    return dict(verify=n * per_seq + shared, commit=commit, per_seq=per_seq)


# ----------------------------------------------------------------------------- packed ragged verify

@dataclasses.dataclass(frozen=True)
class RaggedWorkload:
    """Packed ragged verify: sequence s owns draft rows [cu[s], cu[s+1]) of x and out (T_s =
    lengths[s] rows, 0..T), T is the largest draft count (the window buffer's T).  sglang PR
    #46184, "Related upstream work": target verify on packed ragged tokens, the tile store covering
    the packed rows."""
    name: str
    lengths: tuple  # draft tokens per sequence (0..T)
    T: int
    dim: int
    width: int
    qk_channels: int
    head_dim: int
    dtype: str
    layout: str  # "dense", "dedup", "history" or "recompute"
    bias: bool = False
    l2_eps: float = 1e-6
    pad: tuple = ()  # indices of padded sequences (cache index -1)
    extra_slots: int = 0
    state_offset: bool = False  # read the committed window at a per-sequence offset in 0..T-1
    x_row_stride: Optional[int] = None
    extra_rows: int = 0  # rows of x / out past the last span (never touched)
    window_transposed: bool = False  # dedup rows stored column by column ([n_seq, T+W-2, dim])
    seed: int = 0

    @property
    def n_seq(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths)) + self.extra_rows

    @property
    def n_slots(self) -> int:
        return self.n_seq + self.extra_slots

    @property
    def n_pad(self) -> int:
        return len(self.pad)

    @property
    def state_cols(self) -> int:
        if self.layout == "history":
            return self.T + self.width - 2
        return self.width - 1 + (self.T - 1 if self.state_offset else 0)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    state_torch_dtype = torch_dtype

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    state_esize = esize

    def replace(self, **kw) -> "RaggedWorkload":
        return dataclasses.replace(self, **kw)


def ragged_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    """n draft counts drawn uniformly from lo..hi (seeded)."""
    rng = np.random.default_rng(seed)
    return tuple(int(v) for v in rng.integers(lo, hi + 1, size=n))


def make_ragged_inputs(w: RaggedWorkload, seed: Optional[int] = None) -> dict:
    """CPU tensors for one packed ragged verify + commit: x [total_tokens, dim] (a view with token
    stride x_row_stride when set), cu_draft int32 [n_seq+1], conv_state [n_slots, dim, state_cols],
    weight, bias, cache_idx (-1 = padded), state_off (or None), accept_len in 1..T_s (1 where
    T_s = 0), and sentinel-filled out [total_tokens, dim] and window (dense [n_seq, T, dim, W-1],
    dedup [n_seq, dim, T+W-2], None for history and recompute)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    dt = w.torch_dtype
    total = w.total_tokens
    row = w.x_row_stride or w.dim
    x_wide = _to_dtype(rng.standard_normal((max(total, 1), row), dtype=np.float32), dt)
    x = x_wide[:total, : w.dim]
    state = _to_dtype(rng.standard_normal((w.n_slots, w.dim, w.state_cols), dtype=np.float32), dt)
    weight = _to_dtype(rng.uniform(-0.5, 0.5, size=(w.dim, w.width)).astype(np.float32), dt)
    bias = _to_dtype(rng.normal(0.0, 0.1, size=(w.dim,)).astype(np.float32), dt) if w.bias else None
    perm = rng.permutation(w.n_slots)[: w.n_seq].astype(np.int32)
    for i in w.pad:
        perm[i] = -1
    cu = np.zeros(w.n_seq + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(w.lengths, dtype=np.int64))
    accept = np.array([int(rng.integers(1, max(L, 1) + 1)) for L in w.lengths], dtype=np.int32)
    state_off = None
    if w.state_offset or w.layout == "history":
        state_off = torch.from_numpy(rng.integers(0, w.T, size=w.n_seq).astype(np.int32))
    out = sentinel_tensor((total, w.dim), dt)
    window = None
    if w.layout == "dense":
        window = sentinel_tensor((w.n_seq, w.T, w.dim, w.width - 1), dt)
    elif w.layout == "dedup" and w.window_transposed:
        window = sentinel_tensor((w.n_seq, w.T + w.width - 2, w.dim), dt).transpose(1, 2)
    elif w.layout == "dedup":
        window = sentinel_tensor((w.n_seq, w.dim, w.T + w.width - 2), dt)
    return dict(x=x, x_base=x_wide, cu_draft=torch.from_numpy(cu), conv_state=state, weight=weight, bias=bias,
                cache_idx=torch.from_numpy(perm.copy()), state_off=state_off, accept_len=torch.from_numpy(accept),
                out=out, window=window)


def ragged_algorithmic_bytes(w: RaggedWorkload) -> dict:
    """Bytes a packed ragged verify and its commit must move: per active sequence with T_s draft
    tokens, x T_s rows read and out T_s rows written, the committed window read and written, and the
    snapshots written (dedup: T_s+W-2 columns when T_s >= 1; dense: T_s (W-1)-runs); weights, bias
    and the index arrays once.  Commit: the window of snapshot a-1 read and the state written, for
    sequences with T_s >= 1."""
    e = w.esize
    R = w.width - 1
    act = [i for i in range(w.n_seq) if i not in w.pad]
    shared = (w.dim * w.width + (w.dim if w.bias else 0)) * e + 4 * (2 * w.n_seq + 1)
    verify = commit = 0
    for i in act:
        L = w.lengths[i]
        snaps = (L + w.width - 2 if L > 0 else 0) if w.layout == "dedup" else L * R
        verify += (2 * L + 2 * R + snaps) * w.dim * e
        if L > 0:
            commit += 2 * R * w.dim * e
    return dict(verify=verify + shared, commit=commit + 8 * w.n_seq)


RAGGED_WORKLOADS = {
    w.name: w
    for w in [
        # the benchmark shape with ragged drafts: 128 sequences of 1..16 draft tokens (about 1100
        # packed rows), 13 padded, dedup rows sized for T = 16
        RaggedWorkload("ragged_n128_t1to16_dim10240_w4_bf16_dedup_pad13", lengths=ragged_lengths(31, 128, 1, 16),
                       T=16, dim=10240, width=4, qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup",
                       pad=tuple(int(i) for i in np.random.default_rng(32).permutation(128)[:13]), extra_slots=16,
                       seed=31),
        # the same drafts with the rows stored column by column (MambaPool's axis-0 layout): every
        # chunk's columns are whole contiguous runs
        RaggedWorkload("ragged_n128_t1to16_dim10240_w4_bf16_dedupT_pad13", lengths=ragged_lengths(31, 128, 1, 16),
                       T=16, dim=10240, width=4, qk_channels=4096, head_dim=128, dtype="bf16", layout="dedup",
                       pad=tuple(int(i) for i in np.random.default_rng(32).permutation(128)[:13]), extra_slots=16,
                       window_transposed=True, seed=31),
    ]
}
RAGGED_ORDER = list(RAGGED_WORKLOADS)


# ----------------------------------------------------------------------------- prefill

@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    """Packed variable-length prefill: sequence s owns tokens [cu[s], cu[s+1]) of x and out."""
    name: str
    lengths: tuple  # tokens per sequence (0 allowed)
    dim: int
    width: int
    qk_channels: int
    head_dim: int
    dtype: str
    bias: bool = False
    l2_eps: float = 1e-6
    pad: tuple = ()  # indices of padded sequences (cache index -1)
    no_init: tuple = ()  # indices of sequences without an initial state (zero window)
    extra_slots: int = 0
    x_row_stride: Optional[int] = None
    seed: int = 0

    @property
    def n_seq(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lengths)) if self.lengths else 0

    @property
    def n_slots(self) -> int:
        return self.n_seq + self.extra_slots

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)


def _mixed_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(v) for v in rng.integers(lo, hi + 1, size=n))


PREFILL_WORKLOADS = {
    w.name: w
    for w in [
        # small: ragged lengths (an empty one, a single token, lengths around the chunk size),
        # a padded sequence and one without an initial state
        PrefillWorkload("prefill_n6_mixed_dim4096_w4_bf16", lengths=(37, 1, 0, 256, 300, 129), dim=4096, width=4,
                        qk_channels=2048, head_dim=128, dtype="bf16", bias=True, pad=(4,), no_init=(1, 3),
                        extra_slots=2, seed=20),
        # the benchmark shape of the verify (dim 10240, q|k 4096, head_dim 128, width 4, bf16) over
        # 8 prompts of 1024..7168 tokens (about 32k tokens), every other one without a cached state
        PrefillWorkload("prefill_n8_len1k_7k_dim10240_w4_bf16", lengths=_mixed_lengths(21, 8, 1024, 7168),
                        dim=10240, width=4, qk_channels=4096, head_dim=128, dtype="bf16", no_init=(1, 3, 5, 7),
                        extra_slots=8, seed=21),
    ]
}
PREFILL_ORDER = list(PREFILL_WORKLOADS)
PREFILL_BENCH = "prefill_n8_len1k_7k_dim10240_w4_bf16"


def make_prefill_inputs(w: PrefillWorkload, seed: Optional[int] = None) -> dict:
    """CPU tensors for one prefill: x [total, dim] (a view with token stride x_row_stride when
    set), conv_state [n_slots, dim, W-1], weight [dim, W], bias [dim] or None, cu_seqlens int32
    [n_seq+1], cache_idx int32 [n_seq] (-1 = padded), has_initial_state int32 [n_seq], and a
    sentinel-filled out [total, dim]."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    dt = w.torch_dtype
    total = w.total_tokens
    row = w.x_row_stride or w.dim
    x_wide = _to_dtype(rng.standard_normal((max(total, 1), row), dtype=np.float32), dt)
    x = x_wide[:total, : w.dim]
    state = _to_dtype(rng.standard_normal((w.n_slots, w.dim, w.width - 1), dtype=np.float32), dt)
    weight = _to_dtype(rng.uniform(-0.5, 0.5, size=(w.dim, w.width)).astype(np.float32), dt)
    bias = _to_dtype(rng.normal(0.0, 0.1, size=(w.dim,)).astype(np.float32), dt) if w.bias else None
    perm = rng.permutation(w.n_slots)[: w.n_seq].astype(np.int32)
    for i in w.pad:
        perm[i] = -1
    cu = np.zeros(w.n_seq + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(w.lengths, dtype=np.int64))
    init = np.ones(w.n_seq, dtype=np.int32)
    for i in w.no_init:
        init[i] = 0
    out = sentinel_tensor((total, w.dim), dt)
    return dict(x=x, x_base=x_wide, conv_state=state, weight=weight, bias=bias, cu_seqlens=torch.from_numpy(cu),
                cache_idx=torch.from_numpy(perm.copy()), has_initial_state=torch.from_numpy(init), out=out)


def prefill_algorithmic_bytes(w: PrefillWorkload) -> int:
    """Bytes a prefill must move: x read and out written for every token of an active sequence,
    the initial window read (sequences with one) and the final window written per active sequence,
    weights and bias once, the index arrays once."""
    e = w.esize
    act = [i for i in range(w.n_seq) if i not in w.pad]
    tokens = sum(w.lengths[i] for i in act)
    windows = sum((2 if i not in w.no_init else 1) for i in act) * (w.width - 1) * w.dim
    shared = (w.dim * w.width + (w.dim if w.bias else 0)) * e + 4 * (3 * w.n_seq + 1)
    return (2 * tokens * w.dim + windows) * e + shared
