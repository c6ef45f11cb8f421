"""Pins of the oracle's packed ragged verify (sglang PR #46184, "Related upstream work": target verify
on packed ragged tokens, with the tile store covering the packed rows).  Sequence s owns draft rows
[cu[s], cu[s+1]) of x and out; its T_s rows are verified exactly as a verify of T_s tokens would
verify them.  Every pin compares against something other than the packed path itself: the plain
verify (pinned in test_oracle_pins.py) run on each sequence alone, float64 conv1d, the shorter
verify for the commit, and sentinels for what must stay untouched."""
from __future__ import annotations

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import assert_bits_equal, bits, clone_inputs
from spec_decode_verify_gb300 import workloads as wl


def small(**over):
    base = dict(name="rag", lengths=(3, 0, 1, 5, 2), T=5, dim=96, width=4, qk_channels=64, head_dim=16,
                dtype="f32", layout="dense", bias=True, pad=(), extra_slots=2, seed=7)
    base.update(over)
    return wl.RaggedWorkload(**base)


def run_ragged(w, inp, status=True):
    r = clone_inputs(inp)
    r["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32) if status else None
    oracle.conv_verify(r["x"], r["conv_state"], r["weight"], r["bias"], r["out"], r["window"], layout=w.layout,
                       qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=r["cache_idx"],
                       state_off=r["state_off"], status=r["status"], cu_draft=r["cu_draft"], T=w.T)
    return r


def commit_ragged(w, r, accept=None):
    st = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_commit(r["conv_state"], r["window"], r["accept_len"] if accept is None else accept, layout=w.layout,
                       T=w.T, width=w.width, cache_idx=r["cache_idx"], status=st,
                       x=r["x"] if w.layout == "recompute" else None, cu_draft=r["cu_draft"],
                       total_tokens=r["x"].shape[0])
    return st


def plain_single(w, inp, s, n_tokens, layout=None):
    """The plain (non-packed) oracle on sequence s alone with its first n_tokens draft rows."""
    layout = layout or w.layout
    b = int(inp["cu_draft"][s])
    slot = int(inp["cache_idx"][s])
    x = inp["x"][b:b + n_tokens].unsqueeze(0).clone()
    state = inp["conv_state"].clone()
    out = wl.sentinel_tensor((1, n_tokens, w.dim), w.torch_dtype)
    R = w.width - 1
    win = None
    if layout == "dense":
        win = wl.sentinel_tensor((1, n_tokens, w.dim, R), w.torch_dtype)
    elif layout == "dedup":
        win = wl.sentinel_tensor((1, w.dim, n_tokens + R - 1), w.torch_dtype)
    off = inp["state_off"][s:s + 1].clone() if inp["state_off"] is not None else None
    oracle.conv_verify(x, state, inp["weight"], inp["bias"], out, win, layout=layout, qk_channels=w.qk_channels,
                       head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=torch.tensor([slot], dtype=torch.int32),
                       state_off=off)
    return out[0], win, state


@pytest.mark.parametrize("layout", ["dense", "dedup", "history", "recompute"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_v1_packed_equals_separate_verifies(layout, dtype):
    """V-1: each sequence's rows, snapshots and state equal a plain verify of its T_s tokens alone,
    bit for bit (T_s = 0: no rows, no snapshot, the state receives the committed window)."""
    w = small(layout=layout, dtype=dtype, state_offset=layout != "recompute", pad=(2,))
    inp = wl.make_ragged_inputs(w)
    r = run_ragged(w, inp)
    cu = inp["cu_draft"]
    R = w.width - 1
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        Ts = w.lengths[s]
        if slot < 0:
            continue
        assert int(r["status"][s]) == 0
        if Ts == 0:
            o = int(inp["state_off"][s]) if inp["state_off"] is not None else 0
            if layout in ("dense", "dedup"):
                want = inp["conv_state"][slot].clone()
                want[:, :R] = inp["conv_state"][slot][:, o:o + R]
                assert_bits_equal(r["conv_state"][slot], want, f"state of empty seq {s}")
                assert_bits_equal(r["window"][s], inp["window"][s], f"window of empty seq {s}")
            else:
                # history: no snapshot to write, so the row (and the window in it) stays; recompute:
                # the verify never writes the state
                assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], f"state of empty seq {s}")
            continue
        out1, win1, st1 = plain_single(w, inp, s, Ts)
        b = int(cu[s])
        assert_bits_equal(r["out"][b:b + Ts], out1, f"out rows of seq {s}")
        assert_bits_equal(r["conv_state"][slot], st1[slot], f"state of seq {s}")
        if layout == "dense":
            assert_bits_equal(r["window"][s, :Ts], win1[0], f"snapshots of seq {s}")
        elif layout == "dedup":
            assert_bits_equal(r["window"][s, :, :Ts + R - 1], win1[0], f"dedup row of seq {s}")


@pytest.mark.parametrize("layout", ["dense", "dedup", "history", "recompute"])
def test_v2_equal_lengths_equal_the_plain_verify(layout):
    """V-2: every sequence with T draft tokens, packed back to back, is the plain batched verify
    bit for bit (outputs, snapshots, state, status)."""
    T = 4
    w = small(lengths=(T,) * 5, T=T, layout=layout, pad=(1,), state_offset=layout != "recompute")
    inp = wl.make_ragged_inputs(w)
    r = run_ragged(w, inp)
    p = clone_inputs(inp)
    p["x"] = inp["x"].reshape(w.n_seq, T, w.dim).clone()
    p["out"] = wl.sentinel_tensor((w.n_seq, T, w.dim), w.torch_dtype)
    p["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_verify(p["x"], p["conv_state"], p["weight"], p["bias"], p["out"], p["window"], layout=layout,
                       qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=p["cache_idx"],
                       state_off=p["state_off"], status=p["status"])
    assert_bits_equal(r["out"], p["out"].reshape(w.n_seq * T, w.dim), "out")
    assert_bits_equal(r["conv_state"], p["conv_state"], "state")
    assert_bits_equal(r["status"], p["status"], "status")
    if r["window"] is not None:
        assert_bits_equal(r["window"], p["window"], "window")


@pytest.mark.parametrize("width", [2, 3, 4])
def test_v3_matches_float64_conv1d(width):
    """V-3: each sequence's outputs equal torch float64 conv1d over [committed window, its packed
    rows] with SiLU and the q|k L2 groups, within the fp32 output tolerance."""
    w = small(width=width, lengths=(4, 1, 0, 6, 3), T=6, state_offset=True)
    inp = wl.make_ragged_inputs(w)
    r = run_ragged(w, inp)
    R = width - 1
    for s in range(w.n_seq):
        Ts = w.lengths[s]
        if Ts == 0:
            continue
        slot, o, b = int(inp["cache_idx"][s]), int(inp["state_off"][s]), int(inp["cu_draft"][s])
        full = torch.cat([inp["conv_state"][slot, :, o:o + R].double(), inp["x"][b:b + Ts].double().t()], dim=1)
        acc = F.conv1d(full[None], inp["weight"].double()[:, None, :], inp["bias"].double(), groups=w.dim)[0]
        y = (acc / (1 + torch.exp(-acc))).t()  # [Ts, dim]
        q = w.qk_channels
        g = y[:, :q].reshape(Ts, q // w.head_dim, w.head_dim)
        y[:, :q] = (g / torch.sqrt((g * g).sum(-1, keepdim=True) + w.l2_eps)).reshape(Ts, q)
        got = r["out"][b:b + Ts].double()
        assert ((got - y).abs() <= 1e-5 * y.abs() + 1e-6).all(), float((got - y).abs().max())


@pytest.mark.parametrize("layout", ["dense", "dedup", "recompute"])
def test_v4_commit_equals_shorter_verify(layout):
    """V-4: verify(T_s) then commit(a) leaves the state of a verify of the first a rows, for every
    a in 1..T_s; a sequence with T_s = 0 commits nothing (status 0, state unchanged)."""
    w = small(layout=layout, lengths=(3, 0, 4, 1), T=4)
    inp = wl.make_ragged_inputs(w)
    for trial in range(4):
        acc = torch.tensor([min(trial + 1, max(L, 1)) for L in w.lengths], dtype=torch.int32)
        r = run_ragged(w, inp)
        after_verify = r["conv_state"].clone()
        st = commit_ragged(w, r, acc)
        assert (st == 0).all(), st
        for s in range(w.n_seq):
            slot = int(inp["cache_idx"][s])
            if w.lengths[s] == 0:
                assert_bits_equal(r["conv_state"][slot], after_verify[slot], f"empty seq {s} after commit")
                continue
            a = int(acc[s])
            _, _, st1 = plain_single(w, inp, s, a, layout="dense")
            assert_bits_equal(r["conv_state"][slot], st1[slot], f"seq {s} committed at {a}")


def test_v5_untouched_regions():
    """V-5: padded sequences, snapshot steps at and past T_s, dedup columns at and past T_s+W-2, x
    and out rows past the last span and unused slots all keep their sentinels."""
    for layout in ("dense", "dedup"):
        w = small(layout=layout, lengths=(2, 0, 5, 1, 3), pad=(3,), extra_rows=3)
        inp = wl.make_ragged_inputs(w)
        r = run_ragged(w, inp)
        R = w.width - 1
        total = sum(w.lengths)
        assert_bits_equal(r["out"][total:], inp["out"][total:], "rows past the last span")
        b3 = int(inp["cu_draft"][3])
        assert_bits_equal(r["out"][b3:b3 + 1], inp["out"][b3:b3 + 1], "padded sequence's row")
        for s, Ts in enumerate(w.lengths):
            if s in w.pad:
                assert_bits_equal(r["window"][s], inp["window"][s], f"padded window {s}")
                continue
            if layout == "dense":
                assert_bits_equal(r["window"][s, Ts:], inp["window"][s, Ts:], f"steps past T_s of {s}")
            else:
                first = Ts + R - 1 if Ts > 0 else 0
                assert_bits_equal(r["window"][s, :, first:], inp["window"][s, :, first:], f"columns past of {s}")
        used = set(int(c) for c in inp["cache_idx"] if c >= 0)
        for slot in range(w.n_slots):
            if slot not in used:
                assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], f"unused slot {slot}")


def test_v6_bad_spans_flagged_and_untouched():
    """V-6: a reversed span, one past total_tokens and one longer than T flag their sequence (16)
    and leave it untouched; the commit flags the same spans, and an accept count past T_s (4)."""
    w = small(lengths=(2, 2, 2, 2, 2), T=3, layout="dedup")
    inp = wl.make_ragged_inputs(w)
    cu = inp["cu_draft"]
    cu[2] = 1  # seq 1: [4 -> 1) reversed ... (and seq 2: [1, 6) longer than T = 3)
    inp["cu_draft"] = cu
    r = run_ragged(w, inp)
    st = r["status"].numpy()
    assert st[1] == 16 and st[2] == 16 and st[0] == 0 and st[3] == 0 and st[4] == 0, st
    for s in (1, 2):
        slot = int(inp["cache_idx"][s])
        assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], f"state of flagged {s}")
        assert_bits_equal(r["window"][s], inp["window"][s], f"window of flagged {s}")
    # one past the end
    w2 = small(lengths=(2, 2), T=3, layout="dense")
    inp2 = wl.make_ragged_inputs(w2)
    inp2["cu_draft"][2] = 5  # total_tokens is 4
    r2 = run_ragged(w2, inp2)
    assert r2["status"].tolist() == [0, 16]
    # the commit: the same spans flagged, and an accept count past T_s
    acc = torch.tensor([3, 1, 1, 1, 1], dtype=torch.int32)  # seq 0 has T_s = 2 < 3
    stc = commit_ragged(w, r, acc)
    assert stc.tolist() == [4, 16, 16, 0, 0]
