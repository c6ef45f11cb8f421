"""Pins of the CPU oracle against facts fixed by the pages and by mathematics (no GPU).

Each test names the passage it pins.  None of them re-types the oracle's formula: they use a
library special case (torch float64 conv1d), closed forms, the pages' invariants (sequential ==
batched-in-T, batched over sequences == separate runs, deduplicated view == dense view, padded rows
untouched, commit == shorter verify) and the pages' printed row layout (tests/golden).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import (assert_bits_equal, assert_out_close, bf16_ordinal, bits, clone_inputs, run_oracle_commit,
                     run_oracle_verify)
from spec_decode_verify_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(**kw) -> wl.VerifyWorkload:
    base = dict(name="small", n_seq=3, T=5, dim=96, width=4, qk_channels=64, head_dim=16, dtype="f32",
                layout="dense", bias=True, seed=11)
    base.update(kw)
    return wl.VerifyWorkload(**base)


def float64_reference(w: wl.VerifyWorkload, inp: dict):
    """Library special case: the causal depthwise conv is torch conv1d with groups=dim, 'valid'
    padding, over [committed window, x]; SiLU and the per-group L2 in float64."""
    outs, states, wins = {}, {}, {}
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        o = int(inp["state_off"][s]) if inp["state_off"] is not None else 0
        win = inp["conv_state"][slot, :, o:o + w.width - 1].double()
        xs = inp["x"][s].double().t()
        full = torch.cat([win, xs], dim=1)
        acc = F.conv1d(full[None], inp["weight"].double()[:, None, :],
                       inp["bias"].double() if inp["bias"] is not None else None, groups=w.dim)[0]
        assert acc.shape == (w.dim, w.T)
        y = acc / (1.0 + torch.exp(-acc))
        for g in range(0, w.qk_channels, w.head_dim):
            blk = y[g:g + w.head_dim]
            y[g:g + w.head_dim] = blk / torch.sqrt((blk * blk).sum(0, keepdim=True) + w.l2_eps)
        outs[s] = y.t()
        states[s] = full[:, w.T:w.T + w.width - 1]
        wins[s] = full
    return outs, states, wins


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["dense", "dedup"])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_p1_matches_float64_conv1d(dtype, layout, width):
    """P-1: conv part == torch conv1d(groups=dim) in float64, then SiLU and L2 in float64."""
    w = small(dtype=dtype, layout=layout, width=width, l2_eps=0.25, n_pad=1, extra_slots=2, seed=100 + width)
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    outs, states, _ = float64_reference(w, inp)
    for s, ref in outs.items():
        got = r["out"][s]
        if dtype == "f32":
            err = (got.double() - ref).abs()
            assert (err <= 1e-5 * ref.abs() + 1e-6).all(), float(err.max())
        else:
            d = np.abs(bf16_ordinal(bits(got)) - bf16_ordinal(bits(ref.to(torch.bfloat16))))
            assert d.max() <= 1, int(d.max())
        slot = int(inp["cache_idx"][s])
        assert torch.equal(r["conv_state"][slot, :, :width - 1].double(), states[s])


def test_p2_impulse_response():
    """P-2 (closed form): zero state, x = unit impulse at t = 0, no bias: acc[t] = w[c][W-1-t] for
    t < W and 0 afterwards (the newest input meets the last tap)."""
    w = small(T=7, width=4, qk_channels=0, bias=False)
    inp = wl.make_inputs(w)
    inp["conv_state"].zero_()
    inp["x"].zero_()
    inp["x"][:, 0, :] = 1.0
    r = run_oracle_verify(w, inp)
    for s in range(w.n_seq):
        for t in range(w.T):
            acc = inp["weight"][:, w.width - 1 - t].double() if t < w.width else torch.zeros(w.dim, dtype=torch.float64)
            ref = acc / (1 + torch.exp(-acc))
            assert torch.allclose(r["out"][s, t].double(), ref, rtol=1e-6, atol=1e-7)


def test_p3_one_hot_taps_and_constant_group():
    """P-3 (closed forms): one-hot weights w = e_j give acc[t] = full[t+j] exactly; a group whose
    channels all carry the same value v normalises to v / sqrt(hd v^2 + eps)."""
    w = small(T=4, width=4, qk_channels=0, bias=False, dtype="f32")
    for j in range(4):
        inp = wl.make_inputs(w)
        inp["weight"].zero_()
        inp["weight"][:, j] = 1.0
        r = run_oracle_verify(w, inp)
        for s in range(w.n_seq):
            slot = int(inp["cache_idx"][s])
            full = torch.cat([inp["conv_state"][slot, :, :3], inp["x"][s].t()], dim=1).double()
            for t in range(w.T):
                a = full[:, t + j]
                assert torch.allclose(r["out"][s, t].double(), a / (1 + torch.exp(-a)), rtol=1e-6, atol=1e-7)
    # constant group, eps large enough to tell sqrt(ss + eps) from max(norm, eps)
    hd, eps = 16, 0.75
    w = small(T=2, width=2, qk_channels=32, head_dim=hd, dim=48, bias=False, l2_eps=eps, n_seq=1)
    inp = wl.make_inputs(w)
    inp["weight"].zero_()
    inp["weight"][:, 1] = 1.0
    inp["x"][0, 0, :] = 0.5
    inp["x"][0, 1, :] = -2.0
    r = run_oracle_verify(w, inp)
    for t, v in enumerate([0.5, -2.0]):
        y = v / (1 + math.exp(-v))
        want = y / math.sqrt(hd * y * y + eps)
        assert torch.allclose(r["out"][0, t, :32].double(), torch.full((32,), want, dtype=torch.float64), rtol=1e-6)
        assert torch.allclose(r["out"][0, t, 32:].double(), torch.full((16,), y, dtype=torch.float64), rtol=1e-6)


@pytest.mark.parametrize("layout", ["dense", "dedup"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_p4_sequential_equals_batched_in_T(layout, dtype):
    """P-4: T single-token updates equal one T-token verify: outputs and state bit-exact, and
    snapshot t equals the state after token t (Atlas: K positions in one launch replace K
    per-token updates + K copies; the K=2 twin is bit-identical; mod.rs decode_k: snapshot t is
    the state after row t)."""
    w = small(T=6, dtype=dtype, layout=layout)
    inp = wl.make_inputs(w)
    full = run_oracle_verify(w, inp)
    w1 = w.replace(T=1, layout="dense")
    cur = clone_inputs(inp)
    for t in range(w.T):
        step = dict(cur)
        step["x"] = inp["x"][:, t:t + 1, :]
        step["out"] = wl.sentinel_tensor((w.n_seq, 1, w.dim), w.torch_dtype)
        step["window"] = wl.sentinel_tensor(wl.window_shape(w1), w.torch_dtype)
        r1 = run_oracle_verify(w1, step)
        assert_bits_equal(r1["out"][:, 0], full["out"][:, t], f"out token {t}")
        for s in range(w.n_seq):
            slot = int(inp["cache_idx"][s])
            snap = r1["conv_state"][slot, :, :w.width - 1]
            if layout == "dense":
                got = full["window"][s, t]
            else:
                got = full["window"][s, :, t:t + w.width - 1]
            assert_bits_equal(got, snap, f"snapshot {t} seq {s}")
        cur["conv_state"] = r1["conv_state"]
    assert_bits_equal(full["conv_state"], cur["conv_state"], "final state")


def test_p5_batched_equals_separate():
    """P-5: a batched run equals n separate single-sequence runs bit for bit (Atlas batched doc:
    bit-identical to n separate calls; only the base addresses differ)."""
    w = small(n_seq=4, dtype="bf16", layout="dedup", n_pad=1, extra_slots=3)
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    for s in range(w.n_seq):
        one = clone_inputs(inp)
        ws = w.replace(n_seq=1, n_pad=0)
        one["x"] = inp["x"][s:s + 1]
        one["cache_idx"] = inp["cache_idx"][s:s + 1].clone()
        one["out"] = wl.sentinel_tensor((1, w.T, w.dim), w.torch_dtype)
        one["window"] = wl.sentinel_tensor(wl.window_shape(ws), w.torch_dtype)
        r1 = run_oracle_verify(ws, one)
        assert_bits_equal(r1["out"][0], r["out"][s], "out")
        assert_bits_equal(r1["window"][0], r["window"][s], "window")
        slot = int(inp["cache_idx"][s])
        if slot >= 0:
            assert_bits_equal(r1["conv_state"][slot], r["conv_state"][slot], "state")


@pytest.mark.parametrize("width", [2, 3, 4])
def test_p6_dedup_view_equals_dense(width):
    """P-6: the deduplicated row read through its overlapping [T, dim, W-1] view gives the dense
    snapshots bitwise (PR #46184: step stride == window stride makes both writes land on the
    same addresses with the same values); also through the transposed row layout."""
    w = small(width=width, dtype="bf16", T=8)
    inp = wl.make_inputs(w)
    dense = run_oracle_verify(w, inp)
    wd = w.replace(layout="dedup")
    inp_d = clone_inputs(inp)
    inp_d["window"] = wl.sentinel_tensor(wl.window_shape(wd), w.torch_dtype)
    dedup = run_oracle_verify(wd, inp_d)
    row = dedup["window"]
    view = row.as_strided((w.n_seq, w.T, w.dim, width - 1), (row.stride(0), row.stride(2), row.stride(1), row.stride(2)))
    assert_bits_equal(view, dense["window"], "dedup view vs dense")
    assert_bits_equal(dedup["out"], dense["out"], "out")
    assert_bits_equal(dedup["conv_state"], dense["conv_state"], "state")
    # transposed row layout ([n_seq, T+W-2, dim] storage seen as [n_seq, dim, T+W-2])
    inp_t = clone_inputs(inp)
    inp_t["window"] = wl.sentinel_tensor((w.n_seq, w.T + width - 2, w.dim), w.torch_dtype).transpose(1, 2)
    tr = run_oracle_verify(wd, inp_t)
    assert_bits_equal(tr["window"], row, "transposed row")


def test_p7_padded_rows_untouched():
    """P-7: padded sequences (cache index -1) leave their out rows, window rows and every unused
    slot untouched (PR #46184: padded rows exit before any store)."""
    w = small(n_seq=6, n_pad=3, extra_slots=4, dtype="bf16", layout="dedup")
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    used = {int(v) for v in inp["cache_idx"] if v >= 0}
    for s in range(w.n_seq):
        if int(inp["cache_idx"][s]) < 0:
            assert_bits_equal(r["out"][s], inp["out"][s], "padded out")
            assert_bits_equal(r["window"][s], inp["window"][s], "padded window")
            assert int(r["status"][s]) == 0
    for slot in range(w.n_slots):
        if slot not in used:
            assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], f"unused slot {slot}")


def test_p8_group_norms_and_v_passthrough():
    """P-8: every q|k group of every token has norm sqrt(ss / (ss + eps)) = 1 to within the fp32
    rounding of the sum; V channels equal a run without L2 bitwise (mod.rs: q/k normalised
    exactly once, V never)."""
    w = small(dim=160, qk_channels=128, head_dim=32, T=6, dtype="f32")
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    r0 = run_oracle_verify(w.replace(qk_channels=0), inp)
    out = r["out"].double()
    for g in range(0, 128, 32):
        n = out[:, :, g:g + 32].pow(2).sum(-1).sqrt()
        assert torch.allclose(n, torch.ones_like(n), atol=2e-6)
    assert_bits_equal(r["out"][:, :, 128:], r0["out"][:, :, 128:], "V channels")
    wb = w.replace(dtype="bf16")
    rb = run_oracle_verify(wb, wl.make_inputs(wb))
    ob = rb["out"].double()
    for g in range(0, 128, 32):
        n = ob[:, :, g:g + 32].pow(2).sum(-1).sqrt()
        assert torch.allclose(n, torch.ones_like(n), atol=2 ** -8)


@pytest.mark.parametrize("layout", ["dense", "dedup"])
def test_p9_commit_equals_shorter_verify(layout):
    """P-9: verify(T) then commit(a) leaves the state of verify over the first a tokens, bitwise
    (the window lets the accepted prefix's state be restored)."""
    w = small(n_seq=5, T=7, dtype="bf16", layout=layout, n_pad=1, extra_slots=2)
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    st = run_oracle_commit(w, r)
    assert (st == 0).all()
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        a = int(inp["accept_len"][s])
        wa = w.replace(T=a, n_seq=1, n_pad=0)
        one = clone_inputs(inp)
        one["x"] = inp["x"][s:s + 1, :a]
        one["cache_idx"] = inp["cache_idx"][s:s + 1].clone()
        one["out"] = wl.sentinel_tensor((1, a, w.dim), w.torch_dtype)
        one["window"] = wl.sentinel_tensor(wl.window_shape(wa), w.torch_dtype)
        ra = run_oracle_verify(wa, one)
        assert_bits_equal(r["conv_state"][slot], ra["conv_state"][slot], f"seq {s} accept {a}")


def test_p10_state_offset_equals_preshifted_state():
    """P-10: reading the committed window at offset o equals reading a state pre-shifted to offset
    0 (PR #46184 covers a num_accept_tokens state offset)."""
    w = small(n_seq=4, T=5, width=3, state_offset=True, dtype="bf16", qk_channels=0)
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        o = int(inp["state_off"][s])
        one = clone_inputs(inp)
        ws = w.replace(n_seq=1, state_offset=False)
        shifted = inp["conv_state"][slot:slot + 1, :, o:o + w.width - 1].clone()
        one["conv_state"] = shifted
        one["x"] = inp["x"][s:s + 1]
        one["cache_idx"] = torch.zeros(1, dtype=torch.int32)
        one["state_off"] = None
        one["out"] = wl.sentinel_tensor((1, w.T, w.dim), w.torch_dtype)
        one["window"] = wl.sentinel_tensor(wl.window_shape(ws), w.torch_dtype)
        r1 = run_oracle_verify(ws, one)
        assert_bits_equal(r1["out"][0], r["out"][s], "out")
        assert_bits_equal(r1["window"][0], r["window"][s], "window")
        assert_bits_equal(r1["conv_state"][0], r["conv_state"][slot, :, :w.width - 1], "committed window")
        # columns at and above W-1 are untouched
        assert_bits_equal(r["conv_state"][slot, :, w.width - 1:], inp["conv_state"][slot, :, w.width - 1:], "tail")


def _history_and_dedup(width, seed=11):
    wh = small(n_seq=5, T=6, width=width, dtype="bf16", layout="history", state_offset=True, n_pad=1,
               extra_slots=2, seed=seed)
    inp = wl.make_inputs(wh)
    assert inp["window"] is None and inp["conv_state"].shape[2] == wh.T + width - 2
    return wh, inp


@pytest.mark.parametrize("width", [2, 3, 4])
def test_h1_history_row_equals_dedup_row(width):
    """History layout (the state row is the deduplicated row of sglang PR #46184, "Motivation"):
    for the same inputs and offsets, each active slot's state row receives bitwise the row the
    dedup layout writes to its window buffer, the outputs are bitwise equal, and columns at and
    above T+W-2, unused slots and padded sequences' slots are untouched."""
    wh, inp = _history_and_dedup(width)
    Q = wh.T + width - 2
    wide = torch.cat([inp["conv_state"], wl.sentinel_tensor((wh.n_slots, wh.dim, 2), wh.torch_dtype)], dim=2)
    ih = clone_inputs(inp)
    ih["conv_state"] = wide.clone()
    rh = run_oracle_verify(wh, ih)
    wd = wh.replace(layout="dedup")
    assert wd.state_cols == Q
    idd = clone_inputs(inp)
    idd["window"] = wl.sentinel_tensor(wl.window_shape(wd), wd.torch_dtype)
    rd = run_oracle_verify(wd, idd)
    assert (rh["status"] == 0).all()
    assert_bits_equal(rh["out"], rd["out"], "out")
    active = set()
    for s in range(wh.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        active.add(slot)
        assert_bits_equal(rh["conv_state"][slot, :, :Q], rd["window"][s], f"seq {s} history row")
    assert_bits_equal(rh["conv_state"][:, :, Q:], wide[:, :, Q:], "columns beyond the row")
    for slot in range(wh.n_slots):
        if slot not in active:
            assert_bits_equal(rh["conv_state"][slot], wide[slot], f"untouched slot {slot}")


def test_h2_history_chain_equals_verify_commit_chain():
    """Two steps with the history layout (verify at offsets o, then verify at accept_len - 1, no
    commit) against the plain layout (verify on the committed windows, commit, verify, commit):
    the outputs of both steps agree bitwise, and after step 2 the history row read at a2 - 1 is the
    state the plain chain commits (PR #46184: the window restores the accepted prefix's state)."""
    wh, inp1 = _history_and_dedup(4, seed=21)
    R = wh.width - 1
    x2 = wl.make_inputs(wh, seed=22)
    cidx = inp1["cache_idx"]
    o1, a1, a2 = inp1["state_off"], inp1["accept_len"], x2["accept_len"]
    # history chain
    h1 = run_oracle_verify(wh, inp1)
    i2 = clone_inputs(inp1)
    i2.update(x=x2["x"], x_base=x2["x_base"], conv_state=h1["conv_state"].clone(), state_off=(a1 - 1).to(torch.int32),
              out=wl.sentinel_tensor((wh.n_seq, wh.T, wh.dim), wh.torch_dtype))
    h2 = run_oracle_verify(wh, i2)
    # plain chain on the committed windows (state pre-shifted to offset 0, pinned by P-10)
    wp = wh.replace(layout="dedup", state_offset=False)
    st0 = wl.sentinel_tensor((wp.n_slots, wp.dim, R), wp.torch_dtype)
    for s in range(wh.n_seq):
        slot = int(cidx[s])
        if slot >= 0:
            st0[slot] = inp1["conv_state"][slot, :, int(o1[s]):int(o1[s]) + R]
    p1in = clone_inputs(inp1)
    p1in.update(conv_state=st0, state_off=None, window=wl.sentinel_tensor(wl.window_shape(wp), wp.torch_dtype))
    p1 = run_oracle_verify(wp, p1in)
    assert (run_oracle_commit(wp, p1, accept_len=a1) == 0).all()
    p2in = clone_inputs(p1)
    p2in.update(x=x2["x"], x_base=x2["x_base"], out=wl.sentinel_tensor((wh.n_seq, wh.T, wh.dim), wh.torch_dtype),
                window=wl.sentinel_tensor(wl.window_shape(wp), wp.torch_dtype))
    p2 = run_oracle_verify(wp, p2in)
    assert (run_oracle_commit(wp, p2, accept_len=a2) == 0).all()
    assert_bits_equal(h1["out"], p1["out"], "step 1 out")
    assert_bits_equal(h2["out"], p2["out"], "step 2 out")
    for s in range(wh.n_seq):
        slot = int(cidx[s])
        if slot < 0:
            continue
        a = int(a2[s])
        assert_bits_equal(h2["conv_state"][slot, :, a - 1:a - 1 + R], p2["conv_state"][slot], f"seq {s} committed")


def test_h3_history_sequential_single_tokens():
    """P-4 in the history layout: T calls of one token each, every call reading the committed
    window at column 0 of the row the previous call wrote (the whole token accepted), give the
    outputs of one call over the T tokens bitwise, and the last call's row starts with the window
    the T-token call leaves at column T-1."""
    T = 7
    wh = small(n_seq=3, T=T, width=4, dtype="f32", layout="history", state_offset=False)
    inp = wl.make_inputs(wh)
    R = wh.width - 1
    whole = run_oracle_verify(wh, inp)
    w1 = wh.replace(T=1)
    st = wl.sentinel_tensor((wh.n_slots, wh.dim, R), wh.torch_dtype)
    st[:] = inp["conv_state"][:, :, :R]
    for t in range(T):
        one = clone_inputs(inp)
        one.update(x=inp["x"][:, t:t + 1], conv_state=st, out=wl.sentinel_tensor((wh.n_seq, 1, wh.dim), wh.torch_dtype))
        r = run_oracle_verify(w1, one)
        st = r["conv_state"]
        assert_bits_equal(r["out"][:, 0], whole["out"][:, t], f"token {t}")
    for s in range(wh.n_seq):
        slot = int(inp["cache_idx"][s])
        assert_bits_equal(st[slot], whole["conv_state"][slot, :, T - 1:T - 1 + R], f"seq {s} final window")


def test_h4_column_major_rows_are_storage_only():
    """The state rows' storage order is not part of the method: the oracle run on column-major
    rows ([n_slots, S, dim] seen transposed) writes the same values as on row-major rows, and
    leaves the column-major storage column-major."""
    w = small(n_seq=4, T=5, width=4, dtype="bf16", layout="history", state_offset=True)
    inp = wl.make_inputs(w)
    ref = run_oracle_verify(w, inp)
    cm = clone_inputs(inp)
    st = torch.empty((w.n_slots, w.state_cols, w.dim), dtype=w.torch_dtype).transpose(1, 2)
    st.copy_(inp["conv_state"])
    cm["conv_state"] = st
    got = run_oracle_verify(w, cm)
    assert got["conv_state"].stride(1) == 1
    assert_bits_equal(got["conv_state"], ref["conv_state"], "state rows")
    assert_bits_equal(got["out"], ref["out"], "out")


@pytest.mark.parametrize("width", [2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_r1_recompute_verify_writes_outputs_only(width, dtype):
    """Recompute layout (memra-engine ssm_conv_ring_rebuild_dc keeps the pre-verify ring): the
    outputs equal the dense layout's bitwise, and no state element changes."""
    wr = small(n_seq=4, T=6, width=width, dtype=dtype, layout="recompute", n_pad=1, extra_slots=2, seed=41)
    inp = wl.make_inputs(wr)
    assert inp["window"] is None
    rr = run_oracle_verify(wr, inp)
    wd = wr.replace(layout="dense")
    idn = clone_inputs(inp)
    idn["window"] = wl.sentinel_tensor(wl.window_shape(wd), wd.torch_dtype)
    rd = run_oracle_verify(wd, idn)
    assert_bits_equal(rr["out"], rd["out"], "out")
    assert_bits_equal(rr["conv_state"], inp["conv_state"], "state untouched")
    assert_bits_equal(rr["status"], rd["status"], "status")


@pytest.mark.parametrize("layout", ["dense", "dedup"])
def test_r2_recompute_commit_equals_snapshot_commit(layout):
    """For every accept count a in 1..T, the rebuilt state equals the state the snapshot path
    commits (P-9 pins that one to a shorter verify), bitwise; padded and unused slots untouched."""
    T = 7
    wr = small(n_seq=T + 1, T=T, width=4, dtype="bf16", layout="recompute", n_pad=1, extra_slots=2, seed=43)
    inp = wl.make_inputs(wr)
    inp["accept_len"] = torch.tensor([1 + s % T for s in range(wr.n_seq)], dtype=torch.int32)
    rr = run_oracle_verify(wr, inp)
    assert (run_oracle_commit(wr, rr) == 0).all()
    wd = wr.replace(layout=layout)
    idn = clone_inputs(inp)
    idn["window"] = wl.sentinel_tensor(wl.window_shape(wd), wd.torch_dtype)
    rd = run_oracle_verify(wd, idn)
    assert (run_oracle_commit(wd, rd) == 0).all()
    assert_bits_equal(rr["conv_state"], rd["conv_state"], "rebuilt state")


def test_r3_recompute_commit_closed_form():
    """Closed form: with a >= W-1 the rebuilt window is x_{a-W+1} .. x_{a-1} (inputs only); with
    a < W-1 it is the old window shifted left by a, then x_0 .. x_{a-1}."""
    W, T = 4, 5
    wr = small(n_seq=T, T=T, width=W, dtype="f32", layout="recompute", seed=47)
    inp = wl.make_inputs(wr)
    inp["accept_len"] = torch.arange(1, T + 1, dtype=torch.int32)
    rr = run_oracle_verify(wr, inp)
    run_oracle_commit(wr, rr)
    for s in range(wr.n_seq):
        slot, a = int(inp["cache_idx"][s]), int(inp["accept_len"][s])
        old = inp["conv_state"][slot]           # [dim, W-1]
        xs = inp["x"][s].t()                    # [dim, T]
        want = xs[:, a - (W - 1):a] if a >= W - 1 else torch.cat([old[:, a:], xs[:, :a]], dim=1)
        assert_bits_equal(rr["conv_state"][slot], want.contiguous(), f"seq {s} a {a}")


def test_p11_single_token_update():
    """P-11: T = 1 is the standard single-token causal conv update: the state shifts left by one
    and takes x; out = SiLU(sum_j w_j [state, x]_j + bias)."""
    w = small(T=1, qk_channels=0, dtype="f32")
    inp = wl.make_inputs(w)
    r = run_oracle_verify(w, inp)
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        st = inp["conv_state"][slot]
        want_state = torch.cat([st[:, 1:], inp["x"][s, 0][:, None]], dim=1)
        assert_bits_equal(r["conv_state"][slot], want_state, "shifted state")
        full = torch.cat([st, inp["x"][s, 0][:, None]], dim=1).double()
        acc = (full * inp["weight"].double()).sum(1) + inp["bias"].double()
        assert torch.allclose(r["out"][s, 0].double(), acc / (1 + torch.exp(-acc)), rtol=1e-5, atol=1e-6)


def test_bf16_rounding_matches_torch():
    """The oracle's fp32 -> bf16 rounding (nearest, ties to even) equals torch's conversion on
    random values, ties, subnormals, infinities and signed zeros."""
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-40, 39, 20000),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  1.0 + 2 ** -8 + 2 ** -20, 1.17e-38, 5.9e-39], dtype=np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_f32_to_bf16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.round_f32_to_bf16_bits(float("nan")) & 0x7FFF > 0x7F80


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


def test_golden_dedup_row_columns():
    """The page's printed row layout (tests/golden/dedup_row_columns.txt): the row is the committed
    window without its oldest column followed by x_0 .. x_{T-1} (T+2 columns for width 4), and the
    window of step t is its 3 columns from column t, for the T values the page tests."""
    for line in _read_golden("dedup_row_columns.txt"):
        T_s, cols = line.split(":")
        T = int(T_s)
        labels = cols.split()
        assert len(labels) == T + 2
        w = small(n_seq=1, T=T, dim=8, width=4, qk_channels=0, dtype="f32", layout="dedup", bias=False)
        inp = wl.make_inputs(w)
        slot = int(inp["cache_idx"][0])
        # every input gets a distinct exactly representable tag
        for k in range(3):
            inp["conv_state"][slot, :, k] = 1000.0 + k
        for t in range(T):
            inp["x"][0, t, :] = 2000.0 + t
        r = run_oracle_verify(w, inp)
        tag = {f"state[{k}]": 1000.0 + k for k in range(3)}
        tag.update({f"x_{t}": 2000.0 + t for t in range(T)})
        want = torch.tensor([tag[l] for l in labels], dtype=torch.float32)
        for c in range(w.dim):
            assert torch.equal(r["window"][0, c], want)
            for t in range(T):
                assert torch.equal(r["window"][0, c, t:t + 3], want[t:t + 3])


def test_status_codes_and_untouched():
    """Out-of-range slot, state offset or accept count flags the sequence and touches nothing."""
    w = small(n_seq=4, T=4, state_offset=True, dtype="bf16")
    inp = wl.make_inputs(w)
    inp["cache_idx"][0] = w.n_slots  # slot out of range
    inp["state_off"][1] = w.state_cols - w.width + 2  # window would run past the row
    inp["state_off"][2] = -1
    r = run_oracle_verify(w, inp)
    assert r["status"].tolist()[:3] == [1, 2, 2] and int(r["status"][3]) == 0
    for s in range(3):
        assert_bits_equal(r["out"][s], inp["out"][s], "flagged out")
        assert_bits_equal(r["window"][s], inp["window"][s], "flagged window")
    acc = inp["accept_len"].clone()
    acc[3] = w.T + 1
    before = r["conv_state"].clone()
    st = run_oracle_commit(w, r, accept_len=acc)
    assert int(st[3]) == 4 and int(st[0]) == 1
    slot3 = int(inp["cache_idx"][3])
    assert_bits_equal(r["conv_state"][slot3], before[slot3], "rejected commit")


def test_nan_and_signed_zero_copies():
    """Snapshots and state are raw copies: NaN payloads and -0 survive; outputs follow IEEE."""
    w = small(n_seq=1, T=3, dtype="bf16", layout="dense", qk_channels=0)
    inp = wl.make_inputs(w)
    slot = int(inp["cache_idx"][0])
    inp["conv_state"].view(torch.int16)[slot, 0, 1] = 0x7FA1  # NaN with a payload
    inp["x"].view(torch.int16)[0, 0, 1] = -32768  # -0.0
    r = run_oracle_verify(w, inp)
    wb = bits(r["window"])
    assert wb[0, 0, 0, 0] == 0x7FA1
    assert wb[0, 0, 1, 2] == 0x8000 and wb[0, 1, 1, 1] == 0x8000 and wb[0, 2, 1, 0] == 0x8000
    assert np.isnan(r["out"][0, :2, 0].float().numpy()).all()


def _mixed(layout, x_dtype, state_dtype, seed=61, **kw):
    w = small(n_seq=4, T=5, width=4, dtype=x_dtype, state_dtype=state_dtype, layout=layout, n_pad=1, extra_slots=1,
              seed=seed, **kw)
    return w, wl.make_inputs(w)


@pytest.mark.parametrize("layout", ["dense", "dedup", "history"])
def test_m1_bf16_inputs_fp32_state_equal_the_bf16_run(layout):
    """Mixed dtypes (sglang PR #46184, "Accuracy Tests": mixed input and state dtypes).  bf16 x with
    an fp32 state holding bf16 values computes what the all-bf16 run computes: outputs bitwise, and
    snapshots and state equal the bf16 ones widened to fp32 (an exact conversion)."""
    w = small(n_seq=4, T=5, width=4, dtype="bf16", layout=layout, n_pad=1, extra_slots=1, seed=61,
              state_offset=(layout == "history"))
    inp = wl.make_inputs(w)
    rb = run_oracle_verify(w, inp)
    wm = w.replace(state_dtype="f32")
    im = clone_inputs(inp)
    im["conv_state"] = inp["conv_state"].float()
    if inp["window"] is not None:
        im["window"] = inp["window"].float()
    rm = run_oracle_verify(wm, im)
    assert_bits_equal(rm["out"], rb["out"], "out")
    assert_bits_equal(rm["conv_state"], rb["conv_state"].float(), "state")
    if layout != "history":
        assert_bits_equal(rm["window"], rb["window"].float(), "window")


@pytest.mark.parametrize("layout", ["dense", "dedup"])
def test_m2_fp32_inputs_bf16_state_equal_the_fp32_run(layout):
    """fp32 x holding bf16 values with a bf16 state computes what the all-fp32 run computes on the
    widened state: outputs bitwise; snapshots and state are the fp32 ones narrowed (exactly)."""
    w = small(n_seq=4, T=5, width=4, dtype="f32", layout=layout, n_pad=1, extra_slots=1, seed=63)
    inp = wl.make_inputs(w)
    inp["x_base"] = inp["x_base"].bfloat16().float()
    inp["x"] = inp["x_base"].as_strided(inp["x"].shape, inp["x"].stride(), inp["x"].storage_offset())
    inp["conv_state"] = inp["conv_state"].bfloat16().float()
    rf = run_oracle_verify(w, inp)
    wm = w.replace(state_dtype="bf16")
    im = clone_inputs(inp)
    im["conv_state"] = inp["conv_state"].bfloat16()
    im["window"] = inp["window"].bfloat16()
    rm = run_oracle_verify(wm, im)
    assert_bits_equal(rm["out"], rf["out"], "out")
    assert_bits_equal(rm["conv_state"], rf["conv_state"].bfloat16(), "state")
    assert_bits_equal(rm["window"], rf["window"].bfloat16(), "window")


def test_m3_fp32_inputs_round_into_bf16_snapshots():
    """fp32 x (not bf16-representable) into a bf16 state: the snapshot elements that come from x
    equal torch's round-to-nearest-even conversion of x, those from the old state its raw bits."""
    w, inp = _mixed("dense", "f32", "bf16", seed=65)
    r = run_oracle_verify(w, inp)
    R = w.width - 1
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        full = torch.cat([inp["conv_state"][slot], inp["x"][s].t().to(torch.bfloat16)], dim=1)  # [dim, R+T]
        for t in range(w.T):
            assert_bits_equal(r["window"][s, t], full[:, t + 1:t + 1 + R].contiguous(), f"seq {s} snapshot {t}")
        assert_bits_equal(r["conv_state"][slot], full[:, w.T:w.T + R].contiguous(), f"seq {s} state")


@pytest.mark.parametrize("xd,sd", [("bf16", "f32"), ("f32", "bf16")])
def test_m4_mixed_matches_float64_conv1d(xd, sd):
    """Library special case with mixed dtypes: outputs equal torch float64 conv1d over [state
    window, x] (each widened from its own dtype) with SiLU and L2, within 1e-5 relative."""
    w, inp = _mixed("dense", xd, sd, seed=67)
    r = run_oracle_verify(w, inp)
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        full = torch.cat([inp["conv_state"][slot].double(), inp["x"][s].double().t()], dim=1)
        acc = F.conv1d(full[None], inp["weight"].double()[:, None, :], inp["bias"].double(), groups=w.dim)[0]
        y = (acc / (1 + torch.exp(-acc))).t()
        g = y[:, : w.qk_channels].reshape(w.T, -1, w.head_dim)
        y[:, : w.qk_channels] = (g / torch.sqrt((g * g).sum(-1, keepdim=True) + w.l2_eps)).reshape(w.T, -1)
        got = r["out"][s].double()
        tol = 1e-5 if xd == "f32" else 2 ** -7
        assert torch.allclose(got, y, rtol=tol, atol=1e-6), float((got - y).abs().max())


def _tree_inputs(w, parents, seed_shift=0):
    inp = wl.make_inputs(w, seed=w.seed + seed_shift)
    inp["parent"] = torch.tensor(parents, dtype=torch.int32).reshape(w.n_seq, w.T).contiguous()
    return inp


@pytest.mark.parametrize("width", [2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tr1_chain_parents_equal_the_plain_verify(width, dtype):
    """Tree verify (sglang PR #46184, "Scope": tree verify keeps dense windows): parents t-1 make a
    chain, which must reproduce the plain verify bitwise (outputs, snapshots, state)."""
    w = small(n_seq=4, T=6, width=width, dtype=dtype, layout="dense", n_pad=1, extra_slots=1, seed=71,
              state_offset=True)
    chain = [[t - 1 for t in range(w.T)] for _ in range(w.n_seq)]
    inp = _tree_inputs(w, chain)
    rt = run_oracle_verify(w, inp)
    plain = dict(inp)
    plain.pop("parent")
    rp = run_oracle_verify(w, plain)
    for k in ("out", "window", "conv_state", "status"):
        assert_bits_equal(rt[k], rp[k], k)


def _paths(parents):
    """Root-to-node token lists of a parent array."""
    out = []
    for t in range(len(parents)):
        p, path = t, []
        while p >= 0:
            path.append(p)
            p = parents[p]
        out.append(path[::-1])
    return out


def test_tr2_tree_paths_equal_chain_verifies():
    """Every node of a branching tree gets the output and snapshot that a chain verify over its
    root-to-node path gives for its last token (bitwise)."""
    T = 7
    parents = [-1, 0, 0, 1, 1, 2, -1]  # two roots, branches at 0 and 1
    w = small(n_seq=1, T=T, width=4, dtype="bf16", layout="dense", n_pad=0, extra_slots=0, seed=73)
    inp = _tree_inputs(w, [parents])
    rt = run_oracle_verify(w, inp)
    for t, path in enumerate(_paths(parents)):
        L = len(path)
        wc = w.replace(T=L)
        one = clone_inputs(inp)
        one.pop("parent")
        xc = inp["x"][:, path].contiguous()
        one.update(x=xc, x_base=xc, out=wl.sentinel_tensor((1, L, w.dim), w.torch_dtype),
                   window=wl.sentinel_tensor(wl.window_shape(wc), w.torch_dtype))
        rc = run_oracle_verify(wc, one)
        assert_bits_equal(rt["out"][0, t], rc["out"][0, L - 1], f"node {t} out")
        assert_bits_equal(rt["window"][0, t], rc["window"][0, L - 1], f"node {t} snapshot")


def test_tr3_commit_of_an_accepted_node_equals_its_path_state():
    """Committing the window of an accepted path's last token (accept_len = its index + 1) leaves
    the state a chain verify over that path leaves, bitwise."""
    T = 6
    parents = [-1, 0, 0, 2, 1, 4]
    w = small(n_seq=1, T=T, width=3, dtype="f32", layout="dense", n_pad=0, extra_slots=0, seed=75)
    inp = _tree_inputs(w, [parents])
    for node, path in enumerate(_paths(parents)):
        rt = run_oracle_verify(w, inp)
        assert (run_oracle_commit(w, rt, accept_len=torch.tensor([node + 1], dtype=torch.int32)) == 0).all()
        wc = w.replace(T=len(path))
        one = clone_inputs(inp)
        one.pop("parent")
        xc = inp["x"][:, path].contiguous()
        one.update(x=xc, x_base=xc, out=wl.sentinel_tensor((1, len(path), w.dim), w.torch_dtype),
                   window=wl.sentinel_tensor(wl.window_shape(wc), w.torch_dtype))
        rc = run_oracle_verify(wc, one)
        assert_bits_equal(rt["conv_state"], rc["conv_state"], f"node {node}")


def test_tree_invalid_parents_flagged():
    """A parent outside [-1, t) flags the sequence (32) and touches nothing of it."""
    w = small(n_seq=3, T=4, width=4, dtype="bf16", layout="dense", n_pad=0, extra_slots=0, seed=77)
    inp = _tree_inputs(w, [[-1, 0, 1, 2], [-1, 1, 0, 0], [-2, 0, 0, 0]])
    r = run_oracle_verify(w, inp)
    assert r["status"].tolist() == [0, 32, 32]
    for s in (1, 2):
        slot = int(inp["cache_idx"][s])
        assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], "state")
        assert_bits_equal(r["window"][s], inp["window"][s], "window")


@pytest.mark.parametrize("layout", ["dense", "dedup"])
def test_p_extreme_conv_values_match_float64(layout):
    """Conv results far from zero on both sides (x and state scaled by 200: about a fifth of them
    below -80, where exp(-acc) passes 1e34 and, past -88.7, overflows fp32): the oracle's fp32
    SiLU and L2 still match the float64 definition within the fp32 output tolerance."""
    w = small(dtype="f32", layout=layout, width=4, n_pad=0, extra_slots=1, seed=303)
    inp = wl.make_inputs(w)
    inp["x_base"].mul_(200.0)
    inp["conv_state"].mul_(200.0)
    r = run_oracle_verify(w, inp)
    outs, _, _ = float64_reference(w, inp)
    below = 0
    for s, ref in outs.items():
        got = r["out"][s].double()
        err = (got - ref).abs()
        assert (err <= 1e-5 * ref.abs() + 1e-6).all(), float(err.max())
        slot = int(inp["cache_idx"][s])
        full = torch.cat([inp["conv_state"][slot, :, :3].double(), inp["x"][s].double().t()], dim=1)
        acc = F.conv1d(full[None], inp["weight"].double()[:, None, :], inp["bias"].double(), groups=w.dim)[0]
        below += int((acc < -80).sum())
    assert below > 0.1 * w.n_seq * w.T * w.dim  # the range the exact SiLU form covers is exercised
