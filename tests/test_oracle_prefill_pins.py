"""Pins of the CPU oracle's prefill (no GPU): a library special case, the verify oracle (pinned on
its own), splitting a prompt in two, the zero initial window and per-sequence independence.

glm5next_kda mod.rs (the layer's prefill path): the conv with SiLU over all prompt tokens, the L2
normalisation of q|k per head group; the state keeps the last W-1 inputs.
"""
from __future__ import annotations

import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import assert_bits_equal, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl


def small(**kw) -> wl.PrefillWorkload:
    base = dict(name="p", lengths=(7, 1, 0, 19, 12), dim=96, width=4, qk_channels=64, head_dim=16, dtype="f32",
                bias=True, pad=(2,), no_init=(3,), extra_slots=2, seed=31)
    base.update(kw)
    return wl.PrefillWorkload(**base)


def run_prefill(w: wl.PrefillWorkload, inp: dict) -> dict:
    r = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    r["x"] = inp["x"]
    r["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_prefill(r["x"], r["conv_state"], r["weight"], r["bias"], r["out"], r["cu_seqlens"],
                        qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=r["cache_idx"],
                        has_initial_state=r["has_initial_state"], status=r["status"])
    return r


@pytest.mark.parametrize("width", [2, 3, 4])
def test_pf1_matches_float64_conv1d(width):
    """Library special case: per sequence, torch float64 conv1d(groups=dim) over [initial window
    (zeros without an initial state), x] with SiLU and the per-group L2, within 1e-6 relative;
    the final state is the last W-1 inputs exactly."""
    w = small(width=width)
    inp = wl.make_prefill_inputs(w)
    r = run_prefill(w, inp)
    assert (r["status"] == 0).all()
    cu = inp["cu_seqlens"].tolist()
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        if slot < 0:
            continue
        b, e = cu[s], cu[s + 1]
        init = inp["conv_state"][slot].double() if int(inp["has_initial_state"][s]) else \
            torch.zeros(w.dim, width - 1, dtype=torch.float64)
        full = torch.cat([init, inp["x"][b:e].double().t()], dim=1)  # [dim, W-1+L]
        assert_bits_equal(r["conv_state"][slot], full[:, e - b:].to(w.torch_dtype).contiguous(), f"seq {s} state")
        if e == b:
            continue
        acc = F.conv1d(full[None], inp["weight"].double()[:, None, :], inp["bias"].double(), groups=w.dim)[0]
        y = (acc / (1 + torch.exp(-acc))).t()  # [L, dim]
        g = y[:, : w.qk_channels].reshape(e - b, -1, w.head_dim)
        y[:, : w.qk_channels] = (g / torch.sqrt((g * g).sum(-1, keepdim=True) + w.l2_eps)).reshape(e - b, -1)
        got = r["out"][b:e].double()
        assert torch.allclose(got, y, rtol=1e-5, atol=1e-6), float((got - y).abs().max())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pf2_equals_verify_over_the_same_tokens(dtype):
    """A prompt of L tokens with an initial state equals the verify oracle (pinned separately)
    over T = L draft tokens on the same window, bitwise: outputs, and the final state equals the
    verify's committed window."""
    L = 23
    w = small(lengths=(L,), pad=(), no_init=(), dtype=dtype, seed=33)
    inp = wl.make_prefill_inputs(w)
    r = run_prefill(w, inp)
    wv = wl.VerifyWorkload("v", n_seq=1, T=L, dim=w.dim, width=w.width, qk_channels=w.qk_channels,
                           head_dim=w.head_dim, dtype=dtype, layout="dense", bias=True, seed=0)
    vin = dict(x=inp["x"][None], x_base=inp["x"].clone(), conv_state=inp["conv_state"], weight=inp["weight"],
               bias=inp["bias"], cache_idx=inp["cache_idx"], state_off=None, accept_len=torch.ones(1, dtype=torch.int32),
               out=wl.sentinel_tensor((1, L, w.dim), w.torch_dtype),
               window=wl.sentinel_tensor(wl.window_shape(wv), w.torch_dtype))
    vin["x_base"] = vin["x"]
    rv = run_oracle_verify(wv, vin)
    assert_bits_equal(r["out"], rv["out"][0], "out")
    assert_bits_equal(r["conv_state"], rv["conv_state"], "state")


def test_pf3_split_prompt_equals_whole():
    """Prefill of a prompt equals prefill of its first part followed by prefill of the rest with
    the state the first part left, bitwise (outputs and final state), for every split point."""
    L = 17
    w = small(lengths=(L,), pad=(), no_init=(), seed=35)
    inp = wl.make_prefill_inputs(w)
    whole = run_prefill(w, inp)
    for cut in range(0, L + 1):
        a = dict(inp)
        a["x"], a["cu_seqlens"] = inp["x"][:cut], torch.tensor([0, cut], dtype=torch.int32)
        a["out"] = wl.sentinel_tensor((cut, w.dim), w.torch_dtype)
        ra = run_prefill(w.replace(lengths=(cut,)), a)
        b = dict(inp)
        b["x"], b["cu_seqlens"] = inp["x"][cut:], torch.tensor([0, L - cut], dtype=torch.int32)
        b["conv_state"] = ra["conv_state"]
        b["out"] = wl.sentinel_tensor((L - cut, w.dim), w.torch_dtype)
        rb = run_prefill(w.replace(lengths=(L - cut,)), b)
        assert_bits_equal(torch.cat([ra["out"], rb["out"]]), whole["out"], f"out, cut {cut}")
        assert_bits_equal(rb["conv_state"], whole["conv_state"], f"state, cut {cut}")


def test_pf4_no_initial_state_is_a_zero_window():
    """Without an initial state the window before the first token is zeros: the same as a run
    with the flag set on a zeroed state row (bitwise)."""
    w = small()
    inp = wl.make_prefill_inputs(w)
    r = run_prefill(w, inp)
    z = dict(inp)
    z["conv_state"] = inp["conv_state"].clone()
    for s in w.no_init:
        slot = int(inp["cache_idx"][s])
        if slot >= 0:
            z["conv_state"][slot] = 0
    z["has_initial_state"] = torch.ones(w.n_seq, dtype=torch.int32)
    rz = run_prefill(w, z)
    assert_bits_equal(r["out"], rz["out"], "out")
    assert_bits_equal(r["conv_state"], rz["conv_state"], "state")


def test_pf5_packed_equals_separate_and_untouched():
    """The packed batch equals each sequence run alone (bitwise); a padded sequence's tokens and
    slot, unused slots and an empty sequence's outputs are untouched; an empty sequence keeps (or
    zeroes, without an initial state) its window."""
    w = small(lengths=(7, 1, 0, 19, 12, 0), pad=(2,), no_init=(3, 5), seed=37)
    inp = wl.make_prefill_inputs(w)
    r = run_prefill(w, inp)
    cu = inp["cu_seqlens"].tolist()
    touched = set()
    for s in range(w.n_seq):
        slot = int(inp["cache_idx"][s])
        b, e = cu[s], cu[s + 1]
        if slot < 0:
            assert_bits_equal(r["out"][b:e], inp["out"][b:e], "padded out")
            continue
        touched.add(slot)
        one = dict(inp)
        one["x"], one["cu_seqlens"] = inp["x"][b:e], torch.tensor([0, e - b], dtype=torch.int32)
        one["cache_idx"] = inp["cache_idx"][s:s + 1]
        one["has_initial_state"] = inp["has_initial_state"][s:s + 1]
        one["out"] = wl.sentinel_tensor((e - b, w.dim), w.torch_dtype)
        r1 = run_prefill(w.replace(lengths=(e - b,), pad=(), no_init=()), one)
        assert_bits_equal(r["out"][b:e], r1["out"], f"seq {s} out")
        assert_bits_equal(r["conv_state"][slot], r1["conv_state"][slot], f"seq {s} state")
        if e == b:
            want = inp["conv_state"][slot] if int(inp["has_initial_state"][s]) else torch.zeros_like(inp["conv_state"][slot])
            assert_bits_equal(r["conv_state"][slot], want, f"empty seq {s}")
    for slot in range(w.n_slots):
        if slot not in touched:
            assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], f"slot {slot}")


def test_pf_bad_spans_flagged():
    """A span outside the packed tokens (or reversed) is flagged (16) and touches nothing."""
    w = small(lengths=(5, 6, 7), pad=(), no_init=(), seed=39)
    inp = wl.make_prefill_inputs(w)
    inp["cu_seqlens"] = torch.tensor([0, 5, 3, 40], dtype=torch.int32)
    r = run_prefill(w, inp)
    assert r["status"].tolist() == [0, 16, 16]
    for s in (1, 2):
        slot = int(inp["cache_idx"][s])
        assert_bits_equal(r["conv_state"][slot], inp["conv_state"][slot], "flagged state")
