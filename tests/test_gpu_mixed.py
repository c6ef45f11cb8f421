"""GPU parity with mixed dtypes: the state and the snapshots in the other dtype than x (bf16 x with
fp32 state, fp32 x with bf16 state).  State, snapshots and status bitwise; outputs within the
output tolerance of x's dtype."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_commit, run_gpu_verify
from helpers import assert_bits_equal, assert_out_close, run_oracle_commit, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def check(cv, w, inp, commit=True):
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cv, w, inp)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    if inp["window"] is not None:
        assert_bits_equal(got["window"].cpu(), ref["window"], "window")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    if commit and w.layout in ("dense", "dedup"):
        st_ref = run_oracle_commit(w, ref)
        st_got = run_gpu_commit(cv, w, got)
        assert_bits_equal(st_got.cpu(), st_ref, "commit err")
        assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "committed state")


@pytest.mark.parametrize("case", range(24))
def test_mixed_random_sweep(cuda_lib, case):
    """Random shapes in both directions and every layout: W 2..4, T up to 17 and beyond, ragged
    dims, head dims, bias, padded rows, state offsets."""
    rng = np.random.default_rng(11000 + case)
    xd = "bf16" if case % 2 == 0 else "f32"
    sd = "f32" if xd == "bf16" else "bf16"
    layout = ["dense", "dedup", "history", "recompute"][case % 4]
    over = dict(dtype=xd, state_dtype=sd, layout=layout, state_offset=bool(case % 3 == 1) or layout == "history")
    if case % 5 == 0:
        over.update(n_pad=1, extra_slots=2, n_seq=4)
    w = wl.random_case(rng, **over)
    if w.n_pad >= w.n_seq:
        w = w.replace(n_pad=w.n_seq - 1)
    check(cuda_lib, w, wl.make_inputs(w))


def test_mixed_benchmark_shape(cuda_lib):
    """128 x 8 x 10240: bf16 x, fp32 state and fp32 dedup rows, with the commit."""
    w = wl.WORKLOADS["n128_t8_dim10240_w4_bf16x_f32state_dedup_pad13"]
    check(cuda_lib, w, wl.make_inputs(w))


def test_mixed_nan_and_rounding(cuda_lib):
    """fp32 x into a bf16 state: NaN inputs become the quiet NaN 0x7fc0 in the snapshots and the
    state, ties round to even, and values round as the oracle (and torch) round them."""
    w = wl.VerifyWorkload("mixnan", n_seq=2, T=4, dim=64, width=4, qk_channels=0, head_dim=8, dtype="f32",
                          state_dtype="bf16", layout="dense", seed=3)
    inp = wl.make_inputs(w)
    x = inp["x"]
    x[0, 1, 3] = float("nan")
    x[1, 2, 5] = torch.tensor(0x7fa12345, dtype=torch.int32).view(torch.float32)  # signalling NaN payload
    x[0, 3, 7] = torch.tensor(0x3f808000, dtype=torch.int32).view(torch.float32)  # a tie: rounds to even
    x[1, 3, 9] = -0.0
    check(cuda_lib, w, inp, commit=False)


def _plan_path(cv, w, inp):
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    return cv.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                          qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                          state_off=d["state_off"]).path


@pytest.mark.parametrize("case", range(16))
def test_mixed_pipelined_sweep(cuda_lib, case):
    """Packed buffers with T <= 8 take the pipelined kernel in both directions and every layout:
    W 2..4, dims that leave a ragged last channel block, L2 groups of 8..128, bias, padded
    sequences, unused pool slots, wide state rows read at offsets (dense and dedup) and history
    rows."""
    rng = np.random.default_rng(12000 + case)
    xd = "bf16" if case % 2 == 0 else "f32"
    sd = "f32" if xd == "bf16" else "bf16"
    layout = ["dense", "dedup", "history", "recompute"][(case // 2) % 4]
    T = int(rng.integers(1, 9))
    width = int(rng.integers(2, 5))
    hd = int(rng.choice([8, 32, 64, 128]))
    qk = int(rng.integers(0, 4)) * hd
    dim = qk + 8 * int(rng.integers(1, 200))
    w = wl.VerifyWorkload("mixpipe", n_seq=int(rng.integers(2, 40)), T=T, dim=dim, width=width, qk_channels=qk,
                          head_dim=hd, dtype=xd, state_dtype=sd, layout=layout, bias=bool(case % 3),
                          n_pad=1, extra_slots=2, state_offset=layout == "history" or (case % 8 >= 4 and T > 1),
                          seed=700 + case)
    inp = wl.make_inputs(w)
    assert _plan_path(cuda_lib, w, inp) == 3
    check(cuda_lib, w, inp)


@pytest.mark.parametrize("T", [4, 9])
def test_mixed_state_nan_payloads_kept(cuda_lib, T):
    """A bf16 state holding NaNs with payloads, read with fp32 x: state columns move as raw bits
    (snapshots and the committed window keep each payload) while x enters as rounded bf16; on the
    pipelined kernel (T = 4) and the general one (T = 9)."""
    w = wl.VerifyWorkload("mixstnan", n_seq=3, T=T, dim=256, width=4, qk_channels=128, head_dim=64, dtype="f32",
                          state_dtype="bf16", layout="dedup", bias=True, seed=9 + T)
    inp = wl.make_inputs(w)
    st = inp["conv_state"].view(torch.int16)
    slots = inp["cache_idx"].tolist()
    st[slots[0], 5, 2] = 0x7fa1
    st[slots[1], 17, 1] = -1  # 0xffff: a negative quiet NaN with a full payload
    st[slots[2], 200, 0] = 0x7f81
    assert _plan_path(cuda_lib, w, inp) == (3 if T <= 8 else 0)
    check(cuda_lib, w, inp)


@pytest.mark.parametrize("xd,layout,T", [("bf16", "dedup", 8), ("f32", "dense", 5), ("bf16", "history", 3),
                                         ("f32", "recompute", 7), ("bf16", "dense", 1)])
def test_mixed_pipelined_head_dim_256(cuda_lib, xd, layout, T):
    """L2 groups of 256 channels: the pipelined kernel with 8 channels per thread, in both
    directions, with a ragged last channel block, padded sequences and a bias."""
    sd = "f32" if xd == "bf16" else "bf16"
    w = wl.VerifyWorkload("mix256", n_seq=9, T=T, dim=512 + 1024 + 40, width=4, qk_channels=1024, head_dim=256,
                          dtype=xd, state_dtype=sd, layout=layout, bias=True, n_pad=2, extra_slots=3,
                          state_offset=layout == "history", seed=T)
    inp = wl.make_inputs(w)
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    pl = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=layout,
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path == 3 and pl.channels_per_block == 8 * pl.threads
    check(cuda_lib, w, inp)
