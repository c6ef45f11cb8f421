"""GPU parity of the recompute rollback (no snapshots: the verify writes the outputs only and the
commit rebuilds the state from the kept window and the verify's inputs).

The state after verify (untouched), the state after commit and the status codes must match the
oracle bitwise, the outputs within the output tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_commit, run_gpu_verify
from helpers import assert_bits_equal, assert_out_close, clone_inputs, run_oracle_commit, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def check(cv, w, inp, accept=None):
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cv, w, inp)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    assert_bits_equal(got["conv_state"].cpu(), inp["conv_state"], "state untouched by the verify")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    st_ref = run_oracle_commit(w, ref, accept_len=accept)
    st_got = run_gpu_commit(cv, w, got, accept_len=accept)
    assert_bits_equal(st_got.cpu(), st_ref, "commit err")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "rebuilt state")


@pytest.mark.parametrize("case", range(30))
def test_recompute_random_sweep(cuda_lib, case):
    """Random shapes: W 2..4, T in {1,2,3,4,8,9,16,17} and beyond, ragged dims, fp32/bf16, bias,
    padded rows, unused slots, and state rows wider than W-1 (the general kernel)."""
    rng = np.random.default_rng(7000 + case)
    over = dict(layout="recompute")
    if case % 3 == 0:
        over.update(n_pad=1, extra_slots=2, n_seq=4)
    if case % 7 == 5:
        over["T"] = int(rng.choice([18, 24, 33]))
    if case % 5 == 4:
        over["state_offset"] = True  # wider rows; the verify reads at the offset
    w = wl.random_case(rng, **over)
    if w.n_pad >= w.n_seq:
        w = w.replace(n_pad=w.n_seq - 1)
    check(cuda_lib, w, wl.make_inputs(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_recompute_every_accept_count(cuda_lib, dtype, width):
    """Every accept count 1..T (the rebuilt window mixes old state columns and x rows for a < W-1
    and is x alone after), plus out-of-range counts 0 and T+1 (flagged, untouched)."""
    T = 9
    w = wl.VerifyWorkload("rc", n_seq=T + 2, T=T, dim=1024 + 40, width=width, qk_channels=512, head_dim=64,
                          dtype=dtype, layout="recompute", bias=True, extra_slots=3, seed=width)
    inp = wl.make_inputs(w)
    acc = torch.tensor(list(range(1, T + 1)) + [0, T + 1], dtype=torch.int32)
    check(cuda_lib, w, inp, accept=acc)


def test_recompute_benchmark_shape_two_steps(cuda_lib):
    """128 x 8 x 10240 bf16, two verify + commit steps in a row, against the oracle's two steps."""
    w = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_recompute_pad13"]
    inp = wl.make_inputs(w)
    ref1 = run_oracle_verify(w, inp)
    run_oracle_commit(w, ref1)
    got = run_gpu_verify(cuda_lib, w, inp)
    run_gpu_commit(cuda_lib, w, got)
    assert_bits_equal(got["conv_state"].cpu(), ref1["conv_state"], "step 1 state")
    nxt = wl.make_inputs(w, seed=w.seed + 5)
    step2 = clone_inputs(inp)
    step2.update(x=nxt["x"], x_base=nxt["x_base"], conv_state=ref1["conv_state"].clone(),
                 accept_len=nxt["accept_len"], out=wl.sentinel_tensor(nxt["out"].shape, w.torch_dtype))
    check(cuda_lib, w, step2)
