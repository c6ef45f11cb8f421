"""GPU parity of the history-row state layout (no window buffer: the state row receives the
deduplicated snapshot row and the next call reads its committed window at accept_len - 1).

State rows and status codes must match the oracle bitwise, outputs within the output tolerance;
columns beyond the row, unused slots and padded sequences' slots keep their sentinels.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_verify
from helpers import assert_bits_equal, assert_out_close, clone_inputs, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _widen(inp: dict, w: wl.VerifyWorkload, extra: int) -> dict:
    """The same inputs with `extra` sentinel columns appended to every state row."""
    r = clone_inputs(inp)
    if extra:
        pad = wl.sentinel_tensor((w.n_slots, w.dim, extra), w.torch_dtype)
        r["conv_state"] = torch.cat([inp["conv_state"], pad], dim=2).contiguous()
    return r


def check(cv, w, inp, path=None):
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cv, w, inp)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state rows")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    if path is not None:
        d = got
        pl = cv.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], None, layout="history",
                            qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                            state_off=d["state_off"])
        assert pl.path == path
    return ref, got


def test_history_benchmark_shape_two_steps(cuda_lib):
    """128 x 8 x 10240 bf16 (13 padded, 16 unused slots), two chained steps: step 2 reads each
    sequence's committed window at accept_len - 1 of step 1, from the rows step 1 wrote."""
    w = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_history_pad13"]
    inp = wl.make_inputs(w)
    ref1, got1 = check(cuda_lib, w, inp, path=3)
    nxt = wl.make_inputs(w, seed=w.seed + 77)
    step2 = clone_inputs(inp)
    step2.update(x=nxt["x"], x_base=nxt["x_base"], conv_state=ref1["conv_state"].clone(),
                 state_off=(inp["accept_len"] - 1).to(torch.int32), out=wl.sentinel_tensor(nxt["out"].shape, w.torch_dtype))
    check(cuda_lib, w, step2, path=3)


@pytest.mark.parametrize("case", range(40))
def test_history_random_sweep(cuda_lib, case):
    """Random shapes in the history layout: W 2..4, T in {1,2,3,4,8,9,16,17} and beyond, ragged
    dims, fp32/bf16, padded rows, offsets, and rows wider than T+W-2 (the general kernel)."""
    rng = np.random.default_rng(5000 + case)
    over = dict(layout="history", state_offset=bool(case % 4 != 3))
    if case % 3 == 0:
        over.update(n_pad=1, extra_slots=2, n_seq=4)
    if case % 7 == 5:
        over["T"] = int(rng.choice([18, 24, 33]))
    w = wl.random_case(rng, **over)
    if w.n_pad >= w.n_seq:
        w = w.replace(n_pad=w.n_seq - 1)
    extra = int(rng.choice([0, 0, 1, 3]))
    check(cuda_lib, w, _widen(wl.make_inputs(w), w, extra))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 5, 8, 17])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_history_packed_paths(cuda_lib, dtype, T, width):
    """Packed [dim][T+W-2] rows take the pipelined kernel (fp32 up to T = 8), every offset in
    0..T-1 appears, and the result equals the oracle's."""
    w = wl.VerifyWorkload("hist", n_seq=2 * T + 1, T=T, dim=1024 + 64, width=width, qk_channels=512, head_dim=64,
                          dtype=dtype, layout="history", bias=True, n_pad=1, extra_slots=3, state_offset=True,
                          seed=100 * T + width)
    inp = wl.make_inputs(w)
    inp["state_off"] = torch.arange(w.n_seq, dtype=torch.int32) % T
    want = 3 if (dtype == "bf16" or T <= 8) else 0
    check(cuda_lib, w, inp, path=want)


def test_history_bad_offsets_flagged(cuda_lib):
    """An offset with offset + W-1 > state_cols (or negative) flags the sequence and touches
    nothing of it; the others are processed."""
    w = wl.VerifyWorkload("hist_bad", n_seq=6, T=4, dim=512, width=4, qk_channels=0, head_dim=8, dtype="bf16",
                          layout="history", state_offset=True, seed=9)
    inp = wl.make_inputs(w)
    inp["state_off"] = torch.tensor([0, 3, 4, -1, 2, 7], dtype=torch.int32)
    ref, got = check(cuda_lib, w, inp, path=3)
    assert ref["status"].tolist() == [0, 0, 2, 2, 0, 2]
