"""GPU parity of the history-row state layout (no window buffer: the state row receives the
deduplicated snapshot row and the next call reads its committed window at accept_len - 1).

State rows and status codes must match the oracle bitwise, outputs within the output tolerance;
columns beyond the row, unused slots and padded sequences' slots keep their sentinels.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_verify, to_device
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


# ---------------------------------------------------------------- column-major state rows

def _col_major(t: torch.Tensor) -> torch.Tensor:
    """The same [n_slots, dim, S] values stored column by column ([n_slots, S, dim] seen transposed)."""
    c = torch.empty((t.shape[0], t.shape[2], t.shape[1]), dtype=t.dtype).transpose(1, 2)
    c.copy_(t)
    return c


def test_history_column_major_benchmark_two_steps(cuda_lib):
    """The commit-free step with column-major rows at 128 x 8 x 10240 bf16 (13 padded, 16 unused
    slots), two chained steps (step 2 reads each window at accept_len - 1 of step 1's rows); the
    state rows compare as values, whatever their storage order."""
    w = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_historyT_pad13"]
    inp = wl.make_inputs(w)
    assert inp["conv_state"].stride(1) == 1 and inp["conv_state"].stride(2) == w.dim
    ref1, got1 = check(cuda_lib, w, inp, path=3)
    assert got1["conv_state"].stride(1) == 1
    nxt = wl.make_inputs(w, seed=w.seed + 77)
    step2 = clone_inputs(inp)
    step2.update(x=nxt["x"], x_base=nxt["x_base"], conv_state=_col_major(ref1["conv_state"]),
                 state_off=(inp["accept_len"] - 1).to(torch.int32), out=wl.sentinel_tensor(nxt["out"].shape, w.torch_dtype))
    check(cuda_lib, w, step2, path=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 5, 8, 17])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_history_column_major_paths(cuda_lib, dtype, T, width):
    """Column-major rows with 16-byte-aligned columns take the pipelined kernel (W-1 columns
    staged, T+W-2 stored, one bulk copy each; fp32 up to T = 8, else the general kernel); every
    offset 0..T-1 appears; two columns past the row must keep their sentinels."""
    w = wl.VerifyWorkload("histT", n_seq=2 * T + 1, T=T, dim=1024 + 64, width=width, qk_channels=512, head_dim=64,
                          dtype=dtype, layout="history", bias=True, n_pad=1, extra_slots=3, state_offset=True,
                          seed=300 * T + width)
    inp = _widen(wl.make_inputs(w), w, 2)
    inp["conv_state"] = _col_major(inp["conv_state"])
    inp["state_off"] = torch.arange(w.n_seq, dtype=torch.int32) % T
    want = 3 if (dtype == "bf16" or T <= 8) else 0
    check(cuda_lib, w, inp, path=want)


@pytest.mark.parametrize("case", ["odd_dim", "f32_state", "bad_offsets"])
def test_history_column_major_cases(cuda_lib, case):
    """Column-major rows with a channel count that is not a multiple of 8 take the general kernel;
    fp32 state rows under bf16 x (mixed dtypes) stay pipelined; bad offsets flag their sequences
    and leave them untouched."""
    dim = 1001 if case == "odd_dim" else 1024
    w = wl.VerifyWorkload("histTc", n_seq=7, T=6, dim=dim, width=4, qk_channels=512, head_dim=128, dtype="bf16",
                          layout="history", bias=True, n_pad=1, extra_slots=2, state_offset=True,
                          state_dtype="f32" if case == "f32_state" else None, state_transposed=True, seed=len(case))
    inp = wl.make_inputs(w)
    if case == "bad_offsets":
        inp["state_off"] = torch.tensor([0, 5, 6, -1, 2, 9, 1], dtype=torch.int32)
    ref, got = check(cuda_lib, w, inp, path={"odd_dim": 0, "f32_state": 3, "bad_offsets": 3}[case])
    if case == "bad_offsets":
        bad = [o < 0 or o + 3 > w.state_cols for o in inp["state_off"].tolist()]
        live = [c >= 0 for c in inp["cache_idx"].tolist()]
        assert [v != 0 for v in ref["status"].tolist()] == [b and l for b, l in zip(bad, live)]
        assert sum(b and l for b, l in zip(bad, live)) >= 2


def test_history_column_major_unaligned_column_stride(cuda_lib):
    """Columns dim + 1 elements apart (not a 16-byte multiple: no bulk copies) take the general
    kernel; the unused element after each column keeps its sentinel."""
    w = wl.VerifyWorkload("histTs", n_seq=5, T=4, dim=512, width=4, qk_channels=256, head_dim=128, dtype="bf16",
                          layout="history", bias=True, n_pad=1, extra_slots=1, state_offset=True, seed=44)
    inp = wl.make_inputs(w)
    ref = run_oracle_verify(w, inp)
    d = to_device(inp)
    S = w.state_cols
    buf = wl.sentinel_tensor((w.n_slots, S, w.dim + 1), w.torch_dtype).to("cuda")
    st = buf[:, :, : w.dim].transpose(1, 2)
    st.copy_(d["conv_state"])
    d["err"] = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    pl = cuda_lib.verify_plan(d["x"], st, d["weight"], d["bias"], d["out"], None, layout="history",
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path == 0
    cuda_lib.conv_verify(d["x"], st, d["weight"], d["bias"], d["out"], None, layout="history",
                         qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                         state_off=d["state_off"], err=d["err"])
    torch.cuda.synchronize()
    assert_bits_equal(d["err"].cpu(), ref["status"], "err")
    assert_bits_equal(st.cpu(), ref["conv_state"], "state rows")
    assert_bits_equal(buf[:, :, w.dim].cpu(), wl.sentinel_tensor((w.n_slots, S), w.torch_dtype), "gap elements")
    assert_out_close(d["out"].cpu(), ref["out"], "out")
