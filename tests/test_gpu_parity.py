"""Parity of the CUDA library (through the C ABI) with the CPU oracle, element by element.

State, snapshots, commit and status codes must match bitwise; outputs within 1e-5 relative (+1e-7
absolute floor) in fp32 and 2 bf16 ulp in bf16.  Every buffer starts filled with a sentinel so
untouched regions (padded sequences, unused slots, state columns past W-1) are compared too.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_commit, run_gpu_verify, to_device
from helpers import assert_bits_equal, assert_out_close, clone_inputs, run_oracle_commit, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def check_verify_and_commit(cv, w: wl.VerifyWorkload, inp: dict, commit=True):
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cv, w, inp)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    if w.layout not in ("history", "recompute"):
        assert_bits_equal(got["window"].cpu(), ref["window"], "window")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    if commit and w.layout != "history":  # the history layout has nothing to commit
        st_ref = run_oracle_commit(w, ref)
        st_got = run_gpu_commit(cv, w, got)
        assert_bits_equal(st_got.cpu(), st_ref, "commit err")
        assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "committed state")
    return ref, got


@pytest.mark.parametrize("name", wl.WORKLOAD_ORDER)
def test_named_workloads(cuda_lib, name):
    """All named workloads at full size, in the launch configuration the bench times."""
    w = wl.WORKLOADS[name]
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


def test_named_workloads_second_seed(cuda_lib):
    for name in wl.WORKLOAD_ORDER[:2] + wl.WORKLOAD_ORDER[3:]:
        w = wl.WORKLOADS[name]
        check_verify_and_commit(cuda_lib, w, wl.make_inputs(w, seed=w.seed + 1000))


@pytest.mark.parametrize("case", range(60))
def test_random_sweep(cuda_lib, case):
    """Random small shapes: W in 2..4, T in {1,2,3,4,8,9,16,17}, ragged dims (not multiples of 8 or
    of the block), head_dim 8..128, fp32/bf16, dense/dedup, bias on/off, padded rows, offsets."""
    rng = np.random.default_rng(1000 + case)
    over = {}
    if case % 3 == 0:
        over["n_pad"] = 1
        over["extra_slots"] = 2
        over["n_seq"] = 4
    if case % 4 == 1:
        over["state_offset"] = True
    w = wl.random_case(rng, **over)
    if w.n_pad >= w.n_seq:
        w = w.replace(n_pad=w.n_seq - 1)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dim", [1, 7, 8, 9, 1023, 1024, 1025, 2048 + 8 + 3])
def test_ragged_dims(cuda_lib, dtype, dim):
    w = wl.VerifyWorkload("ragged", n_seq=3, T=5, dim=dim, width=4, qk_channels=0, head_dim=8, dtype=dtype,
                          layout="dedup", bias=True, n_pad=1, extra_slots=1, seed=dim)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


@pytest.mark.parametrize("hd", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_dims(cuda_lib, hd, dtype):
    w = wl.VerifyWorkload("hd", n_seq=2, T=3, dim=4 * hd + 40, width=4, qk_channels=4 * hd, head_dim=hd,
                          dtype=dtype, layout="dense", bias=True, seed=hd)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


@pytest.mark.parametrize("T", [1, 31, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_long_T(cuda_lib, T, dtype):
    w = wl.VerifyWorkload("longT", n_seq=2, T=T, dim=1000, width=4, qk_channels=512, head_dim=128, dtype=dtype,
                          layout="dedup" if T % 2 else "dense", seed=T)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


def test_unaligned_strided_x(cuda_lib):
    """x as an odd-offset, odd-stride slice (no 16-byte vectors possible): scalar load path."""
    w = wl.VerifyWorkload("xodd", n_seq=3, T=4, dim=300, width=4, qk_channels=256, head_dim=64, dtype="bf16",
                          layout="dense", x_row_stride=301, seed=5)
    inp = wl.make_inputs(w)
    base = inp["x_base"]
    inp["x"] = base.view(-1)[1:].as_strided((3, 4, 300), (4 * 301, 301, 1))
    check_verify_and_commit(cuda_lib, w, inp)


def test_transposed_dedup_row(cuda_lib):
    """The dedup row stored column-major ([n_seq, T+W-2, dim] seen as [n_seq, dim, T+W-2])."""
    for dtype in ["f32", "bf16"]:
        w = wl.VerifyWorkload("tr", n_seq=3, T=8, dim=1200, width=4, qk_channels=512, head_dim=128, dtype=dtype,
                              layout="dedup", bias=True, seed=7)
        inp = wl.make_inputs(w)
        inp["window"] = wl.sentinel_tensor((w.n_seq, w.T + 2, w.dim), w.torch_dtype).transpose(1, 2)
        check_verify_and_commit(cuda_lib, w, inp)


def test_dense_window_permuted(cuda_lib):
    """Dense snapshots with the token axis innermost-but-one: arbitrary strides take the element path."""
    w = wl.VerifyWorkload("perm", n_seq=2, T=5, dim=520, width=3, qk_channels=0, head_dim=8, dtype="bf16",
                          layout="dense", seed=9)
    inp = wl.make_inputs(w)
    inp["window"] = wl.sentinel_tensor((w.n_seq, w.dim, w.width - 1, w.T), w.torch_dtype).permute(0, 3, 1, 2)
    check_verify_and_commit(cuda_lib, w, inp)


def test_sequential_equals_batched_in_T_on_gpu(cuda_lib):
    """P-4 on the GPU: T single-token launches give bit-identical outputs and final state."""
    w = wl.VerifyWorkload("seq", n_seq=3, T=6, dim=1100, width=4, qk_channels=512, head_dim=128, dtype="bf16",
                          layout="dense", bias=True, seed=21)
    inp = wl.make_inputs(w)
    full = run_gpu_verify(cuda_lib, w, inp)
    w1 = w.replace(T=1)
    cur = clone_inputs(inp)
    for t in range(w.T):
        step = dict(cur)
        step["x"] = inp["x"][:, t:t + 1]
        step["out"] = wl.sentinel_tensor((w.n_seq, 1, w.dim), w.torch_dtype)
        step["window"] = wl.sentinel_tensor(wl.window_shape(w1), w.torch_dtype)
        r1 = run_gpu_verify(cuda_lib, w1, step)
        assert_bits_equal(r1["out"][:, 0].cpu(), full["out"][:, t].cpu(), f"out {t}")
        assert_bits_equal(r1["window"][:, 0].cpu(), full["window"][:, t].cpu(), f"snapshot {t}")
        cur["conv_state"] = r1["conv_state"].cpu()
    assert_bits_equal(cur["conv_state"], full["conv_state"].cpu(), "final state")


def test_batched_equals_separate_on_gpu(cuda_lib):
    """P-5 on the GPU: batched launch == one launch per sequence, bitwise."""
    w = wl.VerifyWorkload("bat", n_seq=4, T=8, dim=2100, width=4, qk_channels=1024, head_dim=128, dtype="bf16",
                          layout="dedup", n_pad=1, extra_slots=2, seed=22)
    inp = wl.make_inputs(w)
    full = run_gpu_verify(cuda_lib, w, inp)
    for s in range(w.n_seq):
        ws = w.replace(n_seq=1, n_pad=0)
        one = clone_inputs(inp)
        one["x"] = inp["x"][s:s + 1]
        one["cache_idx"] = inp["cache_idx"][s:s + 1].clone()
        one["out"] = wl.sentinel_tensor((1, w.T, w.dim), w.torch_dtype)
        one["window"] = wl.sentinel_tensor(wl.window_shape(ws), w.torch_dtype)
        r1 = run_gpu_verify(cuda_lib, ws, one)
        assert_bits_equal(r1["out"][0].cpu(), full["out"][s].cpu(), "out")
        assert_bits_equal(r1["window"][0].cpu(), full["window"][s].cpu(), "window")


def test_dedup_equals_dense_on_gpu(cuda_lib):
    """P-6 on the GPU: the dedup row read through its view equals the dense snapshots bitwise."""
    w = wl.VerifyWorkload("dd", n_seq=3, T=9, dim=3000, width=4, qk_channels=1024, head_dim=128, dtype="bf16",
                          layout="dense", seed=23)
    inp = wl.make_inputs(w)
    dense = run_gpu_verify(cuda_lib, w, inp)
    wd = w.replace(layout="dedup")
    inp_d = clone_inputs(inp)
    inp_d["window"] = wl.sentinel_tensor(wl.window_shape(wd), w.torch_dtype)
    dd = run_gpu_verify(cuda_lib, wd, inp_d)
    row = dd["window"]
    view = row.as_strided((w.n_seq, w.T, w.dim, 3), (row.stride(0), row.stride(2), row.stride(1), row.stride(2)))
    assert_bits_equal(view.cpu(), dense["window"].cpu(), "view")
    assert_bits_equal(dd["out"].cpu(), dense["out"].cpu(), "out")


def test_commit_equals_shorter_verify_on_gpu(cuda_lib):
    """P-9 on the GPU: verify(T) + commit(a) state == verify(first a tokens) state, bitwise."""
    w = wl.VerifyWorkload("cm", n_seq=6, T=8, dim=2048, width=4, qk_channels=1024, head_dim=128, dtype="bf16",
                          layout="dedup", n_pad=1, extra_slots=2, seed=24)
    inp = wl.make_inputs(w)
    d = run_gpu_verify(cuda_lib, w, inp)
    assert (run_gpu_commit(cuda_lib, w, d).cpu() == 0).all()
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
        ra = run_gpu_verify(cuda_lib, wa, one)
        assert_bits_equal(d["conv_state"][slot].cpu(), ra["conv_state"][slot].cpu(), f"seq {s}")


def test_status_codes_on_gpu(cuda_lib):
    """Bad slot / offset / accept: flagged per sequence, the sequence untouched, others unaffected."""
    w = wl.VerifyWorkload("bad", n_seq=5, T=4, dim=900, width=4, qk_channels=256, head_dim=64, dtype="bf16",
                          layout="dense", state_offset=True, seed=25)
    inp = wl.make_inputs(w)
    inp["cache_idx"][0] = w.n_slots + 3
    inp["state_off"][1] = w.state_cols - w.width + 2
    inp["state_off"][2] = -4
    inp["cache_idx"][3] = -1
    ref, got = check_verify_and_commit(cuda_lib, w, inp, commit=False)
    assert got["err"].tolist() == [1, 2, 2, 0, 0]
    acc = inp["accept_len"].clone()
    acc[4] = 0
    st_ref = run_oracle_commit(w, ref, accept_len=acc)
    st_got = run_gpu_commit(cuda_lib, w, got, accept_len=acc)
    assert_bits_equal(st_got.cpu(), st_ref, "commit err")
    assert st_got.tolist() == [1, 0, 0, 0, 4]
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")


def test_nan_payload_and_signed_zero_on_gpu(cuda_lib):
    w = wl.VerifyWorkload("nan", n_seq=2, T=3, dim=64, width=4, qk_channels=0, head_dim=8, dtype="bf16",
                          layout="dedup", seed=26)
    inp = wl.make_inputs(w)
    slot = int(inp["cache_idx"][0])
    inp["conv_state"].view(torch.int16)[slot, 3, 1] = 0x7FA1
    inp["conv_state"].view(torch.int16)[slot, 4, 2] = -32768
    inp["x"].view(torch.int16)[0, 1, 5] = 0x7F81
    check_verify_and_commit(cuda_lib, w, inp)


def test_empty_batch_is_noop(cuda_lib):
    w = wl.VerifyWorkload("empty", n_seq=1, T=2, dim=64, width=4, qk_channels=0, head_dim=8, dtype="bf16",
                          layout="dense", seed=27)
    d = to_device(wl.make_inputs(w))
    before = d["conv_state"].clone()
    cuda_lib.conv_verify(d["x"][:0], d["conv_state"], d["weight"], None, d["out"][:0], d["window"][:0],
                         layout="dense", qk_channels=0, head_dim=8)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), d["conv_state"].view(torch.int16))


def test_all_padded_touches_nothing(cuda_lib):
    w = wl.VerifyWorkload("allpad", n_seq=3, T=4, dim=512, width=4, qk_channels=256, head_dim=128, dtype="bf16",
                          layout="dedup", n_pad=3, seed=28)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))


def test_cpu_tensors_rejected(cuda_lib):
    """No CPU path: CPU tensors raise instead of computing."""
    w = wl.WORKLOADS[wl.WORKLOAD_ORDER[0]]
    inp = wl.make_inputs(w)
    with pytest.raises(ValueError):
        cuda_lib.conv_verify(inp["x"], inp["conv_state"], inp["weight"], None, inp["out"], inp["window"],
                             layout="dense", qk_channels=256, head_dim=64)


def _run_with_state_view(cuda_lib, w, inp, state_dev, x_dev):
    d = to_device(inp)
    d["conv_state"] = state_dev
    d["x"] = x_dev
    d["err"] = torch.zeros(w.n_seq, dtype=torch.int32, device="cuda")
    plan = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"],
                                layout=w.layout, qk_channels=w.qk_channels, head_dim=w.head_dim,
                                cache_idx=d["cache_idx"])
    cuda_lib.conv_verify(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                         qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"], err=d["err"])
    torch.cuda.synchronize()
    return plan.path, d


@pytest.mark.parametrize("layout", ["dense", "dedup"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_paths_bit_identical(cuda_lib, layout, dtype):
    """The same inputs through the pipelined kernel (packed state rows, and packed rows one column
    wider, staged whole), the static-T kernel (rows with a gap between them, element stores) and
    the general kernel (x shifted off 16-byte alignment) give bit-identical outputs, snapshots and
    committed windows -- and match the oracle."""
    # 640 sequences x 3 channel blocks: enough units per block (3.2) for the pipelined kernel
    w = wl.VerifyWorkload("paths", n_seq=640, T=6, dim=1536, width=4, qk_channels=512, head_dim=128, dtype=dtype,
                          layout=layout, bias=True, n_pad=7, extra_slots=2, seed=31)
    inp = wl.make_inputs(w)
    ref = run_oracle_verify(w, inp)
    R = w.width - 1
    results = {}
    # packed state
    p3, d3 = _run_with_state_view(cuda_lib, w, inp, inp["conv_state"].cuda(), to_device(inp)["x"])
    # packed rows one column wider: [n_slots, dim, R+1], the window in columns 0..R-1
    wide = wl.sentinel_tensor((w.n_slots, w.dim, R + 1), w.torch_dtype)
    wide[:, :, :R] = inp["conv_state"]
    p3w, d3w = _run_with_state_view(cuda_lib, w, inp, wide.cuda(), to_device(inp)["x"])
    # rows with a gap: a [.., R+1] view of [.., R+2] storage (channel stride R+2)
    gap = wl.sentinel_tensor((w.n_slots, w.dim, R + 2), w.torch_dtype)
    gap[:, :, :R] = inp["conv_state"]
    gap_dev = gap.cuda()
    p1, d1 = _run_with_state_view(cuda_lib, w, inp, gap_dev[:, :, :R + 1], to_device(inp)["x"])
    # x one element off alignment (copy into a buffer shifted by one element)
    xb = torch.zeros(w.n_seq * w.T * w.dim + 1, dtype=w.torch_dtype)
    xb[1:] = inp["x"].reshape(-1)
    x_odd = xb.cuda()[1:].view(w.n_seq, w.T, w.dim)
    p0, d0 = _run_with_state_view(cuda_lib, w, inp, inp["conv_state"].cuda(), x_odd)
    assert (p3, p3w, p1, p0) == (3, 3, 1, 0)
    for name, d in (("pipelined", d3), ("pipelined wide", d3w), ("static", d1), ("general", d0)):
        assert_bits_equal(d["out"].cpu(), d3["out"].cpu(), f"out {name}")
        assert_bits_equal(d["window"].cpu(), ref["window"], f"window {name}")
        assert_out_close(d["out"].cpu(), ref["out"], f"out {name}")
    assert_bits_equal(d3["conv_state"].cpu(), ref["conv_state"], "state pipelined")
    assert_bits_equal(d0["conv_state"].cpu(), ref["conv_state"], "state general")
    assert_bits_equal(d3w["conv_state"][:, :, :R].cpu(), ref["conv_state"], "state pipelined wide")
    assert_bits_equal(d3w["conv_state"][:, :, R:].cpu(), wide[:, :, R:], "state pipelined wide, column past the window")
    assert_bits_equal(d1["conv_state"][:, :, :R].cpu(), ref["conv_state"], "state static")
    assert_bits_equal(gap_dev[:, :, R:].cpu(), gap[:, :, R:], "state static, columns past the window")


@pytest.mark.parametrize("name", ["n128_t8_dim10240_w4_bf16_dedup_pad13", "n64_t8_dim6144_w3_bf16_dense_nol2_stateoff",
                                  "n128_t8_dim10240_w4_bf16_history_pad13",
                                  "n128_t8_dim10240_w4_bf16_recompute_pad13"])
def test_chained_steps_without_host_sync(cuda_lib, name):
    """Three decode steps queued back to back on one stream with no host synchronisation between
    the launches (each launch may be scheduled while the previous grid finishes): every step's
    outputs and the final state equal the oracle's three steps, so each kernel still sees all the
    previous kernel's writes (state rows, snapshots) and none of its reads are overtaken."""
    import spec_decode_verify_gb300 as cv
    w = wl.WORKLOADS[name]
    steps = [wl.make_inputs(w, seed=w.seed + 31 * i) for i in range(3)]
    base = steps[0]
    hist = w.layout == "history"
    # oracle chain
    ref = clone_inputs(base)
    outs_ref = []
    for i, si in enumerate(steps):
        ref.update(x=si["x"], x_base=si["x_base"], out=wl.sentinel_tensor(si["out"].shape, w.torch_dtype))
        if i > 0 and hist:
            ref["state_off"] = (steps[i - 1]["accept_len"] - 1).to(torch.int32)
        ref = run_oracle_verify(w, ref)
        if not hist:
            run_oracle_commit(w, ref, accept_len=si["accept_len"])
        outs_ref.append(ref["out"].clone())
    # GPU chain: every input staged on the device first, then all launches without a sync
    dev = torch.device("cuda")
    state = base["conv_state"].to(dev)
    weight, bias = base["weight"].to(dev), (base["bias"].to(dev) if base["bias"] is not None else None)
    cidx = base["cache_idx"].to(dev)
    xs = [si["x_base"].to(dev).as_strided(si["x"].shape, si["x"].stride(), si["x"].storage_offset()) for si in steps]
    accs = [si["accept_len"].to(dev) for si in steps]
    offs = [base["state_off"].to(dev) if base["state_off"] is not None else None]
    offs += [(steps[i - 1]["accept_len"] - 1).to(torch.int32).to(dev) if hist else offs[0] for i in (1, 2)]
    outs = [base["out"].to(dev) for _ in steps]
    win = base["window"].to(dev) if base["window"] is not None else None
    torch.cuda.synchronize()
    for i in range(3):
        cv.conv_verify(xs[i], state, weight, bias, outs[i], win, layout=w.layout, qk_channels=w.qk_channels,
                       head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=cidx, state_off=offs[i])
        if not hist:
            cv.conv_commit(state, win, accs[i], layout=w.layout, T=w.T, width=w.width, cache_idx=cidx,
                           x=xs[i] if w.layout == "recompute" else None)
    torch.cuda.synchronize()
    for i in range(3):
        assert_out_close(outs[i].cpu(), outs_ref[i], f"step {i} out")
    assert_bits_equal(state.cpu(), ref["conv_state"], "state after three steps")


@pytest.mark.parametrize("layout", ["dense", "dedup", "recompute"])
@pytest.mark.parametrize("T,width", [(1, 2), (3, 3), (8, 4), (12, 3), (17, 4)])
def test_wide_state_rows_pipelined(cuda_lib, layout, T, width):
    """Packed state rows wider than the window (read at a per-sequence offset) take the pipelined
    kernel when every block walks several units: it stages the rows whole and stores the committed
    window into their first W-1 columns directly; every offset 0..T-1 appears and the result equals
    the oracle's."""
    w = wl.VerifyWorkload("wide", n_seq=300 + T, T=T, dim=4096 + 512, width=width, qk_channels=1024, head_dim=128,
                          dtype="bf16", layout=layout, bias=True, n_pad=1, extra_slots=3, state_offset=True,
                          seed=50 * T + width)
    inp = wl.make_inputs(w)
    inp["state_off"] = (torch.arange(w.n_seq, dtype=torch.int32) % T).contiguous()
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    pl = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=layout,
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path == 3
    check_verify_and_commit(cuda_lib, w, inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout,T,width", [("dense", 3, 2), ("dense", 8, 3), ("dedup", 4, 4), ("dedup", 8, 4),
                                            ("dense", 17, 3), ("dense", 24, 4)])
def test_wide_state_rows_one_pass(cuda_lib, dtype, layout, T, width):
    """Packed state rows wider than the window on the one-pass kernel (a small batch): each block
    stages its rows whole and stores them back whole, with the committed window over the first W-1
    columns; every offset 0..T-1 appears, dim 1000 leaves a partial last block, and the columns
    past the window must come back with their own bits (compared bitwise, like everything else)."""
    w = wl.VerifyWorkload("wide1", n_seq=6, T=T, dim=1000, width=width, qk_channels=512, head_dim=128,
                          dtype=dtype, layout=layout, bias=True, n_pad=1, extra_slots=2, state_offset=True,
                          seed=70 * T + width)
    inp = wl.make_inputs(w)
    inp["state_off"] = (torch.arange(w.n_seq, dtype=torch.int32) % T).contiguous()
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    pl = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=layout,
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path in (1, 2)
    check_verify_and_commit(cuda_lib, w, inp)


@pytest.mark.parametrize("layout,T", [("dense", 8), ("dedup", 5), ("dense", 20)])
def test_wide_state_rows_unaligned(cuda_lib, layout, T):
    """Wide state rows whose base is not 16-byte aligned cannot be staged by 16-byte copies: the
    one-pass kernel reads and writes them element by element instead, with the same results."""
    w = wl.VerifyWorkload("wideu", n_seq=5, T=T, dim=1000, width=4, qk_channels=512, head_dim=128, dtype="bf16",
                          layout=layout, bias=True, n_pad=1, extra_slots=2, state_offset=True, seed=90 + T)
    inp = wl.make_inputs(w)
    inp["state_off"] = (torch.arange(w.n_seq, dtype=torch.int32) % T).contiguous()
    ref = run_oracle_verify(w, inp)
    d = to_device(inp)
    st = d["conv_state"]
    buf = torch.empty(st.numel() + 8, dtype=st.dtype, device="cuda")
    d["conv_state"] = buf[1:1 + st.numel()].view(st.shape)  # 2 bytes past a 16-byte boundary
    d["conv_state"].copy_(st)
    err = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    pl = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=layout,
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path in (1, 2)
    cuda_lib.conv_verify(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=layout,
                         qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                         state_off=d["state_off"], err=err)
    torch.cuda.synchronize()
    assert_bits_equal(err.cpu(), ref["status"], "err")
    assert_bits_equal(d["window"].cpu(), ref["window"], "window")
    assert_bits_equal(d["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(d["out"].cpu(), ref["out"], "out")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,width", [(5, 4), (6, 3), (9, 2), (17, 4), (24, 4), (40, 3), (128, 4)])
@pytest.mark.parametrize("offset", [False, True])
def test_token_groups_one_pass(cuda_lib, dtype, T, width, offset):
    """Small dense batches on the chunked one-pass kernel with the draft tokens split among thread
    groups: a later group starts from the x rows before its first token, only the group holding
    token T-1 writes the state; wide rows read at per-sequence offsets, padded rows, a partial last
    channel block, L2 groups of 64 channels."""
    w = wl.VerifyWorkload("tgroups", n_seq=3, T=T, dim=1000, width=width, qk_channels=512, head_dim=64,
                          dtype=dtype, layout="dense", bias=True, n_pad=1, extra_slots=2, state_offset=offset,
                          seed=7 * T + width + (100 if offset else 0))
    inp = wl.make_inputs(w)
    if offset:
        inp["state_off"] = (torch.arange(w.n_seq, dtype=torch.int32) % T).contiguous()
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    pl = cuda_lib.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout="dense",
                              qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                              state_off=d["state_off"])
    assert pl.path == 2 and pl.token_groups > 1
    check_verify_and_commit(cuda_lib, w, inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width", [2, 3, 4])
@pytest.mark.parametrize("T,dim", [(2, 8), (3, 520), (8, 1000), (17, 264), (128, 256)])
def test_commit_wide_rows(cuda_lib, dtype, width, T, dim):
    """Dense snapshots committed into packed state rows wider than the window (the rows a verify
    reads at a state offset): the rows are staged whole and written back whole, so besides the new
    window in the first W-1 columns every other column must keep its bits.  Partial last channel
    blocks, padded sequences, a pool of unused slots, every accept count; rows of up to 130 fp32
    columns."""
    w = wl.VerifyWorkload("widecommit", n_seq=6, T=T, dim=dim, width=width, qk_channels=0, head_dim=8, dtype=dtype,
                          layout="dense", bias=True, n_pad=1, extra_slots=3, state_offset=True,
                          seed=1000 * width + 10 * T + dim)
    inp = wl.make_inputs(w)
    inp["accept_len"] = (torch.arange(w.n_seq, dtype=torch.int32) % T + 1).contiguous()
    inp["state_off"] = (inp["accept_len"] - 1).contiguous()
    check_verify_and_commit(cuda_lib, w, inp)


def test_maximum_batch_on_gpu(cuda_lib):
    """The largest batch the ABI accepts (65535 sequences; the pipelined kernel then walks every
    sequence without a shared-memory list), with padded sequences and a pool of unused slots."""
    w = wl.VerifyWorkload("maxbatch", n_seq=65535, T=3, dim=64, width=4, qk_channels=32, head_dim=16, dtype="bf16",
                          layout="dedup", bias=True, n_pad=1000, extra_slots=100, seed=65535)
    check_verify_and_commit(cuda_lib, w, wl.make_inputs(w))
