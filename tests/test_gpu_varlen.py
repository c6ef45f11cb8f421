"""GPU parity of the packed ragged verify (sglang PR #46184, "Related upstream work": target verify on
packed ragged tokens, the tile store covering the packed rows) with the CPU oracle, through the C
ABI: outputs within the output tolerance; snapshots, state, commit and status bitwise; every region
a sequence must not touch (snapshot steps and deduplicated columns past its draft count, padded
sequences, rows past the last span, unused slots) keeps its sentinel."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_bits_equal, assert_out_close, clone_inputs
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_oracle(w, inp):
    r = clone_inputs(inp)
    r["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_verify(r["x"], r["conv_state"], r["weight"], r["bias"], r["out"], r["window"], layout=w.layout,
                       qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=r["cache_idx"],
                       state_off=r["state_off"], status=r["status"], cu_draft=r["cu_draft"], T=w.T)
    return r


def oracle_commit(w, r, accept=None):
    st = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_commit(r["conv_state"], r["window"], r["accept_len"] if accept is None else accept, layout=w.layout,
                       T=w.T, width=w.width, cache_idx=r["cache_idx"], status=st,
                       x=r["x"] if w.layout == "recompute" else None, cu_draft=r["cu_draft"],
                       total_tokens=r["x"].shape[0])
    return st


def to_dev(inp, x_shift=0):
    """Copy to the GPU (a transposed window keeps its strides); x_shift > 0 places x that many
    elements past a 16-byte boundary."""
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    if inp.get("window") is not None and not inp["window"].is_contiguous():
        w = inp["window"]
        d["window"] = torch.empty_strided(w.shape, w.stride(), dtype=w.dtype, device="cuda").copy_(w)
    xb = inp["x_base"]
    if x_shift:
        flat = torch.zeros(xb.numel() + x_shift, dtype=xb.dtype, device="cuda")
        flat[x_shift:] = xb.reshape(-1).to("cuda")
        base = flat[x_shift:].view(xb.shape)
    else:
        base = xb.to("cuda")
    x = inp["x"]
    d["x_base"] = base
    # (as_strided takes an offset into the whole storage, which starts x_shift elements earlier)
    d["x"] = base.as_strided(x.shape, x.stride(), base.storage_offset() + x.storage_offset())
    return d


def run_gpu(cv, w, inp, x_shift=0):
    d = to_dev(inp, x_shift)
    d["err"] = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    plan = cv.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                          qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                          state_off=d["state_off"], cu_draft=d["cu_draft"], T=w.T)
    cv.conv_verify(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                   qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                   state_off=d["state_off"], err=d["err"], cu_draft=d["cu_draft"], T=w.T)
    torch.cuda.synchronize()
    return plan.path, d


def gpu_commit(cv, w, d, accept=None):
    e = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    acc = d["accept_len"] if accept is None else accept.to("cuda")
    cv.conv_commit(d["conv_state"], d["window"], acc, layout=w.layout, T=w.T, width=w.width, cache_idx=d["cache_idx"],
                   err=e, x=d["x"] if w.layout == "recompute" else None, cu_draft=d["cu_draft"],
                   total_tokens=d["x"].shape[0])
    torch.cuda.synchronize()
    return e


def check(cv, w, inp, x_shift=0, commit=True, path=None):
    ref = run_oracle(w, inp)
    p, got = run_gpu(cv, w, inp, x_shift)
    if path is not None:
        assert p == path, f"launch path {p}, expected {path}"
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    if inp["window"] is not None:
        assert_bits_equal(got["window"].cpu(), ref["window"], "window")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    if commit and w.layout != "history":
        st_ref = oracle_commit(w, ref)
        st_got = gpu_commit(cv, w, got)
        assert_bits_equal(st_got.cpu(), st_ref, "commit err")
        assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "committed state")
    return ref, got


@pytest.mark.parametrize("name", wl.RAGGED_ORDER)
def test_named_ragged_workloads(cuda_lib, name):
    """The benchmark shape with 128 sequences of 1..16 packed draft tokens (13 padded), dedup rows,
    verify and commit, through the pipelined kernel."""
    w = wl.RAGGED_WORKLOADS[name]
    check(cuda_lib, w, wl.make_ragged_inputs(w), path=3)


@pytest.mark.parametrize("case", range(32))
def test_ragged_random_sweep(cuda_lib, case):
    """Random packed batches: every layout, fp32 / bf16, W 2..4, T up to 17 (pipelined) and past it
    (general), draft counts 0..T, padded sequences, state offsets, head dims, bias, rows past the
    last span, and x off 16-byte alignment (general kernel)."""
    rng = np.random.default_rng(21000 + case)
    layout = ["dense", "dedup", "history", "recompute"][case % 4]
    dtype = "bf16" if case % 3 else "f32"
    T = int(rng.choice([1, 2, 3, 5, 8, 11, 16, 17] if case % 7 else [20, 33]))
    n = int(rng.integers(1, 40))
    lengths = tuple(int(v) for v in rng.integers(0, T + 1, size=n))
    hd = int(rng.choice([16, 32, 64, 128]))
    dim = int(rng.choice([256, 512, 1024, 1536]))
    w = wl.RaggedWorkload(f"rag{case}", lengths=lengths, T=T, dim=dim, width=int(rng.integers(2, 5)),
                          qk_channels=hd * int(rng.integers(0, dim // hd // 2 + 1)), head_dim=hd, dtype=dtype,
                          layout=layout, bias=bool(case % 2), pad=tuple(sorted(set(int(i) for i in rng.integers(0, n, size=n // 5)))),
                          extra_slots=2, state_offset=bool(case % 3 == 2) and layout != "recompute",
                          extra_rows=int(rng.integers(0, 3)), seed=case)
    check(cuda_lib, w, wl.make_ragged_inputs(w), x_shift=1 if case % 5 == 3 else 0)


@pytest.mark.parametrize("layout", ["dense", "dedup"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_pipelined_equals_general_bitwise(cuda_lib, layout, dtype):
    """The same packed batch through the pipelined kernel and (x off alignment) the general kernel:
    the same output bits, and both equal to the oracle."""
    w = wl.RaggedWorkload("rag_paths", lengths=wl.ragged_lengths(5, 60, 0, 8), T=8, dim=2048, width=4,
                          qk_channels=1024, head_dim=128, dtype=dtype, layout=layout, bias=True, pad=(3, 17),
                          extra_slots=4, seed=5)
    inp = wl.make_ragged_inputs(w)
    _, a = check(cuda_lib, w, inp, path=3, commit=False)
    _, b = check(cuda_lib, w, inp, x_shift=1, path=0, commit=False)
    assert_bits_equal(a["out"].cpu(), b["out"].cpu(), "out pipelined vs general")


def test_ragged_equal_lengths_equal_plain_verify(cuda_lib):
    """Every sequence with T drafts, packed: the plain verify's outputs, snapshots and state, bit for bit."""
    T = 8
    w = wl.RaggedWorkload("rag_eq", lengths=(T,) * 50, T=T, dim=4096, width=4, qk_channels=2048, head_dim=128,
                          dtype="bf16", layout="dedup", pad=(7,), extra_slots=3, seed=6)
    inp = wl.make_ragged_inputs(w)
    _, got = run_gpu(cuda_lib, w, inp)
    d = to_dev(inp)
    x3 = d["x"].reshape(w.n_seq, T, w.dim)
    out3 = d["out"].reshape(w.n_seq, T, w.dim)
    cuda_lib.conv_verify(x3, d["conv_state"], d["weight"], d["bias"], out3, d["window"], layout="dedup",
                         qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"])
    torch.cuda.synchronize()
    assert_bits_equal(got["out"].cpu(), d["out"].cpu(), "out")
    assert_bits_equal(got["window"].cpu(), d["window"].cpu(), "window")
    assert_bits_equal(got["conv_state"].cpu(), d["conv_state"].cpu(), "state")


def test_ragged_bad_spans_on_gpu(cuda_lib):
    """A reversed span and one longer than T flag CV_SEQ_BAD_SPAN and leave the sequence untouched,
    in the verify and the commit; an accept count past T_s flags CV_SEQ_BAD_ACCEPT."""
    w = wl.RaggedWorkload("rag_bad", lengths=(2, 2, 2, 2, 2), T=3, dim=1024, width=4, qk_channels=512, head_dim=64,
                          dtype="bf16", layout="dedup", seed=8)
    inp = wl.make_ragged_inputs(w)
    inp["cu_draft"][2] = 1
    inp["accept_len"] = torch.tensor([3, 1, 1, 1, 1], dtype=torch.int32)
    check(cuda_lib, w, inp)


@pytest.mark.parametrize("layout", ["dense", "dedup", "dedupT", "recompute"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [24, 40])
def test_ragged_chunked_on_pipelined_kernel(cuda_lib, layout, dtype, T):
    """Drafts longer than 8 tokens run on the pipelined kernel in 8-token chunks (each later chunk
    reads its first inputs from the x rows before it, chunk 0 writes the committed window from the
    draft's last rows): every layout, both dtypes, draft counts 0..T including exact multiples of
    8, padded sequences, state offsets, against the oracle."""
    rng = np.random.default_rng(23000 + T)
    lengths = tuple(int(v) for v in rng.integers(0, T + 1, size=30)) + (0, 1, 8, 16, T)
    w = wl.RaggedWorkload(f"chunks{T}", lengths=lengths, T=T, dim=1024, width=4, qk_channels=512, head_dim=128,
                          dtype=dtype, layout="dedup" if layout == "dedupT" else layout, bias=True,
                          pad=(2, 11), extra_slots=3, state_offset=layout != "recompute", extra_rows=2,
                          window_transposed=layout == "dedupT", seed=T)
    check(cuda_lib, w, wl.make_ragged_inputs(w), path=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [5, 8, 12])
def test_ragged_column_major_history(cuda_lib, dtype, T):
    """Packed drafts (0..T tokens each) on column-major history rows: the pipelined kernel for
    T <= 8 (a sequence writes columns [0, T_s+W-2) of its row, one bulk copy each; T_s = 0 writes
    nothing), the general kernel beyond (history rows are not chunked)."""
    rng = np.random.default_rng(900 + T)
    n = 41
    lengths = tuple(int(v) for v in rng.integers(0, T + 1, size=n))
    w = wl.RaggedWorkload(f"ragHT{T}", lengths=lengths, T=T, dim=1024, width=4, qk_channels=512, head_dim=128,
                          dtype=dtype, layout="history", bias=True, pad=(3, 17), extra_slots=2, state_offset=True,
                          seed=T)
    inp = wl.make_ragged_inputs(w)
    st = inp["conv_state"]
    cm = torch.empty((st.shape[0], st.shape[2], st.shape[1]), dtype=st.dtype).transpose(1, 2)
    cm.copy_(st)
    inp["conv_state"] = cm
    check(cuda_lib, w, inp, path=3 if T <= 8 else 0)
