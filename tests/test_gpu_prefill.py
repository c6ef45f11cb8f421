"""GPU parity of the packed variable-length prefill with the CPU oracle (through the C ABI).

State and status codes bitwise, outputs within the output tolerance; untouched rows and slots keep
their sentinels.  The prefill also equals the GPU verify over the same tokens bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import assert_bits_equal, assert_out_close
from spec_decode_verify_gb300 import workloads as wl
import oracle

pytestmark = pytest.mark.gpu


def run_oracle(w, inp):
    r = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    r["x"] = inp["x"]
    r["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_prefill(r["x"], r["conv_state"], r["weight"], r["bias"], r["out"], r["cu_seqlens"],
                        qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=r["cache_idx"],
                        has_initial_state=r["has_initial_state"], status=r["status"])
    return r


def run_gpu(cv, w, inp, max_seqlen=None):
    d = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    base = inp["x_base"].to("cuda")
    d["x"] = base.as_strided(inp["x"].shape, inp["x"].stride(), inp["x"].storage_offset())
    d["err"] = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    cv.conv_prefill(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["cu_seqlens"],
                    max_seqlen=w.max_seqlen if max_seqlen is None else max_seqlen, qk_channels=w.qk_channels,
                    head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                    has_initial_state=d["has_initial_state"], err=d["err"])
    torch.cuda.synchronize()
    return d


def check(cv, w, inp, max_seqlen=None):
    ref = run_oracle(w, inp)
    got = run_gpu(cv, w, inp, max_seqlen)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    return ref, got


@pytest.mark.parametrize("name", wl.PREFILL_ORDER)
def test_named_prefill_workloads(cuda_lib, name):
    """Both named prefill workloads at full size (the large one: 8 prompts, 30k tokens, dim 10240)."""
    w = wl.PREFILL_WORKLOADS[name]
    check(cuda_lib, w, wl.make_prefill_inputs(w))


@pytest.mark.parametrize("case", range(24))
def test_prefill_random_sweep(cuda_lib, case):
    """Random batches: W 2..4, fp32/bf16, head_dim 8..256, ragged dims, lengths around the chunk
    boundaries (0, 1, 127, 128, 129, 255, 256, 257, ...), padded sequences, missing initial states,
    x rows with an odd stride or an odd dim (the register path) and aligned rows (the shared-memory
    ring, 8-, 16- and 32-byte pieces per thread and row)."""
    rng = np.random.default_rng(9000 + case)
    W = int(rng.integers(2, 5))
    hd = int(rng.choice([8, 16, 32, 64, 128, 256]))
    groups = int(rng.integers(0, 4))
    dim = groups * hd + int(rng.integers(1, 300)) if case % 2 else groups * hd + 8 * int(rng.integers(1, 40))
    n = int(rng.integers(1, 6))
    lengths = tuple(int(rng.choice([0, 1, 2, 7, 127, 128, 129, 255, 256, 257, 300, 513, 1000])) for _ in range(n))
    pad = tuple(i for i in range(n) if rng.random() < 0.2)
    no_init = tuple(i for i in range(n) if rng.random() < 0.4)
    w = wl.PrefillWorkload("rand", lengths=lengths, dim=dim, width=W, qk_channels=groups * hd, head_dim=hd,
                           dtype=str(rng.choice(["f32", "bf16"])), bias=bool(rng.integers(0, 2)), pad=pad,
                           no_init=no_init, extra_slots=int(rng.integers(0, 3)),
                           x_row_stride=(dim + 3 if case % 5 == 4 else None), seed=case)
    check(cuda_lib, w, wl.make_prefill_inputs(w))


@pytest.mark.parametrize("dtype,hd", [("bf16", 128), ("bf16", 256), ("f32", 128), ("f32", 256)])
def test_prefill_ring_pieces(cuda_lib, dtype, hd):
    """Aligned rows take the shared-memory ring of staged x rows: each thread's piece of a row is 8
    bytes (bf16, 4 channels), 16 (bf16, 8 channels for a 256-channel group; fp32, 4 channels) or
    32 (fp32, 8 channels).  Lengths end inside, at and just past the 128-token chunks, with prompts
    without a state, a padded prompt and a partly filled channel block."""
    dim = 2 * hd + 8 * 9
    w = wl.PrefillWorkload("ring", lengths=(1, 128, 129, 300, 1000, 7), dim=dim, width=4, qk_channels=2 * hd,
                           head_dim=hd, dtype=dtype, bias=True, pad=(5,), no_init=(0, 3), extra_slots=2,
                           seed=hd + (1 if dtype == "f32" else 0))
    check(cuda_lib, w, wl.make_prefill_inputs(w))


def test_prefill_bad_spans_and_short_max_seqlen(cuda_lib):
    """Reversed or out-of-range spans, and a span longer than max_seqlen, are flagged (16) and
    touch nothing; the other sequences are processed."""
    w = wl.PrefillWorkload("bad", lengths=(300, 40, 50, 600), dim=512, width=4, qk_channels=256, head_dim=64,
                           dtype="bf16", seed=5)
    inp = wl.make_prefill_inputs(w)
    inp["cu_seqlens"] = torch.tensor([0, 300, 250, 2000, 990], dtype=torch.int32)
    ref, got = check(cuda_lib, w, inp, max_seqlen=600)
    assert ref["status"].tolist() == [0, 16, 16, 16]
    # max_seqlen 400: the 600-token prompt is flagged and untouched, which the oracle reproduces
    # with that sequence padded (the oracle has no max_seqlen)
    inp = wl.make_prefill_inputs(w)
    got = run_gpu(cuda_lib, w, inp, max_seqlen=400)
    assert got["err"].cpu().tolist() == [0, 0, 0, 16]
    padded = dict(inp)
    padded["cache_idx"] = inp["cache_idx"].clone()
    padded["cache_idx"][3] = -1
    ref = run_oracle(w, padded)
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_equals_gpu_verify_bitwise(cuda_lib, dtype):
    """A prompt of T tokens with an initial state gives, on the GPU, the outputs and final state of
    a verify over the same T tokens (dense window), bit for bit, in both dtypes (the fp32 conv rounds
    every product, the bf16 one fuses exact products)."""
    import spec_decode_verify_gb300 as cv
    T = 17 if dtype == "bf16" else 8
    w = wl.PrefillWorkload("pv", lengths=(T, T, T), dim=4096, width=4, qk_channels=2048, head_dim=128,
                           dtype=dtype, bias=True, seed=11)
    inp = wl.make_prefill_inputs(w)
    got = run_gpu(cuda_lib, w, inp)
    dev = torch.device("cuda")
    xv = inp["x"].reshape(3, T, w.dim).to(dev)
    st = inp["conv_state"].to(dev)
    out = torch.empty(3, T, w.dim, dtype=w.torch_dtype, device=dev)
    win = torch.empty(3, T, w.dim, w.width - 1, dtype=w.torch_dtype, device=dev)
    cv.conv_verify(xv, st, inp["weight"].to(dev), inp["bias"].to(dev), out, win, layout="dense",
                   qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=inp["cache_idx"].to(dev))
    torch.cuda.synchronize()
    assert_bits_equal(got["out"].cpu(), out.reshape(3 * T, w.dim).cpu(), "out")
    assert_bits_equal(got["conv_state"].cpu(), st.cpu(), "state")
