"""GPU parity of tree verify (a parent per draft token; dense snapshots): outputs within the output
tolerance, snapshots, state, commit and status bitwise against the oracle; a chain of parents
equals the plain verify bit for bit on the GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import run_gpu_commit, run_gpu_verify, to_device
from helpers import assert_bits_equal, assert_out_close, clone_inputs, run_oracle_commit, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def random_parents(rng, n_seq, T):
    p = np.full((n_seq, T), -1, dtype=np.int32)
    for s in range(n_seq):
        for t in range(1, T):
            p[s, t] = rng.integers(-1, t)  # any earlier token, or the committed window
    return torch.from_numpy(p)


def check(cv, w, inp, accept=None):
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cv, w, inp)
    assert_bits_equal(got["err"].cpu(), ref["status"], "err")
    assert_bits_equal(got["window"].cpu(), ref["window"], "window")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_out_close(got["out"].cpu(), ref["out"], "out")
    st_ref = run_oracle_commit(w, ref, accept_len=accept)
    st_got = run_gpu_commit(cv, w, got, accept_len=accept)
    assert_bits_equal(st_got.cpu(), st_ref, "commit err")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "committed state")


@pytest.mark.parametrize("case", range(16))
def test_tree_random(cuda_lib, case):
    """Random trees: W 2..4, T up to 17 and beyond, ragged dims, head dims, fp32/bf16, bias, padded
    rows, state offsets; the commit restores a random node (accept_len = its index + 1)."""
    rng = np.random.default_rng(13000 + case)
    over = dict(layout="dense", state_offset=bool(case % 3 == 1))
    if case % 4 == 0:
        over.update(n_pad=1, extra_slots=2, n_seq=4)
    if case % 5 == 2:
        over["T"] = int(rng.choice([24, 40]))
    w = wl.random_case(rng, **over)
    if w.n_pad >= w.n_seq:
        w = w.replace(n_pad=w.n_seq - 1)
    inp = wl.make_inputs(w)
    inp["parent"] = random_parents(rng, w.n_seq, w.T)
    check(cuda_lib, w, inp)


def test_tree_bench_shape(cuda_lib):
    """128 sequences of an 8-token tree at dim 10240 bf16 (q|k 4096, head_dim 128)."""
    w = wl.VerifyWorkload("tree", n_seq=128, T=8, dim=10240, width=4, qk_channels=4096, head_dim=128, dtype="bf16",
                          layout="dense", n_pad=13, extra_slots=16, seed=17)
    inp = wl.make_inputs(w)
    inp["parent"] = random_parents(np.random.default_rng(17), w.n_seq, w.T)
    check(cuda_lib, w, inp)


def test_chain_parents_equal_plain_verify_on_gpu(cuda_lib):
    """Parents t-1 through the tree kernel give the plain verify's results bit for bit (the same
    arithmetic as the general kernel)."""
    w = wl.VerifyWorkload("chain", n_seq=6, T=9, dim=1032, width=4, qk_channels=512, head_dim=64, dtype="bf16",
                          layout="dense", bias=True, n_pad=1, extra_slots=1, seed=19)
    inp = wl.make_inputs(w)
    plain = run_gpu_verify(cuda_lib, w, inp)
    tree_in = clone_inputs(inp)
    tree_in["parent"] = torch.arange(-1, w.T - 1, dtype=torch.int32).repeat(w.n_seq, 1).contiguous()
    tree = run_gpu_verify(cuda_lib, w, tree_in)
    for k in ("out", "window", "conv_state", "err"):
        assert_bits_equal(tree[k].cpu(), plain[k].cpu(), k)


def test_tree_invalid_parents_flagged_on_gpu(cuda_lib):
    w = wl.VerifyWorkload("badtree", n_seq=3, T=4, dim=256, width=4, qk_channels=0, head_dim=8, dtype="bf16",
                          layout="dense", seed=23)
    inp = wl.make_inputs(w)
    inp["parent"] = torch.tensor([[-1, 0, 1, 2], [-1, 1, 0, 0], [-2, 0, 0, 0]], dtype=torch.int32)
    ref = run_oracle_verify(w, inp)
    got = run_gpu_verify(cuda_lib, w, inp)
    assert got["err"].cpu().tolist() == [0, 32, 32]
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "state")
    assert_bits_equal(got["window"].cpu(), ref["window"], "window")


@pytest.mark.parametrize("dtype,T,width", [("f32", 128, 4), ("bf16", 100, 3), ("f32", 33, 2)])
def test_tree_long_drafts(cuda_lib, dtype, T, width):
    """Long drafts: the staged rows outgrow the shared-memory budget and the block shrinks (to 32
    threads for 128 fp32 tokens); deep random trees, padded rows, a ragged last channel block."""
    rng = np.random.default_rng(T + width)
    w = wl.VerifyWorkload("treelong", n_seq=3, T=T, dim=1096, width=width, qk_channels=512, head_dim=64,
                          dtype=dtype, layout="dense", bias=True, n_pad=1, extra_slots=2, seed=T)
    inp = wl.make_inputs(w)
    inp["parent"] = random_parents(rng, w.n_seq, w.T)
    check(cuda_lib, w, inp)


def test_tree_root_heavy_and_deep(cuda_lib):
    """Every token a child of the committed window (each window reaches into it), and a single
    deep path, in one batch on the packed-state fast loads."""
    T = 8
    w = wl.VerifyWorkload("treeshape", n_seq=2, T=T, dim=2048, width=4, qk_channels=1024, head_dim=128,
                          dtype="bf16", layout="dense", seed=29)
    inp = wl.make_inputs(w)
    p = torch.full((2, T), -1, dtype=torch.int32)
    p[1] = torch.arange(-1, T - 1, dtype=torch.int32)
    p[1, 4] = 1  # a branch off the path
    inp["parent"] = p
    check(cuda_lib, w, inp)
