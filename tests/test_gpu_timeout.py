"""The bounded-wait failure path of the pipelined verify and the dedup commit, on the GPU, without a
fault: the limit of each unit's first wait for its bulk copies is set so low that the wait runs out
on an ordinary copy (wait_polls < 0: no poll at all; 1: a single poll).  The call must return, flag
CV_SEQ_TIMEOUT on every sequence it did not finish, leave every other sequence exactly as the oracle
computes it, and leave the context usable: the next call with the default limit is exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import to_device
from helpers import assert_bits_equal, assert_out_close, bits, run_oracle_commit, run_oracle_verify
from spec_decode_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W3 = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_dedup_pad13"]


def gpu_verify(cv, w, inp, wait_polls):
    d = to_device(inp)
    d["err"] = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    plan = cv.verify_plan(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                          qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=d["cache_idx"],
                          state_off=d["state_off"])
    assert plan.path == 3, "the bounded waits belong to the pipelined kernel"
    cv.conv_verify(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                   qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                   state_off=d["state_off"], err=d["err"], wait_polls=wait_polls)
    torch.cuda.synchronize()
    return d


def check_unflagged(w, inp, ref, got):
    """Sequences without the timeout bit equal the oracle bitwise (outputs within tolerance);
    padded sequences and unused slots keep their sentinels.  Returns the flagged sequences."""
    err = got["err"].cpu().numpy()
    status = ref["status"].numpy()
    cache = inp["cache_idx"].numpy()
    flagged = [s for s in range(w.n_seq) if err[s] & 8]
    for s in range(w.n_seq):
        if err[s] & 8:
            assert cache[s] >= 0, "a padded sequence was flagged"
            assert (err[s] & ~8) == status[s]
            continue
        assert err[s] == status[s], f"seq {s}: err {err[s]} want {status[s]}"
        if cache[s] < 0:
            assert_bits_equal(got["out"][s].cpu(), ref["out"][s], f"padded out row {s}")
        else:
            assert_out_close(got["out"][s].cpu(), ref["out"][s], f"out row {s}")
        if got.get("window") is not None:
            assert_bits_equal(got["window"][s].cpu(), ref["window"][s], f"window row {s}")
        if cache[s] >= 0:
            assert_bits_equal(got["conv_state"][cache[s]].cpu(), ref["conv_state"][cache[s]], f"state slot {cache[s]}")
    used = set(int(c) for c in cache if c >= 0)
    for slot in range(w.n_slots):
        if slot not in used:
            assert_bits_equal(got["conv_state"][slot].cpu(), inp["conv_state"][slot], f"unused slot {slot}")
    return flagged


@pytest.mark.parametrize("name", ["n128_t8_dim10240_w4_bf16_dedup_pad13", "n128_t8_dim10240_w4_bf16_history_pad13",
                                  "n128_t8_dim10240_w4_bf16_recompute_pad13",
                                  "n128_t8_dim10240_w4_bf16x_f32state_dedup_pad13"])
def test_verify_wait_gives_up_at_once(cuda_lib, name):
    """No poll at all: every block gives up on its first unit, so every active sequence is flagged
    (padded ones are not), the call returns, and the same launch with the default limit then
    matches the oracle exactly."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    ref = run_oracle_verify(w, inp)
    got = gpu_verify(cuda_lib, w, inp, wait_polls=-1)
    err = got["err"].cpu().numpy()
    cache = inp["cache_idx"].numpy()
    for s in range(w.n_seq):
        want = 8 if cache[s] >= 0 else 0
        assert err[s] == want, f"seq {s}: err {err[s]} want {want}"
        if cache[s] < 0:
            assert_bits_equal(got["out"][s].cpu(), inp["out"][s], f"padded out row {s}")
    again = gpu_verify(cuda_lib, w, inp, wait_polls=0)
    assert_bits_equal(again["err"].cpu(), ref["status"], "err")
    assert_bits_equal(again["conv_state"].cpu(), ref["conv_state"], "state")
    if again.get("window") is not None:
        assert_bits_equal(again["window"].cpu(), ref["window"], "window")
    assert_out_close(again["out"].cpu(), ref["out"], "out")


@pytest.mark.parametrize("polls", [1, 2, 4])
def test_verify_short_wait_others_exact(cuda_lib, polls):
    """A limit of a few polls: some units may run out, others not.  Flagged sequences may be
    partly written; every other sequence equals the oracle bitwise."""
    inp = wl.make_inputs(W3, seed=W3.seed + polls)
    ref = run_oracle_verify(W3, inp)
    got = gpu_verify(cuda_lib, W3, inp, wait_polls=polls)
    check_unflagged(W3, inp, ref, got)


def test_commit_wait_gives_up_at_once(cuda_lib):
    """The dedup commit with no poll: every active sequence is flagged and its state keeps the
    verify's committed window; the default limit then commits exactly."""
    w = W3
    inp = wl.make_inputs(w)
    ref = run_oracle_verify(w, inp)
    got = gpu_verify(cuda_lib, w, inp, wait_polls=0)
    before = got["conv_state"].clone()
    e = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    cuda_lib.conv_commit(got["conv_state"], got["window"], got["accept_len"], layout=w.layout, T=w.T, width=w.width,
                         cache_idx=got["cache_idx"], err=e, wait_polls=-1)
    torch.cuda.synchronize()
    cache = inp["cache_idx"].numpy()
    want = np.where(cache >= 0, 8, 0).astype(np.uint32)
    assert np.array_equal(bits(e.cpu()), want)
    assert_bits_equal(got["conv_state"].cpu(), before.cpu(), "state after a commit that gave up")
    st_ref = run_oracle_commit(w, ref)
    e2 = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    cuda_lib.conv_commit(got["conv_state"], got["window"], got["accept_len"], layout=w.layout, T=w.T, width=w.width,
                         cache_idx=got["cache_idx"], err=e2)
    torch.cuda.synchronize()
    assert_bits_equal(e2.cpu(), st_ref, "commit err")
    assert_bits_equal(got["conv_state"].cpu(), ref["conv_state"], "committed state")
