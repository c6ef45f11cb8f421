"""Host-side checks of the C ABI (no GPU): the library loads, exports every function the header
declares, and rejects invalid arguments with the documented status before launching anything."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

import spec_decode_verify_gb300 as cv
from spec_decode_verify_gb300 import build as cvbuild
from spec_decode_verify_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "convverify.h")


@pytest.fixture(scope="module")
def lib():
    cvbuild.build()
    return cv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^CV_API\s[\w\s\*]*?\b(cv_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"cv_conv_verify", "cv_conv_commit", "cv_verify_plan", "cv_status_string", "cv_abi_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"
    version = int(re.search(r"#define CV_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.cv_abi_version() == version


def test_exports_nothing_undeclared(lib):
    """Only the declared C entry points are visible (the kernels and helpers are hidden)."""
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", cv.library_path], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm not available")
    exported = {ln.split()[-1] for ln in r.stdout.splitlines() if " T " in ln}
    ours = {n for n in exported if n.startswith("cv_")}
    assert ours == set(declared_functions())


def _args(w: wl.VerifyWorkload, **over):
    inp = wl.make_inputs(w)
    a = cv.make_verify_args(inp["x"], inp["conv_state"], inp["weight"], inp["bias"], inp["out"], inp["window"],
                            layout=w.layout, qk_channels=w.qk_channels, head_dim=w.head_dim,
                            cache_idx=inp["cache_idx"], parent=inp.get("parent"), check_device=False)
    _args.keep = inp  # the struct holds raw pointers into these tensors
    for k, v in over.items():
        setattr(a, k, v)
    return a


def _plan(lib, a):
    pl = cv.LaunchPlan()
    return lib.cv_verify_plan(ctypes.byref(a), ctypes.byref(pl)), pl


W3 = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_dedup_pad13"]


def _pipe_smem(stage, image, n_seq, varlen_T=None):
    """The pipelined kernel's shared memory: two stages, two image buffers, 48 bytes of barriers and
    unit information (slots, offsets, draft counts, first rows), then the listing scratch (4 warp
    counts; for packed drafts 5 * (TS + 2) sort counts, TS = min(T, 8) tokens per unit) and the list:
    12 bytes per sequence (its index, cache slot and state offset), or for packed drafts 4 bytes per
    chunk of TS tokens."""
    if varlen_T is None:
        return 2 * stage + 2 * image + 48 + 4 * 4 + 12 * n_seq
    ts = min(varlen_T, 8)
    return 2 * stage + 2 * image + 48 + 4 * 5 * (ts + 2) + 4 * n_seq * ((varlen_T + ts - 1) // ts)


def test_plan_for_benchmark_workload(lib):
    """128 x 8 x 10240 bf16 dedup, packed state: the pipelined path.  4 channels per thread (an L2
    group of 128 spans 32 lanes), 128 threads per unit of 512 channels.  Shared memory: two stages
    of (8 x rows + 3 window columns) and two image buffers of (10 dedup columns + 3 window columns),
    plus barriers, slots, offsets and the list of active sequences; 4 blocks fit an SM, and the
    persistent grid is the largest multiple of the 20 channel blocks within 152 * 4 blocks, so each
    block keeps its taps."""
    rc, pl = _plan(lib, _args(W3))
    assert rc == 0
    smem = _pipe_smem((8 + 3) * 512 * 2, (10 + 3) * 512 * 2, 128)
    assert (pl.threads, pl.channels_per_block, pl.path, pl.smem_bytes, pl.stages) == (128, 512, 3, smem, 2)
    assert (pl.grid_x, pl.grid_y) == (600, 1)


HIST = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_history_pad13"]


def test_plan_for_history_workload(lib):
    """History rows: the stages hold whole [10]-column rows and the only image is the row image,
    so one block needs 2 * (8 + 10) * 1024 + 2 * 10 * 1024 bytes plus the index words and 3 blocks
    fit an SM; the grid is the largest multiple of 20 within 152 * 3."""
    a = _args(HIST)
    assert a.window is None and a.state_cols == 10 and a.state_ch_stride == 10
    rc, pl = _plan(lib, a)
    assert rc == 0
    smem = _pipe_smem((8 + 10) * 512 * 2, 10 * 512 * 2, 128)
    assert (pl.threads, pl.channels_per_block, pl.path, pl.smem_bytes, pl.stages) == (128, 512, 3, smem, 2)
    assert (pl.grid_x, pl.grid_y) == (440, 1)


HISTT = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_historyT_pad13"]


def test_plan_for_column_major_history(lib):
    """Column-major history rows: the stages hold 8 x rows and only the W-1 = 3 staged columns of
    the state, the image the 10-column row (stored column by column); 4 blocks fit an SM."""
    a = _args(HISTT)
    assert (a.state_ch_stride, a.state_col_stride, a.state_slot_stride) == (1, 10240, 10 * 10240)
    rc, pl = _plan(lib, a)
    assert rc == 0
    smem = _pipe_smem((8 + 3) * 512 * 2, 10 * 512 * 2, 128)
    assert (pl.threads, pl.channels_per_block, pl.path, pl.smem_bytes, pl.stages) == (128, 512, 3, smem, 2)
    assert (pl.grid_x, pl.grid_y) == (600, 1)
    # rows wider than T+W-2 stay pipelined (only W-1 columns are staged)
    b = _args(HISTT.replace(n_seq=64, n_pad=0, extra_slots=0))
    b.state_cols = 12
    b.state_slot_stride = 12 * 10240
    assert _plan(lib, b)[1].path == 3


def test_column_major_state_validation(lib):
    """A column stride other than 0/1 needs the history layout (else CV_ERR_LAYOUT), a channel
    stride of 1 and a column stride of at least dim (else CV_ERR_STRIDE); negative is
    CV_ERR_STRIDE; column strides that are not 16-byte multiples, or dims that are not multiples
    of 8, take the general kernel."""
    a = _args(HISTT)
    a.state_col_stride = -1
    assert _plan(lib, a)[0] == -9
    a = _args(HISTT)
    a.state_col_stride = 10239
    assert _plan(lib, a)[0] == -9
    a = _args(HISTT)
    a.state_ch_stride = 2
    a.state_col_stride = 2 * 10240
    assert _plan(lib, a)[0] == -9
    a = _args(HISTT)
    a.state_col_stride = 10248  # a 16-byte multiple (bf16): still pipelined
    a.state_slot_stride = 10 * 10248
    assert _plan(lib, a)[1].path == 3
    a.state_col_stride = 10241
    a.state_slot_stride = 10 * 10241
    assert _plan(lib, a)[1].path == 0
    w = W3.replace(n_seq=4, n_pad=0, extra_slots=0)
    a = _args(w)
    a.state_ch_stride, a.state_col_stride = 1, w.dim
    assert _plan(lib, a)[0] == -8
    a = _args(HISTT.replace(dim=10232, qk_channels=4096, n_seq=8, n_pad=0, extra_slots=0))
    assert _plan(lib, a)[1].path == 3
    a = _args(HISTT.replace(dim=10236, qk_channels=4096, n_seq=8, n_pad=0, extra_slots=0))
    assert _plan(lib, a)[1].path == 0


def test_history_validation_and_paths(lib):
    # rows narrower than T+W-2 are rejected
    a = _args(HIST)
    a.state_cols = 9
    assert _plan(lib, a)[0] == -3
    # wider rows (not the packed row) take the general kernel
    a = _args(HIST)
    a.state_cols, a.state_ch_stride = 11, 11
    assert _plan(lib, a)[1].path == 0
    # the history layout ignores the window strides; commit rejects the layout
    a = _args(HIST)
    a.win_seq_stride = -5
    assert _plan(lib, a)[0] == 0
    inp = wl.make_inputs(HIST.replace(n_seq=2, n_pad=0, extra_slots=0))
    c = cv.make_commit_args(inp["conv_state"], None, inp["accept_len"], layout="history", T=8, width=4,
                            check_device=False)
    assert lib.cv_conv_commit(ctypes.byref(c), None) == -8
    # long T: the general kernel
    assert _plan(lib, _args(HIST.replace(T=18)))[1].path == 0
    assert _plan(lib, _args(HIST.replace(T=8, dtype="f32")))[1].path == 3


@pytest.mark.parametrize("name,path", [
    ("n1_t2_dim512_w4_f32_dense", 1), ("n4_t4_dim4096_w4_bf16_dedup_bias", 1),
    ("n8_t17_dim8192_w4_bf16_dense_qkvsplit_xstride12288", 2), ("n64_t8_dim6144_w3_bf16_dense_nol2_stateoff", 1),
    ("n128_t8_dim10240_w4_bf16_history_pad13", 3), ("n128_t8_dim10240_w4_bf16_recompute_pad13", 3),
    ("n128_t8_dim10240_w4_bf16_tree_dense_pad13", 5), ("n128_t8_dim10240_w4_bf16x_f32state_dedup_pad13", 3)])
def test_plan_paths_of_named_workloads(lib, name, path):
    w = wl.WORKLOADS[name]
    rc, pl = _plan(lib, _args(w))
    assert rc == 0 and pl.path == path
    units = w.n_seq * -(-w.dim // pl.channels_per_block)
    if path in (3, 5):  # persistent grids
        assert pl.grid_y == 1 and 1 <= pl.grid_x <= units
    else:
        assert pl.grid_y == w.n_seq and pl.grid_x * pl.channels_per_block >= w.dim
    # small batches are split into at least two units per SM where the L2 groups allow it
    assert units >= 2 * 152 or pl.threads == 32 or pl.channels_per_block // 2 < max(w.head_dim, 8)


def test_recompute_plan_and_commit_validation(lib):
    """Recompute layout: the stages hold x rows and committed windows and there are no images;
    its commit needs x and no window."""
    w = wl.WORKLOADS["n128_t8_dim10240_w4_bf16_recompute_pad13"]
    a = _args(w)
    assert a.window is None
    rc, pl = _plan(lib, a)
    assert rc == 0 and pl.path == 3 and pl.smem_bytes == _pipe_smem((8 + 3) * 512 * 2, 0, 128)
    a.state_ch_stride, a.state_cols = 4, 4  # wider packed rows: still pipelined (staged whole)
    assert _plan(lib, a)[1].path == 3
    a.state_ch_stride = 6  # rows with gaps: the general kernel
    assert _plan(lib, a)[1].path == 0
    inp = wl.make_inputs(w.replace(n_seq=2, n_pad=0, extra_slots=0))
    c = cv.make_commit_args(inp["conv_state"], None, inp["accept_len"], layout="recompute", T=8, width=4,
                            x=inp["x"], check_device=False)
    assert c.x is not None and c.x_tok_stride == w.dim and c.x_seq_stride == 8 * w.dim
    c.x = None
    assert lib.cv_conv_commit(ctypes.byref(c), None) == -2
    c = cv.make_commit_args(inp["conv_state"], None, inp["accept_len"], layout="recompute", T=8, width=4,
                            x=inp["x"], check_device=False)
    c.x_tok_stride = -1
    assert lib.cv_conv_commit(ctypes.byref(c), None) == -9


def test_plan_sequence_list_only_with_cache_indices(lib):
    """The pipelined kernel lists the active sequences in shared memory when there are cache
    indices (and at most 1024 sequences); without indices every sequence is active."""
    a = _args(W3)
    base = _plan(lib, a)[1]
    a.cache_idx = None
    pl = _plan(lib, a)[1]
    assert pl.stages == base.stages and pl.smem_bytes == base.smem_bytes - 16 - 12 * 128
    a = _args(W3.replace(n_seq=1025, n_pad=0))
    pl = _plan(lib, a)[1]
    assert pl.path == 3 and pl.stages == base.stages and pl.smem_bytes == base.smem_bytes - 16 - 12 * 128


def test_plan_general_path_cases(lib):
    """Odd dims, long dedup rows and transposed rows with unaligned columns take the general kernel;
    transposed rows with 16-byte-aligned columns take the pipelined one (a bulk copy per column)."""
    assert _plan(lib, _args(W3.replace(dim=10236, qk_channels=4096)))[1].path == 0
    assert _plan(lib, _args(W3.replace(T=18)))[1].path == 0
    assert _plan(lib, _args(W3.replace(T=9, dtype="f32")))[1].path == 0
    assert _plan(lib, _args(W3.replace(T=8, dtype="f32")))[1].path == 3
    pl = _plan(lib, _args(W3.replace(head_dim=256, qk_channels=4096)))[1]
    assert pl.path == 3 and pl.channels_per_block == 8 * pl.threads  # a 256-channel group needs 8 per thread
    a = _args(W3)
    a.state_ch_stride = 4  # packed rows wider than the window: staged whole (4+ units per block)
    a.state_cols = 4
    pl = _plan(lib, a)[1]
    # stages of 8 x rows + 4 state columns; images of the 10-column dedup row + the 4-column rows
    assert pl.path == 3 and pl.smem_bytes == _pipe_smem((8 + 4) * 512 * 2, (10 + 4) * 512 * 2, 128)
    a.n_seq = 32  # too few units per block for wide rows: the one-pass kernel, the rows staged whole
    pl = _plan(lib, a)[1]
    assert pl.path == 1 and pl.smem_bytes == pl.channels_per_block * (10 + 4) * 2
    a.n_seq = 128
    a.state_ch_stride = 8  # rows with a gap between them: no bulk copy of the state
    assert _plan(lib, a)[1].path == 1
    assert _plan(lib, _args(W3.replace(T=12)))[1].path == 3
    a = _args(W3)
    a.win_ch_stride, a.win_col_stride, a.win_step_stride = 1, W3.dim, W3.dim
    pl = _plan(lib, a)[1]
    # the transposed row image and the committed-window image
    assert pl.path == 3 and pl.smem_bytes == _pipe_smem((8 + 3) * 512 * 2, (10 + 3) * 512 * 2, 128)
    a.win_col_stride = a.win_step_stride = W3.dim + 4  # columns 8 bytes off 16-byte alignment
    assert _plan(lib, a)[1].path == 0
    a = _args(W3)
    a.x_tok_stride = W3.dim + 1
    assert _plan(lib, a)[1].path == 0


@pytest.mark.parametrize("field,value,status", [
    ("dtype", 7, -6), ("width", 1, -5), ("width", 5, -5), ("T", 0, -4), ("T", 129, -4), ("n_seq", -1, -3),
    ("n_seq", 65536, -3), ("dim", 0, -3), ("n_slots", 0, -3), ("state_cols", 2, -3), ("window_layout", 5, -8), ("window_layout", 0, -8), ("window_layout", 3, -3),
    ("win_step_stride", 5, -8), ("qk_channels", 10240 + 128, -7), ("head_dim", 96, -7), ("head_dim", 4, -7),
    ("head_dim", 512, -7), ("qk_channels", 4000, -7), ("x_tok_stride", -1, -9), ("state_ch_stride", 2, -9),
    ("x", None, -2), ("weight", None, -2), ("window", None, -2),
])
def test_invalid_arguments_rejected(lib, field, value, status):
    a = _args(W3, **{field: value})
    assert _plan(lib, a)[0] == status
    # the launching entry point returns the same code without touching the GPU
    assert lib.cv_conv_verify(ctypes.byref(a), None) == status
    assert cv.status_string(status) not in ("", "unknown status")


def test_aliasing_rejected(lib):
    a = _args(W3)
    a.out = a.x
    assert _plan(lib, a)[0] == -10
    a = _args(W3)
    a.window = a.conv_state
    assert _plan(lib, a)[0] == -10
    a = _args(W3)
    a.window = a.out
    assert _plan(lib, a)[0] == -10


def test_null_args_and_plan(lib):
    assert lib.cv_conv_verify(None, None) == -1
    assert lib.cv_conv_commit(None, None) == -1
    a = _args(W3)
    assert lib.cv_verify_plan(ctypes.byref(a), None) == -2


def test_zero_sequences_is_ok_without_gpu(lib):
    a = _args(W3, n_seq=0, x=None, out=None)
    assert lib.cv_conv_verify(ctypes.byref(a), None) == 0


@pytest.mark.parametrize("T,dtype,threads", [(18, "bf16", 128), (32, "bf16", 128), (64, "f32", 32),
                                             (128, "f32", 32), (128, "bf16", 32)])
def test_general_plan_fits_shared_memory(lib, T, dtype, threads):
    """General kernel: the tile (T+W-1 rows of 8*threads channels plus 16 bytes) shrinks the block
    until it fits."""
    w = W3.replace(T=T, dtype=dtype, n_seq=2, n_pad=0, extra_slots=0)
    rc, pl = _plan(lib, _args(w))
    esize = 2 if dtype == "bf16" else 4
    assert rc == 0 and pl.path == 0 and pl.threads == threads
    assert pl.smem_bytes == (T + 3) * (8 * threads * esize + 16)
    assert pl.smem_bytes <= 96 * 1024 or threads == 32
    assert pl.smem_bytes <= 227 * 1024


def test_commit_validation(lib):
    w = W3.replace(n_seq=2, n_pad=0, extra_slots=0)
    inp = wl.make_inputs(w)
    a = cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"], layout="dedup", T=w.T,
                            width=w.width, check_device=False)
    a.accept_len = None
    assert lib.cv_conv_commit(ctypes.byref(a), None) == -2
    a = cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"], layout="dedup", T=w.T,
                            width=w.width, check_device=False)
    a.width = 6
    assert lib.cv_conv_commit(ctypes.byref(a), None) == -5
    a.width = 4
    a.win_step_stride = 99
    assert lib.cv_conv_commit(ctypes.byref(a), None) == -8


def test_binding_rejects_cpu_tensors(lib):
    w = wl.WORKLOADS[wl.WORKLOAD_ORDER[0]]
    inp = wl.make_inputs(w)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cv.conv_verify(inp["x"], inp["conv_state"], inp["weight"], None, inp["out"], inp["window"], layout="dense",
                       qk_channels=256, head_dim=64)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        cv.load_library(str(tmp_path / "nope.so"))


def _prefill_args(**over):
    w = wl.PREFILL_WORKLOADS[wl.PREFILL_ORDER[0]]
    inp = wl.make_prefill_inputs(w)
    a = cv.make_prefill_args(inp["x"], inp["conv_state"], inp["weight"], inp["bias"], inp["out"], inp["cu_seqlens"],
                             max_seqlen=w.max_seqlen, qk_channels=w.qk_channels, head_dim=w.head_dim,
                             cache_idx=inp["cache_idx"], has_initial_state=inp["has_initial_state"], check_device=False)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("dtype", 3, -6), ("width", 5, -5), ("n_seq", -1, -3), ("dim", 0, -3), ("total_tokens", -1, -3),
    ("max_seqlen", -2, -3), ("max_seqlen", 256 * 65536 + 1, -3), ("head_dim", 48, -7), ("qk_channels", 4096 + 8, -7),
    ("x_tok_stride", -1, -9), ("state_ch_stride", 1, -9), ("cu_seqlens", None, -2), ("weight", None, -2),
    ("x", None, -2),
])
def test_prefill_invalid_arguments_rejected(lib, field, value, status):
    a = _prefill_args(**{field: value})
    assert lib.cv_conv_prefill(ctypes.byref(a), None) == status


def test_prefill_aliasing_and_empty(lib):
    a = _prefill_args()
    a.out = a.x
    assert lib.cv_conv_prefill(ctypes.byref(a), None) == -10
    a = _prefill_args(n_seq=0)
    assert lib.cv_conv_prefill(ctypes.byref(a), None) == 0


def test_mixed_dtypes_plan_and_validation(lib):
    """bf16 x with an fp32 state (and the reverse) plan the pipelined kernel for T <= 8, its stage
    and image parts sized in each part's own dtype (no committed-window image: mixed dtypes store
    those runs from registers), and the general kernel with an fp32 tile above
    that; unknown state dtypes are rejected."""
    part = lambda b: (b + 127) // 128 * 128
    w = W3.replace(state_dtype="f32", n_seq=4, n_pad=0, extra_slots=0)
    a = _args(w)
    assert a.state_dtype == 1  # CV_STATE_F32
    rc, pl = _plan(lib, a)
    assert rc == 0 and pl.path == 3 and pl.stages == 2
    bc = pl.channels_per_block
    stage = part(8 * bc * 2) + part(3 * bc * 4)  # bf16 x rows, fp32 committed windows
    image = part(10 * bc * 4)  # fp32 dedup row (the committed windows go straight to the state)
    assert pl.smem_bytes == _pipe_smem(stage, image, 4)
    a.state_dtype = 3
    assert _plan(lib, a)[0] == -6
    w2 = W3.replace(dtype="f32", state_dtype="bf16", n_seq=4, n_pad=0, extra_slots=0)
    a2 = _args(w2)
    rc, pl2 = _plan(lib, a2)
    assert a2.state_dtype == 2 and rc == 0 and pl2.path == 3
    bc = pl2.channels_per_block
    assert pl2.smem_bytes == _pipe_smem(part(8 * bc * 4) + part(3 * bc * 2), part(10 * bc * 2), 4)
    # T = 9: no mixed pipelined kernel; the general kernel's tile holds fp32 bits
    w3 = W3.replace(state_dtype="f32", T=9, n_seq=4, n_pad=0, extra_slots=0)
    rc, pl3 = _plan(lib, _args(w3))
    assert rc == 0 and pl3.path == 0
    assert pl3.smem_bytes == (9 + 3) * (8 * pl3.threads + 4) * 4


def test_plan_token_groups(lib):
    """Small dense batches split the draft tokens among thread groups of the chunked one-pass kernel
    (path 2) while fewer than 8 warps per SM would run, each group keeping at least W-1 tokens and
    a block at most 256 threads; other layouts and large batches keep one group."""
    w4 = wl.WORKLOADS["n8_t17_dim8192_w4_bf16_dense_qkvsplit_xstride12288"]
    rc, pl = _plan(lib, _args(w4))
    # 8 x 64 blocks of one warp = 512 warps < 8 x 152: 4 groups of ceil(17 / 4) = 5 tokens
    assert rc == 0 and (pl.path, pl.threads, pl.token_groups) == (2, 32, 4)
    rc, pl = _plan(lib, _args(w4.replace(T=5)))
    assert (pl.path, pl.token_groups) == (2, 2)  # groups of 3 and 2 tokens (4 would hold 2 each)
    rc, pl = _plan(lib, _args(w4.replace(T=4)))
    assert (pl.path, pl.token_groups) == (1, 1)  # 2 groups would hold 2 tokens each
    rc, pl = _plan(lib, _args(w4.replace(layout="dedup")))
    assert pl.token_groups == 1
    rc, pl = _plan(lib, _args(W3))
    assert pl.token_groups == 1
    rc, pl = _plan(lib, _args(wl.WORKLOADS["n64_t8_dim6144_w3_bf16_dense_nol2_stateoff"]))
    assert (pl.path, pl.token_groups) == (1, 1)  # 64 x 12 blocks of 4 warps are enough


def test_tree_plan_and_validation(lib):
    """Tree verify: its own kernel (path 5) for the dense layout; other layouts and mixed dtypes
    are rejected."""
    w = wl.WORKLOADS["n8_t17_dim8192_w4_bf16_dense_qkvsplit_xstride12288"]
    inp = wl.make_inputs(w)
    parent = torch.arange(-1, w.T - 1, dtype=torch.int32).repeat(w.n_seq, 1).contiguous()
    a = cv.make_verify_args(inp["x"], inp["conv_state"], inp["weight"], inp["bias"], inp["out"], inp["window"],
                            layout="dense", qk_channels=w.qk_channels, head_dim=w.head_dim,
                            cache_idx=inp["cache_idx"], parent=parent, check_device=False)
    rc, pl = _plan(lib, a)
    # persistent two-warp blocks over (sequence, 256 channels) units, two unit buffers of
    # (W-1+T) rows of 256 bf16 + the packed [256][W-1] window run + T int32 parents (16-byte rounded)
    buf = (3 + 17) * 256 * 2 + 256 * 3 * 2 + 80
    assert rc == 0 and pl.path == 5 and pl.threads == 64 and pl.channels_per_block == 256
    assert pl.smem_bytes == 2 * buf and pl.stages == 2
    # 9 blocks per SM fit (232448 // (2 * buf + 1024)); 8 x 32 = 256 units bound the grid
    assert (pl.grid_x, pl.grid_y) == (256, 1)
    a.window_layout = 2
    a.win_step_stride = a.win_col_stride
    assert _plan(lib, a)[0] == -8
    a = _args(W3.replace(state_dtype="f32", layout="dense", n_seq=2, n_pad=0, extra_slots=0))
    a.parent = parent.data_ptr()
    assert _plan(lib, a)[0] == -6
    # 128 fp32 tokens: two buffers of 131 staged rows of 1 KB do not fit, one does
    w = W3.replace(dtype="f32", layout="dense", T=128, n_seq=2, n_pad=0, extra_slots=0)
    a = _args(w)
    big = torch.arange(-1, 127, dtype=torch.int32).repeat(2, 1).contiguous()
    a.parent = big.data_ptr()
    rc, pl = _plan(lib, a)
    assert rc == 0 and pl.path == 5 and pl.threads == 64 and pl.stages == 1
    assert pl.smem_bytes == (3 + 128) * 256 * 4 + 256 * 3 * 4 + 512
    assert pl.grid_x == 2 * 10240 // 256  # one block per SM would be 152 > the 80 units
    # the benchmark shape: 10 blocks per SM, a multiple of the 40 channel blocks
    a = _args(W3.replace(layout="dense"))
    par8 = torch.arange(-1, 7, dtype=torch.int32).repeat(W3.n_seq, 1).contiguous()
    a.parent = par8.data_ptr()
    rc, pl = _plan(lib, a)
    buf = (3 + 8) * 256 * 2 + 256 * 3 * 2 + 32
    per_sm = min(10, 232448 // (2 * buf + 1024))
    assert rc == 0 and pl.smem_bytes == 2 * buf and pl.grid_x == 152 * per_sm // 40 * 40 == 1520
    # one draft token: one warp
    a.T = 1
    assert _plan(lib, a)[1].threads == 32


def _verify_inputs(layout="dedup", **over):
    w = wl.VerifyWorkload("bind", n_seq=3, T=4, dim=64, width=4, qk_channels=32, head_dim=16, dtype="bf16",
                          layout=layout, bias=True, seed=1, **over)
    return w, wl.make_inputs(w)


def _make(w, inp, **over):
    kw = dict(layout=w.layout, qk_channels=w.qk_channels, head_dim=w.head_dim, cache_idx=inp["cache_idx"],
              state_off=inp.get("state_off"), parent=inp.get("parent"), check_device=False)
    kw.update({k: v for k, v in over.items() if k in kw})
    args = [over.get(k, inp[k]) for k in ("x", "conv_state", "weight", "bias", "out", "window")]
    return cv.make_verify_args(*args, **kw)


@pytest.mark.parametrize("what", ["out", "bias", "weight", "window", "state_dim", "cache_idx_short",
                                  "cache_idx_int64", "parent_shape", "parent_float", "err_short"])
def test_binding_rejects_buffers_smaller_than_described(what):
    """The library sees only pointers, so the binding checks every buffer against the sizes the
    arguments describe: a wrong shape or index dtype raises before anything reaches the library."""
    w, inp = _verify_inputs(layout="dense")
    n, T, dim = w.n_seq, w.T, w.dim
    bad = {
        "out": dict(out=torch.empty(n, T, dim - 8, dtype=torch.bfloat16)),
        "bias": dict(bias=torch.empty(dim + 1, dtype=torch.bfloat16)),
        "weight": dict(weight=torch.empty(dim - 8, 4, dtype=torch.bfloat16)),
        "window": dict(window=torch.empty(n, T - 1, dim, 3, dtype=torch.bfloat16)),
        "state_dim": dict(conv_state=torch.empty(w.n_slots, dim - 8, 3, dtype=torch.bfloat16)),
        "cache_idx_short": dict(cache_idx=torch.zeros(n - 1, dtype=torch.int32)),
        "cache_idx_int64": dict(cache_idx=torch.zeros(n, dtype=torch.int64)),
        "parent_shape": dict(parent=torch.full((n, T - 1), -1, dtype=torch.int32)),
        "parent_float": dict(parent=torch.full((n, T), -1.0, dtype=torch.float32)),
        "err_short": dict(err=torch.zeros(n - 1, dtype=torch.int32)),
    }[what]
    if "err" in bad:
        with pytest.raises(ValueError):
            cv.make_verify_args(inp["x"], inp["conv_state"], inp["weight"], inp["bias"], inp["out"], inp["window"],
                                layout="dense", qk_channels=w.qk_channels, head_dim=w.head_dim, err=bad["err"],
                                check_device=False)
        return
    with pytest.raises(ValueError):
        _make(w, inp, **bad)
    _make(w, inp)  # the unmodified inputs pass


def test_binding_commit_and_prefill_shapes():
    """The commit checks its window against (n_seq, T, dim) and its index arrays; the prefill its
    out, taps and per-sequence arrays against cu_seqlens."""
    w, inp = _verify_inputs(layout="dedup")
    ok = dict(layout="dedup", T=w.T, width=w.width, cache_idx=inp["cache_idx"], check_device=False)
    cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"], **ok)
    with pytest.raises(ValueError):
        cv.make_commit_args(inp["conv_state"], inp["window"][:, :, :-1], inp["accept_len"], **ok)
    with pytest.raises(ValueError):
        cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"].to(torch.int64), **ok)
    with pytest.raises(ValueError):
        cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"],
                            **dict(ok, cache_idx=inp["cache_idx"][:-1]))
    pw = wl.PREFILL_WORKLOADS[wl.PREFILL_ORDER[0]]
    p = wl.make_prefill_inputs(pw)
    kw = dict(max_seqlen=pw.max_seqlen, qk_channels=pw.qk_channels, head_dim=pw.head_dim, check_device=False)
    cv.make_prefill_args(p["x"], p["conv_state"], p["weight"], p["bias"], p["out"], p["cu_seqlens"], **kw)
    with pytest.raises(ValueError):
        cv.make_prefill_args(p["x"], p["conv_state"], p["weight"], p["bias"], p["out"][:-1], p["cu_seqlens"], **kw)
    with pytest.raises(ValueError):
        cv.make_prefill_args(p["x"], p["conv_state"], p["weight"], p["bias"], p["out"], p["cu_seqlens"],
                             cache_idx=torch.zeros(p["cu_seqlens"].numel() - 2, dtype=torch.int32), **kw)


def test_struct_layouts_match_header(tmp_path):
    """The binding's ctypes mirrors have the C structs' field offsets and sizes (a field added to
    the header but not to the binding, or the reverse, would shift every later field)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mirrors = {"cv_verify_args": cv.VerifyArgs, "cv_commit_args": cv.CommitArgs,
               "cv_prefill_args": cv.PrefillArgs, "cv_launch_plan": cv.LaunchPlan}
    lines = ["#include <stddef.h>", "#include <stdio.h>", f'#include "{HEADER}"', "int main(void) {"]
    for cname, py in mirrors.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-o", str(exe), str(src)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    c_side = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in got if ln.strip()}
    for cname, py in mirrors.items():
        assert c_side[(cname, "size")] == ctypes.sizeof(py), f"{cname}: sizeof differs"
        for fname, _ in py._fields_:
            assert c_side[(cname, fname)] == getattr(py, fname).offset, f"{cname}.{fname}: offset differs"


RAG = wl.RAGGED_WORKLOADS["ragged_n128_t1to16_dim10240_w4_bf16_dedup_pad13"]


def _ragged_args(w, **over):
    inp = wl.make_ragged_inputs(w)
    a = cv.make_verify_args(inp["x"], inp["conv_state"], inp["weight"], inp["bias"], inp["out"], inp["window"],
                            layout=w.layout, qk_channels=w.qk_channels, head_dim=w.head_dim,
                            cache_idx=inp["cache_idx"], state_off=inp["state_off"], cu_draft=inp["cu_draft"], T=w.T,
                            check_device=False)
    _ragged_args.keep = inp
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_plan_packed_drafts_pipelined(lib):
    """Packed ragged drafts of up to 16 tokens at the benchmark shape take the pipelined kernel in
    units of 8-token chunks: stages of 8 + 3 x rows (the chunk, then its halo or the draft's tail)
    and the committed windows, row images of 8 + 2 columns (no committed-window image), the sort
    scratch and a list of 2 chunks per sequence."""
    a = _ragged_args(RAG)
    rc, pl = _plan(lib, a)
    assert rc == 0 and pl.path == 3
    R, bc = RAG.width - 1, 512
    Q = 8 + R - 1

    def part(b):
        return (b + 127) // 128 * 128
    stage = part((8 + R) * bc * 2) + part(R * bc * 2)
    image = part(Q * bc * 2)  # (the committed windows go straight from registers to the state)
    assert pl.smem_bytes == _pipe_smem(stage, image, RAG.n_seq, varlen_T=RAG.T)
    # longer drafts (T = 40: 5 chunks per sequence) still fit the list; history rows do not chunk
    assert _plan(lib, _ragged_args(RAG.replace(T=40)))[1].path == 3
    assert _plan(lib, _ragged_args(RAG.replace(layout="history", T=8)))[1].path == 3
    assert _plan(lib, _ragged_args(RAG.replace(layout="history", T=16)))[1].path == 0


def test_packed_drafts_argument_checks(lib):
    """cu_draft with a tree is a layout error, a negative total_tokens a shape error; with no rows
    at all x and out may be NULL; unaligned x falls back to the general kernel."""
    rc, _ = _plan(lib, _ragged_args(RAG, parent=_ragged_args.keep["cache_idx"].data_ptr()))
    assert rc == -8
    rc, _ = _plan(lib, _ragged_args(RAG, total_tokens=-1))
    assert rc == -3
    w0 = RAG.replace(lengths=(0,) * 4, pad=(), extra_rows=0)
    a = _ragged_args(w0, x=None, out=None)
    rc, pl = _plan(lib, a)
    assert rc == 0
    a = _ragged_args(RAG)
    a.x = a.x + 2  # one bf16 element off 16-byte alignment
    rc, pl = _plan(lib, a)
    assert rc == 0 and pl.path == 0


def test_packed_commit_argument_checks(lib):
    inp = wl.make_ragged_inputs(RAG)
    ca = cv.make_commit_args(inp["conv_state"], inp["window"], inp["accept_len"], layout=RAG.layout, T=RAG.T,
                             width=RAG.width, cache_idx=inp["cache_idx"], cu_draft=inp["cu_draft"],
                             total_tokens=RAG.total_tokens, check_device=False)
    assert ca.total_tokens == RAG.total_tokens and ca.cu_draft == inp["cu_draft"].data_ptr()
    ca.total_tokens = -1
    assert lib.cv_conv_commit(ctypes.byref(ca), None) == -3
