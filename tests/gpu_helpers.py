"""GPU-side runners for the parity tests (CUDA library through the C ABI)."""
from __future__ import annotations

import torch

from spec_decode_verify_gb300 import workloads as wl


def to_device(inp: dict, device="cuda") -> dict:
    """Copy a make_inputs() dict to the GPU, keeping x as a strided view of its wide buffer."""
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    if "x_base" in inp:
        base = inp["x_base"].to(device)
        x = inp["x"]
        out["x_base"] = base
        out["x"] = base.as_strided(x.shape, x.stride(), x.storage_offset())
    if inp.get("window") is not None:
        w = inp["window"]
        # keep the window's strides (a transposed row stays transposed)
        if not w.is_contiguous():
            st = torch.empty_strided(w.shape, w.stride(), dtype=w.dtype, device=device)
            st.copy_(w)
            out["window"] = st
    return out


def run_gpu_verify(cv, w: wl.VerifyWorkload, inp: dict, err=True) -> dict:
    d = to_device(inp)
    d["err"] = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda") if err else None
    cv.conv_verify(d["x"], d["conv_state"], d["weight"], d["bias"], d["out"], d["window"], layout=w.layout,
                   qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=d["cache_idx"],
                   state_off=d["state_off"], err=d["err"], parent=d.get("parent"))
    torch.cuda.synchronize()
    return d


def run_gpu_commit(cv, w: wl.VerifyWorkload, d: dict, accept_len=None) -> torch.Tensor:
    e = torch.full((w.n_seq,), -7, dtype=torch.int32, device="cuda")
    acc = d["accept_len"] if accept_len is None else accept_len.to("cuda")
    cv.conv_commit(d["conv_state"], d["window"], acc, layout=w.layout, T=w.T, width=w.width,
                   cache_idx=d["cache_idx"], err=e, x=d["x"] if w.layout == "recompute" else None)
    torch.cuda.synchronize()
    return e
