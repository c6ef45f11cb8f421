"""Shared test helpers: tolerance checks and convenience runners (no method arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from spec_decode_verify_gb300 import workloads as wl

# Output tolerances (the stated bar): fp32 |g - r| <= 1e-5 |r| + 1e-7 elementwise (the 1e-7 floor
# covers SiLU outputs next to zero); bf16 at most 2 units in the last place, counted as the
# distance between the two values' positions in the ordered list of bf16 numbers.
F32_RTOL = 1e-5
F32_ATOL = 1e-7
BF16_MAX_ULP = 2


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a CPU tensor as unsigned integers."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype == torch.int32:
        return t.numpy().view(np.uint32)
    raise TypeError(t.dtype)


def bf16_ordinal(b: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotone in the value (-0 and +0 both map to 0)."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_bits_equal(got: torch.Tensor, ref: torch.Tensor, what: str):
    g, r = bits(got), bits(ref)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    bad = np.nonzero(g != r)
    if bad[0].size:
        idx = tuple(int(a[0]) for a in bad)
        raise AssertionError(f"{what}: {bad[0].size} of {g.size} elements differ bitwise; first at {idx}: "
                             f"got {g[idx]:#x} want {r[idx]:#x}")


# bf16 absolute floor at the fp32 exp overflow point: where exp(-acc) overflows on one side and not on
# the other (acc near -88.72), SiLU is -0 on one side and about -2.6e-37 on the other (at most 1000x
# that after an L2 scale); pairs whose two values are both below this magnitude compare equal.
BF16_EXP_OVERFLOW_FLOOR = 1e-30


def assert_out_close(got: torch.Tensor, ref: torch.Tensor, what: str = "out", bf16_floor: float = 0.0):
    """The output tolerance; NaN must match NaN.  bf16_floor: bf16 pairs whose two values are both
    below it in magnitude are accepted (used only where conv results reach the exp overflow point)."""
    assert got.shape == ref.shape and got.dtype == ref.dtype
    g32 = got.detach().cpu().float().numpy()
    r32 = ref.detach().cpu().float().numpy()
    gn, rn = np.isnan(g32), np.isnan(r32)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    m = ~rn
    if got.dtype == torch.bfloat16:
        if bf16_floor > 0:
            m = m & ~((np.abs(g32) < bf16_floor) & (np.abs(r32) < bf16_floor))
        d = np.abs(bf16_ordinal(bits(got)) - bf16_ordinal(bits(ref)))[m]
        if d.size and d.max() > BF16_MAX_ULP:
            i = int(np.argmax(d))
            raise AssertionError(f"{what}: {int((d > BF16_MAX_ULP).sum())} elements beyond {BF16_MAX_ULP} bf16 ulp;"
                                 f" worst {int(d.max())} ulp (got {g32[m][i]} want {r32[m][i]})")
    else:
        err = np.abs(g32[m].astype(np.float64) - r32[m].astype(np.float64))
        lim = F32_RTOL * np.abs(r32[m].astype(np.float64)) + F32_ATOL
        if err.size and (err > lim).any():
            i = int(np.argmax(err - lim))
            raise AssertionError(f"{what}: {int((err > lim).sum())} elements beyond tolerance;"
                                 f" worst got {g32[m][i]} want {r32[m][i]}")


def clone_inputs(inp: dict) -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = v.clone() if isinstance(v, torch.Tensor) else v
    # keep x as a view of its own wide copy so the token stride survives the clone
    if "x_base" in inp:
        base = inp["x_base"].clone()
        x = inp["x"]
        out["x_base"] = base
        out["x"] = base.as_strided(x.shape, x.stride(), x.storage_offset())
    return out


def run_oracle_verify(w: wl.VerifyWorkload, inp: dict, status: bool = True) -> dict:
    """Oracle verify on a copy of ``inp``; returns the copy (state/out/window written)."""
    r = clone_inputs(inp)
    r["status"] = torch.full((w.n_seq,), -7, dtype=torch.int32) if status else None
    oracle.conv_verify(r["x"], r["conv_state"], r["weight"], r["bias"], r["out"], r["window"], layout=w.layout,
                       qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps, cache_idx=r["cache_idx"],
                       state_off=r["state_off"], status=r["status"], parent=r.get("parent"))
    return r


def run_oracle_commit(w: wl.VerifyWorkload, r: dict, accept_len=None) -> torch.Tensor:
    """Oracle commit in place on ``r`` (the result of run_oracle_verify); returns the status."""
    st = torch.full((w.n_seq,), -7, dtype=torch.int32)
    oracle.conv_commit(r["conv_state"], r["window"], r["accept_len"] if accept_len is None else accept_len,
                       layout=w.layout, T=w.T, width=w.width, cache_idx=r["cache_idx"], status=st,
                       x=r["x"] if w.layout == "recompute" else None)
    return st
