"""Benchmark of the batched speculative-verify conv1d update (verify + commit) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole path over one batch: cv_conv_verify (conv + SiLU + L2, snapshots,
committed window) followed by cv_conv_commit (restore the accepted prefix); with the history-row
state layout the step is the verify alone (the next verify reads at accept_len - 1), and with the
recompute rollback the verify writes outputs only and the commit rebuilds the state from x.  Default workload: 128
sequences x 8 draft tokens, dim 10240 (q|k 4096, head_dim 128), conv width 4, bf16, deduplicated
window rows, 13 padded sequences.  Inputs are synthetic and already resident in HBM when the
timed region starts; every step uses the next of several rotating buffer sets whose total size is
at least four times the L2, so each step reads and writes HBM, not L2.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own batch (weak scaling, no
collective on the data path); the step time is the maximum over ranks.  ``--impl reference`` times
the CPU oracle (plain C loop, one core) on the same workload and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from spec_decode_verify_gb300 import workloads as wl  # noqa: E402

METRIC = "verify-conv µs/step and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "us/step"
HBM_NOMINAL_GBS = 8000.0  # the metric's roofline: bytes moved / 8 TB/s
PROFILES = os.path.join(ROOT, "profiles")
# the sources of each main kernel (verify: the pipelined path), keyed as in profiles' traffic lines
_CSRC = os.path.join(ROOT, "spec_decode_verify_gb300", "csrc")
KERNEL_SRCS = {
    kind: [os.path.join(_CSRC, f) for f in (src, "cv_device.cuh")]
    for kind, src in (("verify", "cv_verify_pipe.cuh"), ("prefill", "cv_prefill.cuh"), ("fast", "cv_verify_fast.cuh"),
                      ("generic", "cv_verify_generic.cuh"), ("tree", "cv_verify_tree.cuh"))
}
# launch path of cv_verify_plan -> (kernel, source kind)
PATH_KERNELS = {0: ("verify_generic", "generic"), 1: ("verify_fast", "fast"), 2: ("verify_fast", "fast"),
                3: ("verify_pipe", "verify"), 5: ("verify_tree", "tree")}


def kernel_sha(kind: str = "verify") -> str:
    h = hashlib.sha256()
    for path in KERNEL_SRCS[kind]:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profile_traffic(workload: str, kind: str = "verify"):
    """DRAM bytes per launch of the workload's main kernel from a committed ncu summary of this
    workload, if it was taken of the current kernel sources (a `bench-traffic:` line in
    profiles/*.md)."""
    stale = False
    for name in sorted(os.listdir(PROFILES)) if os.path.isdir(PROFILES) else []:
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(PROFILES, name)).read()
        for m in re.finditer(r"bench-traffic: workload=(\S+) dram_bytes_per_launch=(\d+) kernel_sha=([0-9a-f]+)",
                             text):
            if m.group(1) != workload:
                continue
            if m.group(3) != kernel_sha(kind):
                stale = True
                continue
            return int(m.group(2)), f"ncu ({name})"
    return None, ("stale" if stale else None)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler (200 ms) around the loaded region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path=None):
        self.index = index
        self.proc = None
        # the raw samples go to `path` (kept), else to a temporary file
        self.path = path or os.path.join(tempfile.gettempdir(), f"cv_clocks_{os.getpid()}_{index}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("pcap", "sw_power_cap")):
                if r[k].lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def e2e_pipelined(dev, dist, K, sets, inp, launch, ins, outs):
    """Time K end-to-end steps: every step uploads its inputs from pinned host memory, runs the
    path through the C ABI and downloads its result to pinned host memory.  Two device buffer sets
    alternate over three streams (upload, compute, download) with events ordering each buffer's
    reuse, so the copies of neighbouring steps overlap each other and the compute.  Returns
    (us per step, upload bytes per step, download bytes per step)."""
    host_in = [(name, t.clone().pin_memory()) for name, t in ins]
    host_out = [[torch.empty_like(s[name], device="cpu").pin_memory() for name in outs] for s in sets]
    h2d = sum(t.numel() * t.element_size() for _, t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nb = len(sets)
    computed = [torch.cuda.Event() for _ in range(nb)]
    downloaded = [torch.cuda.Event() for _ in range(nb)]
    uploaded = [torch.cuda.Event() for _ in range(nb)]

    def run(n):
        for i in range(n):
            b = i % nb
            s = sets[b]
            up.wait_event(computed[b])  # the set's previous step has read its inputs
            with torch.cuda.stream(up):
                for name, t in host_in:
                    s[name].copy_(t, non_blocking=True)
            uploaded[b].record(up)
            comp.wait_event(uploaded[b])
            comp.wait_event(downloaded[b])  # its previous result has left the device
            if launch(s, b, comp.cuda_stream) != 0:
                raise RuntimeError("launch failed")
            computed[b].record(comp)
            down.wait_event(computed[b])
            with torch.cuda.stream(down):
                for t, name in zip(host_out[b], outs):
                    t.copy_(s[name], non_blocking=True)
            downloaded[b].record(down)

    for b in range(nb):  # the events start recorded
        computed[b].record(comp)
        downloaded[b].record(comp)
    run(3)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    run(K)
    end_ev = torch.cuda.Event()
    end_ev.record(down)
    comp.wait_event(end_ev)
    up.wait_event(end_ev)
    e1.record(up)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    return reduce_max(dist, e0.elapsed_time(e1) * 1e3 / K, dev), h2d, d2h


def launch_ranks(n: int) -> int:
    """Run this same command as n ranks under torch.distributed.run (one node, one rank per GPU,
    rendezvous on 127.0.0.1) and return its exit status.  Used when --gpus N > 1 is given without a
    launcher, so that an N-GPU line always comes from N ranks."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return world, rank, local, dist
    return 1, 0, 0, None


def reduce_max(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device):
    if dist is not None:
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_step_times(w, reps_max: int, budget_s: float):
    """Time oracle verify + commit on the whole workload (one core); returns per-step seconds."""
    import oracle
    ragged = isinstance(w, wl.RaggedWorkload)
    inp = wl.make_ragged_inputs(w) if ragged else wl.make_inputs(w)
    rag_kw = dict(cu_draft=inp["cu_draft"], T=w.T) if ragged else {}
    commit_kw = dict(cu_draft=inp["cu_draft"], total_tokens=w.total_tokens) if ragged else {}
    times = []
    t_begin = time.perf_counter()
    for _ in range(reps_max):
        state = inp["conv_state"].clone()
        out = inp["out"].clone()
        win = inp["window"].clone() if inp["window"] is not None else None
        t0 = time.perf_counter()
        oracle.conv_verify(inp["x"], state, inp["weight"], inp["bias"], out, win, layout=w.layout,
                           qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps,
                           cache_idx=inp["cache_idx"], state_off=inp["state_off"], parent=inp.get("parent"), **rag_kw)
        if w.layout != "history":
            oracle.conv_commit(state, win, inp["accept_len"], layout=w.layout, T=w.T, width=w.width,
                               cache_idx=inp["cache_idx"], x=inp["x"] if w.layout == "recompute" else None,
                               **commit_kw)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_begin > budget_s and len(times) >= 3:
            break
    return times


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    warm = oracle_step_times(w, max(args.warmup, 1), 1e9)
    times = oracle_step_times(w, args.steps, 1e9)
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": round(us, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"whole workload ({w.n_seq} sequences) per step, {len(times)} steps after "
                                   f"{len(warm)} warm-up; plain C loop, one thread"},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# How the GPU arm keeps each step out of L2 (both arms' config carries it, so the two configs are
# identical; the GPU arm's line adds the set count and sizes under "l2_sets").
L2_RULE = "inputs larger than L2: every step uses the next of rotating buffer sets totalling >= 4x L2"


def workload_config(w):
    c = {"workload": w.name, "n_seq": w.n_seq, "padded_seqs": w.n_pad, "T": w.T, "dim": w.dim, "width": w.width,
         "qk_channels": w.qk_channels, "head_dim": w.head_dim, "layout": w.layout, "bias": w.bias,
         "step": "cv_conv_verify" if w.layout == "history" else "cv_conv_verify + cv_conv_commit",
         "l2": L2_RULE}
    if isinstance(w, wl.RaggedWorkload):
        c.update(draft_tokens="packed ragged: T_s per sequence, T = the largest", total_tokens=w.total_tokens,
                 active_draft_tokens=sum(L for i, L in enumerate(w.lengths) if i not in w.pad))
    return c


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, w, world, rank, local, dist):
    import spec_decode_verify_gb300 as cv
    from spec_decode_verify_gb300 import build as cvbuild

    cvbuild.build()
    lib = cv.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    ragged = isinstance(w, wl.RaggedWorkload)
    inp = (wl.make_ragged_inputs if ragged else wl.make_inputs)(w, seed=w.seed + 1009 * rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20
    per_set = sum(inp[k].numel() * inp[k].element_size()
                  for k in ("x_base", "conv_state", "out", "window") if inp[k] is not None)
    has_commit = w.layout != "history"
    n_sets = max(2, math.ceil(4 * l2 / per_set))
    l2_note = f"rotating {n_sets} buffer sets, {n_sets * per_set / 2**20:.0f} MiB >= 4x L2 ({l2 / 2**20:.0f} MiB)"

    weight = inp["weight"].to(dev)
    bias = inp["bias"].to(dev) if inp["bias"] is not None else None
    cache_idx = inp["cache_idx"].to(dev)
    state_off = inp["state_off"].to(dev) if inp["state_off"] is not None else None
    parent = inp["parent"].to(dev) if inp.get("parent") is not None else None
    cu = inp["cu_draft"].to(dev) if ragged else None
    rag_kw = dict(cu_draft=cu, T=w.T) if ragged else {}
    commit_kw = dict(cu_draft=cu, total_tokens=w.total_tokens) if ragged else {}
    sets = []
    for i in range(n_sets):
        xb = inp["x_base"].to(dev)
        x = xb.as_strided(inp["x"].shape, inp["x"].stride(), inp["x"].storage_offset())
        win = None
        if inp["window"] is not None:  # (keeping its strides: a transposed row stays transposed)
            win = torch.empty_strided(inp["window"].shape, inp["window"].stride(), dtype=inp["window"].dtype, device=dev)
            win.copy_(inp["window"])
        s = dict(x_base=xb, x=x, conv_state=inp["conv_state"].to(dev), out=inp["out"].to(dev), window=win,
                 accept=inp["accept_len"].to(dev))
        s["va"] = cv.make_verify_args(x, s["conv_state"], weight, bias, s["out"], s["window"], layout=w.layout,
                                      qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps,
                                      cache_idx=cache_idx, state_off=state_off, parent=parent, **rag_kw)
        if has_commit:
            s["ca"] = cv.make_commit_args(s["conv_state"], s["window"], s["accept"], layout=w.layout, T=w.T,
                                          width=w.width, cache_idx=cache_idx,
                                          x=x if w.layout == "recompute" else None, **commit_kw)
        sets.append(s)
    verify_fn, lib_commit = lib.cv_conv_verify, lib.cv_conv_commit
    vrefs = [ctypes.byref(s["va"]) for s in sets]
    plan = cv.LaunchPlan()
    if lib.cv_verify_plan(vrefs[0], ctypes.byref(plan)) != 0:
        raise RuntimeError("cv_verify_plan rejected the workload")
    kernel_name, kernel_kind = PATH_KERNELS[plan.path]
    crefs = [ctypes.byref(s["ca"]) if has_commit else None for s in sets]

    def commit_fn(ref, stream_ptr):
        return lib_commit(ref, stream_ptr) if has_commit else 0

    def step(i):
        rc = verify_fn(vrefs[i % n_sets], sp)
        rc |= commit_fn(crefs[i % n_sets], sp)
        return rc

    for i in range(args.warmup):
        if step(i) != 0:
            raise RuntimeError("launch failed during warm-up")
    torch.cuda.synchronize(dev)

    # clocks: sample during a loaded stretch right before and through the timed region
    sampler = ClockSampler(dev.index, args.clocks_csv)
    sampler.start()
    t_end = time.perf_counter() + args.clock_probe_s
    i = 0
    while time.perf_counter() < t_end:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    K = args.steps
    # (1) the step time: K steps back to back between two events, nothing else on the stream
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    # keep the GPU busy while the host queues the K steps, so no launch waits on the host
    torch.cuda._sleep(int(min(2e9, 40000 * K + 2e6)))
    start.record(stream)
    for i in range(K):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    # (2) the split into verify and commit: K launches of each kernel alone, back to back, between
    # two events on the launching stream (an event between every two launches would add its own gap)
    def time_alone(fn, refs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(int(min(2e9, 30000 * K + 2e6)))
        e0.record(stream)
        for i in range(K):
            fn(refs[i % n_sets], sp)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / K

    verify_us = time_alone(verify_fn, vrefs)
    commit_us = time_alone(commit_fn, crefs) if has_commit else 0.0
    barrier(dist, dev)
    clocks = sampler.stop()

    step_us = start.elapsed_time(end) * 1e3 / K
    step_us_max = reduce_max(dist, step_us, dev)
    verify_us_max = reduce_max(dist, verify_us, dev)

    # e2e: host buffers through the C ABI, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e_us, h2d, d2h = e2e_pipelined(
            dev, dist, K, sets[:2], inp,
            lambda st, idx, stream_ptr: verify_fn(vrefs[idx], stream_ptr) | commit_fn(crefs[idx], stream_ptr),
            ins=[("x_base", inp["x_base"]), ("accept", inp["accept_len"])], outs=["out"])
        e2e = {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "double-buffered: step i+1's upload and step i-1's download overlap step i"}

    if rank != 0:
        return 0

    nbytes = wl.ragged_algorithmic_bytes(w) if ragged else wl.algorithmic_bytes(w)
    peak, peak_kind = measured_peak()
    achieved = nbytes["verify"] / (verify_us_max * 1e-6) / 1e9
    traffic, traffic_src = profile_traffic(w.name, kernel_kind)
    line = {
        "metric": METRIC, "value": round(step_us_max, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_us_max / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w), "l2_sets": l2_note,
        "verify_us": round(verify_us_max, 3), "commit_us": round(commit_us, 3),
        "verify_gbs": round(achieved, 1), "verify_frac_of_8tbs": round(achieved / HBM_NOMINAL_GBS, 4),
        "verify_algorithmic_bytes": nbytes["verify"], "commit_algorithmic_bytes": nbytes["commit"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_name, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "traffic_source": traffic_src},
        "gpu_launches": (2 if has_commit else 1) * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        times = oracle_step_times(w, 200, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": round(statistics.median(times) * 1e6, 1), "unit": UNIT, "cores": 1,
                                "kind": "oracle",
                                "sample": f"whole workload ({w.n_seq} sequences) per step, median of {len(times)} "
                                          f"steps; plain C loop, one thread"}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- prefill workloads

def prefill_config(w):
    return {"workload": w.name, "n_seq": w.n_seq, "total_tokens": w.total_tokens, "max_seqlen": w.max_seqlen,
            "dim": w.dim, "width": w.width, "qk_channels": w.qk_channels, "head_dim": w.head_dim,
            "padded_seqs": len(w.pad), "without_initial_state": len(w.no_init), "step": "cv_conv_prefill",
            "l2": L2_RULE}


def oracle_prefill_times(w, reps_max: int, budget_s: float):
    """Time the oracle prefill on the whole workload (one core); returns per-step seconds."""
    import oracle
    inp = wl.make_prefill_inputs(w)
    times = []
    t_begin = time.perf_counter()
    for _ in range(reps_max):
        state, out = inp["conv_state"].clone(), inp["out"].clone()
        t0 = time.perf_counter()
        oracle.conv_prefill(inp["x"], state, inp["weight"], inp["bias"], out, inp["cu_seqlens"],
                            qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps,
                            cache_idx=inp["cache_idx"], has_initial_state=inp["has_initial_state"])
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_begin > budget_s and len(times) >= 1:
            break
    return times


def run_reference_prefill(args, w, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    warm = oracle_prefill_times(w, 1, 1e9)
    times = oracle_prefill_times(w, args.steps, args.cpu_budget_s * 6)
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world,
        "steps": len(times), "warmup": len(warm), "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": prefill_config(w),
        "cpu_baseline": {"value": round(us, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"whole workload ({w.total_tokens} tokens) per step, {len(times)} steps; "
                                   f"plain C loop, one thread"},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_prefill(args, w, world, rank, local, dist):
    import spec_decode_verify_gb300 as cv
    from spec_decode_verify_gb300 import build as cvbuild

    cvbuild.build()
    lib = cv.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    inp = wl.make_prefill_inputs(w, seed=w.seed + 1009 * rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20
    per_set = sum(inp[k].numel() * inp[k].element_size() for k in ("x_base", "conv_state", "out"))
    n_sets = max(2, math.ceil(4 * l2 / per_set))
    l2_note = f"rotating {n_sets} buffer sets, {n_sets * per_set / 2**20:.0f} MiB >= 4x L2 ({l2 / 2**20:.0f} MiB)"
    weight = inp["weight"].to(dev)
    bias = inp["bias"].to(dev) if inp["bias"] is not None else None
    cu, cidx, init = (inp[k].to(dev) for k in ("cu_seqlens", "cache_idx", "has_initial_state"))
    sets = []
    for _ in range(n_sets):
        xb = inp["x_base"].to(dev)
        x = xb.as_strided(inp["x"].shape, inp["x"].stride(), inp["x"].storage_offset())
        s = dict(x_base=xb, x=x, conv_state=inp["conv_state"].to(dev), out=inp["out"].to(dev))
        s["pa"] = cv.make_prefill_args(x, s["conv_state"], weight, bias, s["out"], cu, max_seqlen=w.max_seqlen,
                                       qk_channels=w.qk_channels, head_dim=w.head_dim, l2_eps=w.l2_eps,
                                       cache_idx=cidx, has_initial_state=init)
        sets.append(s)
    refs = [ctypes.byref(s["pa"]) for s in sets]
    fn = lib.cv_conv_prefill

    for i in range(args.warmup):
        if fn(refs[i % n_sets], sp) != 0:
            raise RuntimeError("launch failed during warm-up")
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index, args.clocks_csv)
    sampler.start()
    t_end = time.perf_counter() + args.clock_probe_s
    i = 0
    while time.perf_counter() < t_end:
        fn(refs[i % n_sets], sp)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(int(min(2e9, 400000 * K + 2e6)))
    start.record(stream)
    for i in range(K):
        fn(refs[i % n_sets], sp)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks = sampler.stop()
    step_us = reduce_max(dist, start.elapsed_time(end) * 1e3 / K, dev)

    e2e = None
    if not args.no_e2e:
        e2e_us, h2d, d2h = e2e_pipelined(dev, dist, K, sets[:2], inp,
                                         lambda st, idx, stream_ptr: fn(refs[idx], stream_ptr),
                                         ins=[("x_base", inp["x_base"])], outs=["out"])
        e2e = {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "double-buffered: step i+1's upload and step i-1's download overlap step i"}
    if rank != 0:
        return 0
    nbytes = wl.prefill_algorithmic_bytes(w)
    peak, peak_kind = measured_peak()
    achieved = nbytes / (step_us * 1e-6) / 1e9
    traffic, traffic_src = profile_traffic(w.name, "prefill")
    line = {
        "metric": METRIC, "value": round(step_us, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": prefill_config(w), "l2_sets": l2_note,
        "prefill_us": round(step_us, 3), "prefill_gbs": round(achieved, 1), "prefill_algorithmic_bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": "prefill_conv",
                     "peak_source": f"{peak_kind} hbm_gbs (copy)", "traffic_source": traffic_src},
        "gpu_launches": K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        times = oracle_prefill_times(w, 20, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": round(statistics.median(times) * 1e6, 1), "unit": UNIT, "cores": 1,
                                "kind": "oracle",
                                "sample": f"whole workload ({w.total_tokens} tokens) per step, median of {len(times)} "
                                          f"steps; plain C loop, one thread"}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- bandwidth probe

PROBE_MIXES = [(1, 0), (0, 1), (1, 1), (2, 1), (1, 2), (10, 19), (1, 3)]


def run_probe_mix(args):
    """HBM bandwidth of read:write mixes (libcvprobe.so, 16-byte vector streams): the roofline the
    verify's own mix (about 1:1.9) can reach, against the 1:1 copy of the measured peak.  Each mix is
    timed like the verify: K launches back to back between two CUDA events, every launch on the
    next of several buffer sets totalling >= 4x L2, each launch moving `--probe-mb` MB.  Prints one
    JSON line per mix."""
    from spec_decode_verify_gb300 import build as cvbuild
    cvbuild.build()
    lib = ctypes.CDLL(cvbuild.PROBE_LIB)
    lib.cv_probe_mix.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.cv_probe_mix.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20
    threads = 256
    sp = torch.cuda.current_stream(dev).cuda_stream
    sink = torch.empty(sms * 2048 * 16, dtype=torch.uint8, device=dev)
    peak, peak_kind = measured_peak()
    sampler = ClockSampler(dev.index, args.clocks_csv)
    sampler.start()
    lines = []
    mixes = PROBE_MIXES if not args.probe_mixes else [tuple(int(v) for v in m.split(":")) for m in args.probe_mixes.split(",")]
    sizes = [float(v) for v in str(args.probe_mb).split(",")]
    bpsms = [int(v) for v in str(args.probe_bpsm).split(",")]
    for (r, w), mb, bpsm in [(m, mb, b) for m in mixes for mb in sizes for b in bpsms]:
        blocks = sms * bpsm
        unit = 16 * (r + w)
        n_units = int(mb * 1e6) // unit
        per_set = n_units * unit
        n_sets = max(2, math.ceil(4 * l2 / per_set))
        sets = [(torch.empty(max(r, 1) * n_units * 16, dtype=torch.uint8, device=dev),
                 torch.empty(max(w, 1) * n_units * 16, dtype=torch.uint8, device=dev)) for _ in range(n_sets)]
        for src, dst in sets:
            src.random_(0, 256)

        def launch(i):
            src, dst = sets[i % n_sets]
            rc = lib.cv_probe_mix(src.data_ptr(), dst.data_ptr(), n_units, r, w, blocks, threads, sink.data_ptr(), sp)
            if rc != 0:
                raise RuntimeError(f"cv_probe_mix({r},{w}) failed: CUDA error {rc}")

        for i in range(max(args.warmup, 3) * n_sets):
            launch(i)
        torch.cuda.synchronize(dev)
        K = args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(min(2e9, 40000 * K + 2e6)))
        e0.record()
        for i in range(K):
            launch(i)
        e1.record()
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / K
        gbs = per_set / (us * 1e-6) / 1e9
        lines.append({"probe": "mix", "read": r, "write": w, "bytes_per_launch": per_set, "us_per_launch": round(us, 3),
                      "gbs": round(gbs, 1), "frac_of_copy_peak": round(gbs / peak, 4), "peak": peak,
                      "peak_source": f"{peak_kind} hbm_gbs (copy)", "grid": [blocks, threads], "sets": n_sets,
                      "steps": K})
        del sets
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    for ln in lines:
        ln["clocks"] = clocks
        print(json.dumps(ln), flush=True)
    return 0


def run_probe_link(args):
    """Host-link rate of the end-to-end copies: the benchmark workload's upload (x) and download (out)
    sizes between pinned host buffers and the device, by the copy engines as the end-to-end loop
    issues them, each direction alone and both at once on two streams, K copies back to back between
    two CUDA events.  Prints one JSON line per case."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[wl.BENCH_WORKLOAD]
    n = w.n_seq * w.T * w.dim * w.esize  # x rows up, out rows down
    hs = [torch.empty(n, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ho = [torch.empty(n, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ds = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    do = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def h2d(i):
        with torch.cuda.stream(up):
            ds[i % 2].copy_(hs[i % 2], non_blocking=True)

    def d2h(i):
        with torch.cuda.stream(down):
            ho[i % 2].copy_(do[i % 2], non_blocking=True)

    def both(i):
        h2d(i)
        d2h(i)

    for name, fn, dirs in (("h2d", h2d, 1), ("d2h", d2h, 1), ("both", both, 2)):
        for i in range(max(args.warmup, 3)):
            fn(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        e0.record(cur)
        up.wait_event(e0)
        down.wait_event(e0)
        for i in range(args.steps):
            fn(i)
        for st in (up, down):
            ev = torch.cuda.Event()
            ev.record(st)
            cur.wait_event(ev)
        e1.record(cur)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        print(json.dumps({"probe": "link", "copies": name, "bytes_per_direction": n, "us_per_step": round(us, 2),
                          "gbs_per_direction": round(n / us / 1e3, 1), "steps": args.steps}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.BENCH_WORKLOAD,
                    choices=wl.WORKLOAD_ORDER + wl.RAGGED_ORDER + wl.PREFILL_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clocks-csv", default=None, help="keep the raw nvidia-smi clock samples in this file")
    ap.add_argument("--clock-probe-s", type=float, default=1.5)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--probe-mix", action="store_true",
                    help="time read:write bandwidth mixes (the verify's roofline) instead of the path")
    ap.add_argument("--probe-mb", default="75.4", help="MB moved per probe launch (comma list)")
    ap.add_argument("--probe-bpsm", default="8", help="probe blocks of 256 threads per SM (comma list)")
    ap.add_argument("--probe-mixes", default="", help="read:write mixes to time, e.g. 10:19,1:1 (default: all)")
    ap.add_argument("--probe-link", action="store_true",
                    help="time the end-to-end copies' host-link rate (the e2e number's ceiling) instead of the path")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.probe_mix:
        return run_probe_mix(args)
    if args.probe_link:
        return run_probe_link(args)
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus)
    if int(os.environ.get("WORLD_SIZE", "1")) != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE {os.environ.get('WORLD_SIZE')}")
    world, rank, local, dist = dist_setup()
    try:
        if args.workload in wl.PREFILL_WORKLOADS:
            w = wl.PREFILL_WORKLOADS[args.workload]
            if args.impl == "reference":
                return run_reference_prefill(args, w, world, rank)
            return run_ours_prefill(args, w, world, rank, local, dist)
        w = wl.WORKLOADS[args.workload] if args.workload in wl.WORKLOADS else wl.RAGGED_WORKLOADS[args.workload]
        if args.impl == "reference":
            return run_reference(args, w, world, rank)
        return run_ours(args, w, world, rank, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
