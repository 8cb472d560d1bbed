#!/usr/bin/env python
"""Benchmark: SSD forward+backward tokens/s of the Mamba2 mixer core on GB300.

One step = ssd_forward + ssd_backward (every kernel of the hot path: conv+SiLU,
dt/cumsum, chunk contractions, segment summaries, exclusive segment scan,
correction/output, and the backward mirror) over one batch of the
"mamba2-1b-fwdbwd" workload: batch 4, L 8192, H 64, P 64, N 128, G 1,
chunk 256, 8 segments, bf16 activations, seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--segments S]

Other workloads: "mamba2-1b-fwd" times the forward alone (same shape),
"long-131k" (b1 L131072 G8, --segments 1..16) and "packed-32k" (packed
sequences) time forward+backward.

Prints ONE JSON line (rank 0).  With N > 1 (torchrun) every rank runs its own
batch (weak scaling, no data-path collective); the timed region is bracketed by
a barrier and a device synchronise, and the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle on host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mamba2_ssd_selective_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "SSD fwd+bwd tokens/s on 1 GB300 (L=8192, bf16) + % of tensor/HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mamba2-1b-fwdbwd"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SM_COUNT, FP32_LANES_PER_SM = 152, 128


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def aggregate(elapsed_s: float, units: float, ws: int) -> tuple[float, float]:
    """(max elapsed over ranks, sum of units over ranks).  Timing bookkeeping only."""
    if ws == 1:
        return elapsed_s, units
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- peaks / clocks

def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc = gpu, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- algorithmic work per kernel launch

def kernel_work(shape, dtype: str) -> dict:
    """name -> (engine, algorithmic flops, algorithmic bytes) per launch.

    flops count the causal products a contraction has to do (the masked upper
    triangle of the intra-chunk products is not counted); bytes count every
    tensor the kernel must read or write once, for the kernel decomposition this
    library uses (its intermediates -- CB, chunk states, W, per-head dB/dC
    partials -- are part of that decomposition)."""
    b, L, H, P, N, G, Q, S = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                              shape.chunk, shape.n_segments)
    eb = 2 if dtype == "bf16" else 4
    nc, Cd, HP, GN = L // Q, shape.conv_dim, H * P, G * N
    tri = Q * (Q + 1) // 2
    PN = P * N
    nti = max(Q // 128, 1)
    tiles = nti * (nti + 1) // 2  # causal 128 x 128 blocks per chunk
    x = b * L * HP * eb
    bc = b * L * GN * eb
    cb = b * nc * G * tiles * 128 * 128 * 4
    st = b * nc * H * PN * 4  # one (b, chunk, head) state array
    st16 = st // 2  # the same in bf16
    seg = b * S * H * PN * 4
    tok = b * H * L * 4
    hpg = H // G
    hb = next((v for v in (16, 8, 4, 2) if hpg % v == 0), 1)
    parts = b * L * (H // hb) * N * 4  # one fp32 dB or dC partial per token and head block
    f_state = b * nc * H * 2 * P * N * Q
    f_cb = b * nc * G * tri * 2 * N
    f_diag = b * nc * H * tri * 2 * P        # (CB o L o dt) X, dM, M^T dy: causal Q x Q x P
    f_off = b * nc * H * 2 * Q * N * P       # one Q x N x P product per chunk and head
    f_bc = b * nc * H * tri * 2 * N          # W B or W^T C: causal Q x Q x N
    w = {
        # the conv forward's launch also runs the dt preparation (dt_raw in; dt, Acs out)
        "conv_fwd": ("mem", 0, b * L * Cd * 2 * eb + b * L * H * (eb + 8)),
        "decay_tables": ("mem", 0, tok + 3 * b * H * nc * 4),
        # bf16 tensor-core path: the local pass only reduces (its combine re-forms the local states)
        "local_pass": ("mem", 0, (st if dtype == "bf16" else 2 * st) + seg),
        "seg_scan": ("mem", 0, 2 * seg + b * H * PN * 4),
        "combine_state": ("mem", 0, st + st16 + seg),
        # Z in, and the local gradients out only when the backward combine does not
        # re-form them itself (bf16 path with up to 8 chunks per segment)
        "local_rev": ("mem", 0, (1 if (dtype == "bf16" and nc // S <= 8) else 2) * st + seg),
        "seg_rscan": ("mem", 0, 2 * seg),
        # bf16 path: the states' decay term (combine_bwd) and dy . x (tc_bwd_col) come precomputed
        "chunk_dt": ("mem", 0, 8 * tok + (0 if dtype == "bf16" else 4 * st + 2 * x) + 2 * b * L * H * eb),
        "combine_bwd": ("mem", 0, 2 * st + 2 * seg + 2 * st16 + b * nc * H * 4 * ((P * N + 2047) // 2048)),
        # the B / C channels' gradients come as head-block partials, summed while staging
        "conv_bwd": ("mem", 0, b * L * (Cd * 2 * eb + HP * 4) + 2 * parts + b * (L // 128) * Cd * 20),
        "param_reduce": ("mem", 0, b * nc * H * 12 + b * (L // 128) * Cd * 20),
        # bf16 path: the state kernel also forms the decay tables (Acs at chunk ends in, three tables out)
        "tc_chunk_state": ("tensor", f_state, x + bc + st + 4 * b * H * nc * 4),
        "tc_chunk_z": ("tensor", f_state, x + bc + st),
        # persistent kernels: CB is formed on chip, W never leaves the SM
        "tc_chunk_out": ("tensor", f_cb + f_diag + f_off, 2 * x + bc + st16 + 2 * tok),
        "tc_bwd_row": ("tensor", f_cb + f_diag + f_bc + 2 * f_off, 2 * x + bc + st16 + 4 * tok + parts),
        "tc_bwd_col": ("tensor", f_cb + 2 * f_diag + f_bc + 2 * f_off,
                       2 * x + bc + st16 + 5 * tok + parts + b * L * HP * 4),
    }
    # fp32 CUDA-core kernels: the same work with CB, chunk states and W through HBM
    wbytes = b * nc * H * tiles * 128 * 128 * 4
    w.update({
        "cb": ("alu", f_cb, 2 * bc + cb),
        "chunk_state": ("alu", f_state, x + bc + st),
        "chunk_out": ("alu", f_diag + f_off, 2 * x + bc + cb + st + seg),
        "chunk_z": ("alu", f_state, x + bc + st),
        "chunk_w": ("alu", f_diag, 2 * x + cb + wbytes + 3 * tok),
        "chunk_dx": ("alu", f_diag + f_off, cb + x + bc + st + seg + b * L * HP * 4),
        "chunk_dcdb": ("alu", 2 * f_bc + 2 * f_off, wbytes + 2 * x + 2 * bc + 2 * st + 2 * seg + 2 * b * L * H * N * 4),
    })
    return w


def method_work(shape, dtype: str) -> dict:
    """The method's own work per token, independent of how this library splits it
    into kernels: every input read and every output written once per pass
    (forward: xBC, dt in, y out; backward: xBC, dt, dy in, dxBC, ddt out), and
    the chunked algorithm's flops counting only the causal half of the Q x Q
    products, with CB and the dB/dC diagonal products once per group and dM
    once.  Also the share of those flops each tensor-core kernel carries."""
    H, P, N, G, Q = shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.chunk
    eb = 2 if dtype == "bf16" else 4
    Cd, HP = shape.conv_dim, H * P
    gqn, hpq, hpn2 = G * Q * N, H * P * Q, 2 * H * P * N  # causal CB, causal Q x Q x P, one P x N contraction
    per_kernel = {
        "tc_chunk_out": gqn + hpq + hpn2,           # CB, (CB o L o dt) X, C S_in^T
        "tc_chunk_state": hpn2,                     # chunk states (forward, and the backward's recompute)
        "tc_chunk_z": hpn2,                         # Z = C^T (em dy)
        "tc_bwd_row": 2 * gqn + hpq + hpn2,         # CB, dM, (sum_h W) B, (em dy) S_in
        "tc_bwd_col": gqn + hpq + 2 * hpn2,         # M^T dy, (sum_h W)^T C, B dS^T, (wdt x) dS
    }
    return {
        "fwd_bytes": (Cd + H + HP) * eb, "bwd_bytes": (Cd + H + HP) * eb + (Cd + H) * eb,
        "fwd_flop": gqn + hpq + 2 * hpn2, "bwd_flop": 3 * gqn + 2 * hpq + 5 * hpn2,
        "per_kernel_flop_per_token": per_kernel,
    }


def method_roofline(kt: list, shape, dtype: str, ms_per_step: float, peaks: dict, backward: bool) -> dict:
    """The step against the method's own minimum: its bytes at the measured HBM
    copy bandwidth and its causal flops at the sustained bf16 tensor peak.  The
    step floor is the larger of the two times; frac = floor / measured step."""
    m = method_work(shape, dtype)
    tok = shape.tokens
    bpt = m["fwd_bytes"] + (m["bwd_bytes"] if backward else 0)
    fpt = m["fwd_flop"] + (m["bwd_flop"] if backward else 0)
    hbm, tpk = peaks["hbm_gbs"], peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    t_b, t_f = bpt * tok / (hbm * 1e9), fpt * tok / (tpk * 1e12)
    floor_ms = max(t_b, t_f) * 1e3
    out = {"bytes_per_token": bpt, "flop_per_token": fpt, "bytes_per_step": bpt * tok, "flop_per_step": fpt * tok,
           "bound": "hbm" if t_b >= t_f else "tensor", "floor_ms": round(floor_ms, 4),
           "frac": round(floor_ms / ms_per_step, 4)}
    tc = [r for r in kt if r[0] in m["per_kernel_flop_per_token"]]
    if tc:
        name, launches, total_ms = max(tc, key=lambda r: r[2] / max(r[1], 1))
        avg_s = total_ms / 1e3 / max(launches, 1)
        f = m["per_kernel_flop_per_token"][name] * tok  # every launch covers all tokens
        ach = f / avg_s / 1e12
        out["dominant_contraction"] = {"kernel": name, "method_flop_per_launch": f, "avg_launch_ms": round(avg_s * 1e3, 4),
                                       "achieved_tflops": round(ach, 2), "peak_tflops": tpk,
                                       "frac_compute": round(ach / tpk, 4)}
    return out


def roofline_for(kt: list, shape, dtype: str, peaks: dict, peak_src: str, clocks: dict | None) -> dict:
    """Roofline of the kernel with the largest share of the step.  Kernels are
    timed inside the step, so the tensor peak is the sustained one."""
    work = kernel_work(shape, dtype)
    name, launches, total_ms = max(kt, key=lambda r: r[2])
    engine, flops, nbytes = work.get(name, ("mem", 0, 0))
    avg_s = total_ms / 1e3 / max(launches, 1)
    hbm = peaks["hbm_gbs"]
    if engine == "tensor":
        cpeak, cnote = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), f"dense bf16 sustained ({peak_src})"
    else:  # fp32 FMA pipe: 152 SMs x 128 lanes x 2 flop x max SM clock
        mhz = peaks.get("sm_max_mhz", 2070.0)
        cpeak, cnote = SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, f"fp32 FMA pipe at {mhz:.0f} MHz (derived)"
    t_flop = flops / (cpeak * 1e12) if flops else 0.0
    t_byte = nbytes / (hbm * 1e9)
    frac_c = flops / avg_s / 1e12 / cpeak if flops else None
    frac_m = nbytes / avg_s / 1e9 / hbm
    if engine == "mem" or t_byte >= t_flop:
        bound, achieved, peak, unit, note = "hbm", nbytes / avg_s / 1e9, hbm, "GB/s", f"HBM copy bandwidth ({peak_src})"
        amount = nbytes
    else:
        bound = "tensor" if engine == "tensor" else "alu"
        achieved, peak, unit, note, amount = flops / avg_s / 1e12, cpeak, "TFLOP/s", cnote, flops
    return {"bound": bound, "kernel": name, "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": committed_traffic(name, shape),
            "peak_source": note, "algorithmic_per_launch": amount, "avg_launch_ms": round(avg_s * 1e3, 4),
            "frac_hbm": round(frac_m, 4), "frac_compute": None if frac_c is None else round(frac_c, 4)}


def step_totals(kt: list, shape, dtype: str, ms_per_step: float, peaks: dict, steps: int) -> dict:
    """Whole-step algorithmic work of this decomposition against the peaks
    (all kernels; kt covers `steps` steps)."""
    work = kernel_work(shape, dtype)
    flops = sum(work.get(n, ("mem", 0, 0))[1] * c for n, c, _ in kt) / steps
    nbytes = sum(work.get(n, ("mem", 0, 0))[2] * c for n, c, _ in kt) / steps
    s = ms_per_step / 1e3
    return {"tensor_tflops": round(flops / s / 1e12, 2),
            "frac_tensor_sustained": round(flops / s / 1e12 / peaks.get("bf16_tflops_sustained", 1742.8), 4),
            "hbm_gbs": round(nbytes / s / 1e9, 1), "frac_hbm": round(nbytes / s / 1e9 / peaks["hbm_gbs"], 4),
            "flop_per_step": flops, "bytes_per_step": nbytes}


def committed_traffic(kernel: str, shape):
    """DRAM bytes per launch from the committed ncu summary, scaled from the
    captured batch to this workload's batch, if it was taken on the current
    sources of the kernel (its file and the headers it is built from);
    otherwise None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(kernel)
    if not e:
        return None
    h = hashlib.sha256()
    for rel in e["sources"]:
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != e["sources_sha256"]:
        return None
    return int(e["dram_bytes_per_launch"] * shape.batch / e.get("captured_batch", shape.batch))


# ---------------------------------------------------------------- CPU oracle timings

def oracle_sample(inp: dict, shape, heads: tuple, nthreads: int = 0, backward: bool = True) -> float:
    import oracle

    t0 = time.perf_counter()
    oracle.forward(inp, shape, heads=heads, rows=[0], nthreads=nthreads)
    if backward:
        oracle.backward(inp, shape, heads=heads, rows=[0], nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(inp: dict, shape, backward: bool) -> dict:
    import oracle

    oracle.build()
    cores = oracle.default_threads()
    what = "fwd + bwd" if backward else "fwd"
    dt = oracle_sample(inp, shape, (0, shape.nheads), backward=backward)
    out = {"value": round(shape.seqlen / dt, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"fp64 C oracle, {what} (S={shape.n_segments}) of batch row 0 (all {shape.nheads} heads, "
                     f"{shape.seqlen} tokens) of the same workload, {cores} threads: {dt:.1f} s"}
    if not backward:  # the forward on one host core as well
        dt1 = oracle_sample(inp, shape, (0, shape.nheads), nthreads=1, backward=False)
        out["one_thread"] = {"value": round(shape.seqlen / dt1, 2), "unit": UNIT, "cores": 1, "seconds": round(dt1, 2)}
    return out


def run_reference(args, shape, dtype, seed, backward: bool):
    """The oracle as it stands, on the host cores: each step is batch row 0 of
    the workload (all heads), the same sample as the line's cpu_baseline."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    cores = oracle.default_threads()
    inp = make_inputs(shape, seed, dtype)
    heads = (0, shape.nheads)
    for _ in range(args.warmup):
        oracle_sample(inp, shape, heads, backward=backward)
    times = [oracle_sample(inp, shape, heads, backward=backward) for _ in range(args.steps)]
    total = sum(times)
    value = shape.seqlen * args.steps / total
    what = "fwd + bwd" if backward else "fwd"
    line = {
        "impl": "reference", "metric": metric_for(args, backward), "value": round(value, 2), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3),
        "ms_per_step_p50": round(statistics.median(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args, shape, dtype, seed),
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 C oracle {what} of batch row 0 (all {shape.nheads} heads, "
                                   f"{shape.seqlen} tokens) of the workload, {cores} threads"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def metric_for(args, backward: bool) -> str:
    if (args.workload == DEFAULT_WORKLOAD and args.segments is None and args.batch is None and args.chunk is None
            and not args.gated_norm):
        return METRIC
    what = "fwd+bwd" if backward else "fwd"
    norm = " + gated RMSNorm" if args.gated_norm else ""
    return f"SSD {what}{norm} tokens/s on 1 GB300 ({args.workload}, bf16) + % of tensor/HBM roofline"


def config_dict(args, shape, dtype, seed) -> dict:
    eb = 2 if dtype == "bf16" else 4
    return {"workload": args.workload, "batch": shape.batch, "seqlen": shape.seqlen, "nheads": shape.nheads,
            "headdim": shape.headdim, "dstate": shape.dstate, "ngroups": shape.ngroups, "d_conv": shape.d_conv,
            "chunk": shape.chunk, "n_segments": shape.n_segments, "packed": shape.packed, "activations": dtype,
            "gated_norm": bool(args.gated_norm), "seed": seed,
            "l2": f"inputs larger than L2 (xBC {shape.tokens * shape.conv_dim * eb / 1e6:.0f}"
                  f" MB, dy {shape.tokens * shape.nheads * shape.headdim * eb / 1e6:.0f}"
                  f" MB per step; L2 is 129 MB)"}


# ---------------------------------------------------------------- our arm

def run_ours(args, shape, dtype, seed, backward: bool):
    import mamba2_ssd_selective_gb300 as ssd
    from mamba2_ssd_selective_gb300.build import build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(ws, "nccl")
    if rank == 0:
        build()
    barrier(ws)
    if rank != 0:
        build()  # stamp is current: only loads
    ssd.load()
    inp = make_inputs(shape, seed + 1000 * rank, dtype, gated_norm=args.gated_norm)
    t = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    runner = ssd.SsdRunner(shape, dtype, gated_norm=args.gated_norm)
    y, fin, seg = runner.alloc_outputs()
    grads = runner.alloc_grads()
    dfinal = None
    stream = torch.cuda.current_stream()

    def step():
        runner.forward(t, out=(y, fin, seg))
        if backward:
            runner.backward(t, t["dy"], dfinal, seg, grads=grads)

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler.start()
    # timed region 1: throughput over exactly K steps, with an event between
    # steps for the per-step median
    barrier(ws)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for k in range(args.steps):
        step()
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed = ev[0].elapsed_time(ev[-1]) / 1e3
    step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(args.steps)]
    # timed region 2: the same steps with per-kernel events on the launch stream
    ssd.ssd_profile_begin()
    for _ in range(args.steps):
        step()
    kt = ssd.ssd_profile_end()
    torch.cuda.synchronize()
    # end to end through the public API with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        in_keys = ("xBC", "dt_raw", "dy") if backward else ("xBC", "dt_raw")
        if args.gated_norm:
            in_keys += ("z",)
        host_in = {k: inp[k].pin_memory() for k in in_keys}
        host_out = {"y": torch.empty(y.shape, dtype=y.dtype).pin_memory(),
                    "final_state": torch.empty(fin.shape, dtype=fin.dtype).pin_memory()}
        if backward:
            host_out.update({k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in grads.items()})
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())

        # Two device copies of the inputs and outputs: step k's upload (copy stream
        # `up`) and step k-1's download (copy stream `down`) overlap the compute of
        # the neighbouring step.  Every step still uploads its own inputs from the
        # pinned host buffers and downloads its results inside the timed region.
        tb = [t, {k: (v.clone() if torch.is_tensor(v) else v) for k, v in t.items()}]
        y2, fin2, seg2 = runner.alloc_outputs()
        ob = [(y, fin, seg, grads), (y2, fin2, seg2, runner.alloc_grads())]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_steps(n, start_event=None):
            if start_event is not None:
                up.wait_event(start_event)
            for k in range(n):
                sl = k % 2
                ti, (yo, fo, so, go) = tb[sl], ob[sl]
                with torch.cuda.stream(up):
                    if k >= 2:
                        up.wait_event(ev_done[sl])  # step k-2 no longer reads this slot
                    for key, v in host_in.items():
                        ti[key].copy_(v, non_blocking=True)
                    ev_in[sl].record(up)
                stream.wait_event(ev_in[sl])
                if k >= 2:
                    stream.wait_event(ev_out[sl])  # step k-2's results were read back
                runner.forward(ti, out=(yo, fo, so))
                if backward:
                    runner.backward(ti, ti["dy"], dfinal, so, grads=go)
                ev_done[sl].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[sl])
                    host_out["y"].copy_(yo, non_blocking=True)
                    host_out["final_state"].copy_(fo, non_blocking=True)
                    if backward:
                        for key, v in go.items():
                            host_out[key].copy_(v, non_blocking=True)
                    ev_out[sl].record(down)
            stream.wait_event(ev_out[(n - 1) % 2])  # the last download is inside the region

        e2e_steps(max(2, args.warmup))
        torch.cuda.synchronize()
        barrier(ws)
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        e2e_steps(args.steps, start_event=e2)
        e3.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        el2, units2 = aggregate(e2.elapsed_time(e3) / 1e3, shape.tokens * args.steps, ws)
        e2e = {"value": round(units2 / el2, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    clocks = sampler.stop()  # sampled through the timed, the profiled and the end-to-end passes
    el, units = aggregate(elapsed, shape.tokens * args.steps, ws)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    ms = el / args.steps * 1e3
    line = {
        "metric": metric_for(args, backward), "value": round(units / el, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "ms_per_step_p50": round(statistics.median(step_ms), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": config_dict(args, shape, dtype, seed),
        "roofline": roofline_for(kt, shape, dtype, peaks, peak_src, clocks),
        "method_roofline": method_roofline(kt, shape, dtype, ms, peaks, backward),
        "step_roofline": step_totals(kt, shape, dtype, ms, peaks, args.steps),
        "e2e": e2e,
        "gpu_launches": int(sum(r[1] for r in kt)),
        "clocks": clocks,
        "kernels": [{"name": n, "launches": c, "ms_per_launch": round(ms_ / max(c, 1), 4),
                     "share": round(ms_ / max(sum(r[2] for r in kt), 1e-9), 4)} for n, c, ms_ in kt],
    }
    if ws == 1 and not args.no_cpu_baseline and not args.gated_norm:
        line["cpu_baseline"] = cpu_baseline(inp, shape, backward)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--segments", type=int, default=None, help="override the workload's segment count")
    ap.add_argument("--chunk", type=int, default=None, help="override the workload's chunk length")
    ap.add_argument("--gated-norm", action="store_true", help="y is the gated RMSNorm of the mixer output")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 untimed warm-up steps
    shape, dtype, seed = WORKLOADS[args.workload]
    if args.batch is not None:
        shape = shape.with_(batch=args.batch)
    if args.segments is not None:
        shape = shape.with_(n_segments=args.segments)
    if args.chunk is not None:
        shape = shape.with_(chunk=args.chunk)
    backward = args.workload != "mamba2-1b-fwd"  # that workload is the forward alone
    if args.impl == "reference":
        run_reference(args, shape, dtype, seed, backward)
    else:
        run_ours(args, shape, dtype, seed, backward)
    ws, _, _ = dist_env()
    if ws > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
