#!/usr/bin/env python
"""Throughput of the S5 layer forward hot path on GB300.

One step = zero-order-hold discretisation (s5_discretize) + the fused forward
(s5_forward: projection, chunked scan with decoupled look-back, readout) over
one batch of the long-sequence workload (B=8, L=16384, H=128, P=128, bf16
u/y; the Path-X sequence length), with inputs resident in HBM.  Four
input/output sets (4 x 67 MB > 129 MB L2) rotate between steps so that every
step reads u from HBM.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the float64 CPU
oracle on the same workload instead (bounded sample per step).

Multi-GPU: replicas only.  Each rank runs an independent copy of the
workload (sequences are independent; the layer needs no exchange), the timed
region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "S5 layer fwd tokens/s (batch*L/s) and fraction of HBM/tensor roofline"
BIDI_METRIC = "S5 bidirectional layer fwd tokens/s (batch*L/s) and fraction of HBM/tensor roofline"
STREAM_METRIC = "S5 streaming step tokens/s (batch tokens per step call / call time)"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000; 20 for the streaming workload, whose step "
                         "is 1024 calls)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 50; 3 for stream)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="pathx_bf16",
                    choices=["small", "fp32", "pathx_bf16", "pathx_bf16_bidir", "pathx_bf16_bilinear",
                             "stream", "irregular", "stack6"])
    ap.add_argument("--e2e-steps", type=int, default=None, help="end-to-end steps (default 30; 3 for stream)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    stream = args.workload == "stream"
    if args.steps is None:
        args.steps = 20 if stream else 2000
    if args.warmup is None:
        args.warmup = 3 if stream else 50
    if args.e2e_steps is None:
        args.e2e_steps = 3 if stream else 30
    return args


# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, dist, device="cuda"):
    """The slowest rank's time: the job is done when its last replica is."""
    if not dist:
        return ms
    import torch
    tt = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(units_per_rank, world, ms):
    """Whole-job rate: every rank's units over the slowest rank's time (ms)."""
    return units_per_rank * world / (ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk.get("bf16_tflops", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch):
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def traffic_for(kernel: str, source: str, workload: str):
    """ncu DRAM bytes per launch recorded for this kernel on this workload, if
    its source is unchanged since the capture (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(kernel)
        sha = hashlib.sha256(open(source, "rb").read()).hexdigest()
        if rec and rec.get("source_sha256") == sha and rec.get("workload", "").split(" ")[0] == workload:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
def algorithmic_bytes(w, u_bytes_per, y_bytes_per):
    params = 8 * w.P + 8 * w.P * w.H * 2 + 4 * w.H
    if w.varying_dt:
        params += 4 * w.P + 4 * w.B * w.L      # log_dt and the gaps
    if w.bidirectional:
        params += 8 * w.P * w.H                # the backward half of C~
    return w.B * w.L * w.H * (u_bytes_per + y_bytes_per) + params


# Nominal dense TF32 : BF16 tensor rates on GB300 (1.1 : 2.25 PFLOP/s); the
# fp32 workloads' tensor peak is the measured bf16 peak scaled by it.
TF32_PER_BF16 = 1.1 / 2.25


def projection_flops(w):
    """Flops of the two dense projections per launch: B_bar u (complex [P,H]
    times real u: 4PH per token) and 2 Re(C~ x) (4PH per token; twice that
    for the bidirectional readout, whose C~ has 2P columns)."""
    per_token = 4 * w.P * w.H + (8 if w.bidirectional else 4) * w.P * w.H
    return w.B * w.L * per_token


def layer_roofline(w, launch_s, kname, traffic, clocks, num_sms, u_bytes, simt):
    """The roofline of one layer launch: its time bound is the larger of the
    algorithmic HBM bytes at the measured copy rate and the projection flops
    at the measured tensor rate (bf16 projections: bf16; fp32 ones: TF32),
    and frac = that bound / the measured launch time.  The other term and,
    for the CUDA-core kernel, the FP32 FMA-pipe fraction are diagnostics."""
    hbm_gbs, bf16_tf, peak_kind = load_peaks()
    alg = algorithmic_bytes(w, u_bytes, u_bytes)
    flops = projection_flops(w)
    tensor_tf = bf16_tf if w.proj_dtype == "bf16" else bf16_tf * TF32_PER_BF16
    t_hbm = alg / (hbm_gbs * 1e9)
    t_tensor = flops / (tensor_tf * 1e12) if tensor_tf else 0.0
    hbm_bound = t_hbm >= t_tensor
    src = ("%s (MEASURED_PEAKS.json)" % peak_kind if peak_kind == "measured"
           else "fallback 6.8 TB/s, 1.9 PFLOP/s bf16")
    r = {
        "bound": "hbm" if hbm_bound else "tensor",
        "kernel": kname,
        "achieved": alg / launch_s / 1e9 if hbm_bound else flops / launch_s / 1e12,
        "peak": hbm_gbs if hbm_bound else tensor_tf,
        "unit": "GB/s" if hbm_bound else "TFLOP/s",
        "frac": max(t_hbm, t_tensor) / launch_s,
        "peak_source": src + (": hbm_gbs" if hbm_bound else
                              ": bf16_tflops" if w.proj_dtype == "bf16" else
                              ": bf16_tflops x 1.1/2.25 (TF32)"),
        "definition": "frac = max(algorithmic bytes / HBM peak, projection flops / tensor "
                      "peak) / launch time",
        "algorithmic_bytes_per_launch": alg,
        "projection_flops_per_launch": flops,
        "hbm_frac": t_hbm / launch_s,
        "tensor_frac": t_tensor / launch_s,
        "tensor_peak_tflops": tensor_tf,
        "launch_us": launch_s * 1e6,
        "traffic": traffic,
    }
    if simt:
        # diagnostic: the FP32 FMA pipe the CUDA-core kernel runs on (SMs x
        # 128 lanes x 2 flops per FMA at the sampled SM clock)
        simt_flops = w.B * w.L * (8 * w.P * w.H + 8 * w.P + 2 * w.H)
        mhz = (clocks or {}).get("sm_mhz") or 2070.0
        alu_tf = num_sms * 128 * 2 * mhz * 1e6 / 1e12
        r.update({"alu_frac": simt_flops / launch_s / 1e12 / alu_tf, "alu_peak_tflops": alu_tf,
                  "alu_peak_source": "%d SMs (device query) x 128 lanes x 2 flops x %.0f MHz"
                                     % (num_sms, mhz)})
    return r


def parity_field(got, ref, tol, sample):
    """rel-L2 and max-abs error of the bench's own output against the oracle."""
    import numpy as np
    got = np.asarray(got, np.complex128 if np.iscomplexobj(got) else np.float64)
    ref = np.asarray(ref, np.complex128 if np.iscomplexobj(ref) else np.float64)
    err = got - ref
    rel = float(np.linalg.norm(err) / np.linalg.norm(ref))
    return {"rel_l2": rel, "max_abs": float(np.max(np.abs(err))),
            "max_abs_ref": float(np.max(np.abs(ref))), "tol_rel_l2": tol, "pass": rel <= tol,
            "sample": sample}


def graph_event(torch):
    """A timing event that can be recorded inside a CUDA graph capture."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:      # torch without external events: plain timing events
        return torch.cuda.Event(enable_timing=True)


def run_ours(args):
    import numpy as np
    import torch

    from diagonal_state_space_gb300 import api
    from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    u_dt = torch.bfloat16 if w.u_dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    lam, log_dt = dev(inp["lambda_"]), dev(inp["log_dt"])
    bt, ct, d = dev(inp["b_tilde"]), dev(inp["c_tilde"]), dev(inp["d"])
    g = dev(inp["g"]) if w.varying_dt else None
    ct2 = dev(inp["c_tilde2"]) if w.bidirectional else None
    NSETS = 4
    u_sets = [dev(inp["u"]).to(u_dt) for _ in range(NSETS)]
    y_sets = [torch.empty_like(u_sets[0]) for _ in range(NSETS)]
    lb = torch.empty(w.P, dtype=torch.complex64, device="cuda")
    bb = torch.empty(w.P, w.H, dtype=torch.complex64, device="cuda")
    if w.bidirectional:
        ws = torch.zeros(api.s5_bidirectional_workspace_size(w.B, w.L, w.H, w.P, u_dt, u_dt),
                         dtype=torch.uint8, device="cuda")
    else:
        ws = api.new_workspace(w.B, w.L, w.H, w.P)
    stream = torch.cuda.current_stream()

    tc_path = (w.u_dtype == "bf16" and w.proj_dtype == "bf16" and w.H == 128 and w.P == 128
               and not w.varying_dt)
    fwd_ev = []

    new_event = lambda: graph_event(torch)

    def discretize(lam_, log_dt_, bt_):
        if w.method == "zoh" and w.clip_re == 0.0 and w.dt_scale == 1.0:
            return api.s5_discretize(lam_, log_dt_, bt_, lb, bb)
        return api.s5_discretize_ex(lam_, log_dt_, bt_, method=w.method, clip_re=w.clip_re,
                                    dt_scale=w.dt_scale, lambda_bar=lb, b_bar=bb)

    def step(i, timed):
        u, y = u_sets[i % NSETS], y_sets[i % NSETS]
        if not w.varying_dt:
            discretize(lam, log_dt, bt)
        if timed:
            e0, e1 = new_event(), new_event()
            e0.record()
        if w.varying_dt:
            api.s5_forward_varying_dt(lam, log_dt, bt, ct, d, g, u, y=y, proj_dtype=w.proj_dtype,
                                      workspace=ws)
        elif w.bidirectional:
            api.s5_forward_bidirectional(lb, bb, ct2, d, u, y=y, proj_dtype=w.proj_dtype, workspace=ws)
        else:
            api.s5_forward(lb, bb, ct, d, u, y=y, proj_dtype=w.proj_dtype, workspace=ws)
        if timed:
            e1.record()
            fwd_ev.append((e0, e1))

    for i in range(max(3, args.warmup)):
        step(i, False)
    torch.cuda.synchronize()
    st = api.s5_sync_status(ws)
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)

    # The K timed steps are captured once into a CUDA graph and replayed once:
    # host launch overhead then does not starve the GPU between ~10 us
    # kernels.  That graph has no event nodes between the steps (an event
    # node between two kernels ends the programmatic overlap of one kernel's
    # start with the previous kernel's tail); a second graph of K steps with
    # an event pair around every forward call, replayed after the timed
    # region, gives the forward call's own duration (launch_us).
    graph = graph_ev = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(i, False)
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            for i in range(args.steps):
                step(i, True)
    except Exception as exc:                      # capture unavailable: eager timed loop
        print("bench: graph capture failed (%s); timing eagerly" % exc, file=sys.stderr)
        graph = graph_ev = None
        fwd_ev.clear()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i, True)
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, dist)
    if graph_ev is not None:
        graph_ev.replay()
        torch.cuda.synchronize()
    st = api.s5_sync_status(ws)
    if st != 0:
        raise RuntimeError("device status %d after the timed region" % st)
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    fwd_avg_s = statistics.fmean(fwd_ms) / 1e3
    ms_step = ms_total / args.steps
    tokens = w.B * w.L
    value = job_throughput(tokens, world, ms_step)

    # End to end through the public API with host buffers: every step copies
    # all its inputs (u and the parameters) in from pinned host memory and its
    # output y back out, inside the timed region.  Three device buffer sets
    # and two copy streams let step i's copies overlap the compute and copies
    # of steps i-1 and i-2 -- how a caller streaming batches runs it; the
    # compute calls are the same.  The host link (~200 GB/s each way, ~326
    # GB/s both ways at once on this machine) bounds it.
    u_host = torch.from_numpy(np.ascontiguousarray(inp["u"])).to(u_dt).pin_memory()
    ESETS = 3   # device buffer sets: step i's copies overlap steps i-1 and i-2
    y_hosts = [torch.empty(u_host.shape, dtype=u_dt).pin_memory() for _ in range(ESETS)]
    # the parameters travel as one pinned block (one copy per step), each at
    # a 256-byte-aligned offset, viewed on the device with its own dtype
    names = ["lambda_", "log_dt", "b_tilde", "c_tilde2" if w.bidirectional else "c_tilde", "d"]
    if w.varying_dt:
        names.append("g")
    arrs = [np.ascontiguousarray(inp[k]) for k in names]
    offs, total = [], 0
    for arr in arrs:
        offs.append(total)
        total += (arr.nbytes + 255) // 256 * 256
    param_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for arr, o in zip(arrs, offs):
        param_host[o:o + arr.nbytes].copy_(torch.from_numpy(arr.reshape(-1).view(np.uint8)))
    tdt = {np.dtype(np.complex64): torch.complex64, np.dtype(np.float32): torch.float32}
    param_devs = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(ESETS)]
    dev_params = [[pd[o:o + arr.nbytes].view(tdt[arr.dtype]).view(arr.shape) for arr, o in zip(arrs, offs)]
                  for pd in param_devs]
    u_devs = u_sets[:ESETS]
    y_devs = y_sets[:ESETS]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(ESETS)]
    ev_cmp = [torch.cuda.Event() for _ in range(ESETS)]
    ev_out = [torch.cuda.Event() for _ in range(ESETS)]
    used = [False] * ESETS

    def e2e_step(i):
        k = i % ESETS
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(ev_cmp[k])      # set k is free once step i-ESETS has computed
            u_devs[k].copy_(u_host, non_blocking=True)
            param_devs[k].copy_(param_host, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if used[k]:
            stream.wait_event(ev_out[k])        # y set k has been read back by step i-ESETS
        dp, u_dev, y_dev = dev_params[k], u_devs[k], y_devs[k]
        if w.varying_dt:
            api.s5_forward_varying_dt(*dp[:5], dp[5], u_dev, y=y_dev, proj_dtype=w.proj_dtype,
                                      workspace=ws)
        else:
            l_, b_ = discretize(dp[0], dp[1], dp[2])
            if w.bidirectional:
                api.s5_forward_bidirectional(l_, b_, dp[3], dp[4], u_dev, y=y_dev,
                                             proj_dtype=w.proj_dtype, workspace=ws)
            else:
                api.s5_forward(l_, b_, dp[3], dp[4], u_dev, y=y_dev, proj_dtype=w.proj_dtype,
                               workspace=ws)
        ev_cmp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[k])
            y_hosts[k].copy_(y_dev, non_blocking=True)
            ev_out[k].record(s_out)
        used[k] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(3, 3 + args.e2e_steps):
        e2e_step(i)
    for ev in ev_out:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist)
    y_host = y_hosts[0]
    h2d = u_host.numel() * u_host.element_size() + param_host.numel()
    d2h = y_host.numel() * y_host.element_size()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None

    ub = 2 if w.u_dtype == "bf16" else 4
    kname = "fwd_tc_kernel" if tc_path else "fwd_simt_kernel"
    src = os.path.join(ROOT, "diagonal_state_space_gb300", "csrc",
                       "s5_forward_tc.cu" if tc_path else "s5_forward_simt.cu")
    traffic = traffic_for(kname, src, w.name)
    if w.bidirectional:
        # the timed call is the whole bidirectional layer: two forward launches
        # plus the split / reverse / add kernels; no single-kernel DRAM capture
        kname = ("bidirectional layer (fwd_tc_kernel + bwd_tc_kernel + split)" if tc_path else
                 "bidirectional layer (2 x %s + split, reverse, add)" % kname)
        traffic = None
    num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    roofline = layer_roofline(w, fwd_avg_s, kname, traffic, clocks, num_sms, ub, not tc_path)
    # the same bound against the whole timed step (discretisation included,
    # kernels overlapping as they do back to back)
    roofline["step_us"] = ms_step * 1e3
    roofline["step_frac"] = roofline["frac"] * fwd_avg_s / (ms_step / 1e3)
    result = {
        "metric": BIDI_METRIC if w.bidirectional else METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if tc_path else "f32",
        "data": "synthetic (seeded numpy PCG64: u~N(0,1), lambda=-1/2+i*pi*n, "
                "log_dt~U[ln1e-3,ln1e-1], B~,C~~CN(0,1/H), D~N(0,1))",
        "config": {
            "workload": "%s: S5 %slayer forward, B=%d L=%d H=%d P=%d (stored complex modes), "
                        "u/y %s, proj %s, complex fp32 scan%s" % (
                            w.name, "bidirectional " if w.bidirectional else "", w.B, w.L, w.H, w.P,
                            w.u_dtype, w.proj_dtype, ", per-step interval" if w.varying_dt else ""),
            "global_batch": w.B * world, "seq_len": w.L, "H": w.H, "P": w.P,
            "step": ("s5_forward_varying_dt" if w.varying_dt else
                     "s5_discretize + s5_forward_bidirectional" if w.bidirectional else
                     "s5_discretize + s5_forward" if w.method == "zoh" and w.clip_re == 0.0
                     and w.dt_scale == 1.0 else
                     "s5_discretize_ex(%s, clip_re=%g, dt_scale=%g) + s5_forward" % (
                         w.method, w.clip_re, w.dt_scale)),
            "arithmetic": ("bf16 tensor-core projections (fp32 accumulate), complex fp32 scan"
                           if tc_path else "fp32 CUDA-core projections, complex fp32 scan"),
            "timing": "K steps captured in one CUDA graph, replayed once between events; "
                      "launch_us from a second K-step graph with events around each forward call",
            "l2": "4 rotating input/output sets (%.0f MB > 129 MB L2)" % (
                NSETS * tokens * w.H * 2 * ub / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": roofline,
        "e2e": {"value": job_throughput(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "note": "public API, pinned host buffers (the parameters as one block); "
                        "three device sets and two copy streams overlap step i's copies with "
                        "steps i-1 and i-2"},
        # per step: discretize + (weight images + tensor-core forward | CUDA-core forward),
        # or, with per-step intervals, mode constants + CUDA-core forward
        # bidirectional, tensor-core path: discretize, split, 2 x (images + scan kernel);
        # CUDA-core path: discretize, split, reverse, 2 x forward, add
        "gpu_launches": args.steps * (6 if w.bidirectional else (3 if tc_path else 2)),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"], oy = cpu_baseline(w, inp)
        tol = 2e-2 if (w.u_dtype == "bf16" or w.proj_dtype == "bf16") else 1e-5
        result["parity"] = parity_field(y_sets[0].float().cpu().numpy(), oy, tol,
                                        "y of a bench step, all %d sequences, against the "
                                        "float64 oracle" % w.B)
    print(json.dumps(result), flush=True)
    if dist:
        dist.destroy_process_group()
    return result


def run_stream(args):
    """Streaming inference through s5_step: one bench step feeds L tokens to
    each of the B sequences, one s5_step call per token."""
    import numpy as np
    import torch

    from diagonal_state_space_gb300 import api
    from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    lam, log_dt, bt, ct, d = (dev(inp[k]) for k in ("lambda_", "log_dt", "b_tilde", "c_tilde", "d"))
    # time-major [L, B, H]: the k-th call reads and writes one contiguous [B, H] slice
    u_t = dev(np.transpose(inp["u"], (1, 0, 2)))
    y_t = torch.empty_like(u_t)
    x = torch.zeros(w.B, w.P, dtype=torch.complex64, device="cuda")
    lb, bb = api.s5_discretize(lam, log_dt, bt)
    stream = torch.cuda.current_stream()
    loop_ev = []

    def step(timed):
        api.s5_discretize(lam, log_dt, bt, lb, bb)
        if timed:
            e0, e1 = graph_event(torch), graph_event(torch)
            e0.record()
        for k in range(w.L):
            api.s5_step(lb, bb, ct, d, x, u_t[k], y=y_t[k])
        if timed:
            e1.record()
            loop_ev.append((e0, e1))

    for _ in range(max(3, args.warmup)):
        step(False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step(True)
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, dist)
    ms_step = ms_total / args.steps
    call_s = statistics.fmean(a.elapsed_time(b) for a, b in loop_ev) / 1e3 / w.L
    tokens = w.B * w.L
    value = job_throughput(tokens, world, ms_step)

    # end to end: host u in, host y out, every call through the public API
    u_host = torch.from_numpy(np.ascontiguousarray(np.transpose(inp["u"], (1, 0, 2)))).pin_memory()
    y_host = torch.empty_like(u_host).pin_memory()
    host_params = [torch.from_numpy(np.ascontiguousarray(inp[k])).pin_memory()
                   for k in ("lambda_", "log_dt", "b_tilde", "c_tilde", "d")]
    dev_params = [torch.empty_like(p, device="cuda") for p in host_params]

    def e2e_step():
        for hp, dp in zip(host_params, dev_params):
            dp.copy_(hp, non_blocking=True)
        u_t.copy_(u_host, non_blocking=True)
        l_, b_ = api.s5_discretize(dev_params[0], dev_params[1], dev_params[2], lb, bb)
        for k in range(w.L):
            api.s5_step(l_, b_, dev_params[3], dev_params[4], x, u_t[k], y=y_t[k])
        y_host.copy_(y_t, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    # The step's copies and calls are captured once in a CUDA graph, as a
    # caller streaming tokens would run them: L eager calls from Python would
    # time the interpreter, not the GPU.  Every replay copies u and the
    # parameters in and y out again.
    g_e2e = None
    try:
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_step()
    except Exception as exc:                      # capture unavailable: eager calls
        print("bench: end-to-end graph capture failed (%s); timing eagerly" % exc, file=sys.stderr)
        g_e2e = None
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        if g_e2e is not None:
            g_e2e.replay()
        else:
            e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist)
    h2d = u_host.numel() * 4 + sum(p.numel() * p.element_size() for p in host_params)
    d2h = y_host.numel() * 4
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None

    hbm_gbs, bf16_tf, peak_kind = load_peaks()
    # per call: lambda_bar, B_bar, C~, D once; the state read and written; u and y
    alg = 8 * w.P + 16 * w.P * w.H + 4 * w.H + 16 * w.B * w.P + 8 * w.B * w.H
    achieved = alg / call_s / 1e9
    # the projections of one call at the TF32 tensor rate: far below the bytes
    t_tensor = w.B * 8 * w.P * w.H / (bf16_tf * TF32_PER_BF16 * 1e12) if bf16_tf else 0.0
    result = {
        "metric": STREAM_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64, the recipe of the layer workloads)",
        "config": {
            "workload": "%s: S5 streaming step, B=%d sequences x %d single-token s5_step calls, "
                        "H=%d P=%d, fp32" % (w.name, w.B, w.L, w.H, w.P),
            "global_batch": w.B * world, "seq_len": w.L, "H": w.H, "P": w.P,
            "step": "s5_discretize + %d x s5_step" % w.L,
            "timing": "K steps captured in one CUDA graph, replayed once between events",
            "l2": "parameters (%.0f KB) stay L2-resident by design: the step reuses them every "
                  "call" % (alg / 1e3),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm", "kernel": "step_kernel", "achieved": achieved, "peak": hbm_gbs,
            "unit": "GB/s", "frac": achieved / hbm_gbs,
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                           if peak_kind == "measured" else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": alg, "launch_us": call_s * 1e6, "traffic": None,
            "tensor_frac": t_tensor / call_s,
            "definition": "frac = max(algorithmic bytes / HBM peak, projection flops / tensor "
                          "peak) / call time; the bytes term is the larger",
            "note": "a dependent chain of small launches: bound by launch latency, not bandwidth",
        },
        "e2e": {"value": job_throughput(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "public API, pinned host buffers; one step's copies and calls captured "
                        "in a CUDA graph and replayed"},
        "gpu_launches": args.steps * (1 + w.L),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        # one pass from the zero state (the timed steps carry the state on)
        x.zero_()
        api.s5_discretize(lam, log_dt, bt, lb, bb)
        for k in range(w.L):
            api.s5_step(lb, bb, ct, d, x, u_t[k], y=y_t[k])
        y_bl = y_t.transpose(0, 1).cpu().numpy()
        result["cpu_baseline"], oy = cpu_baseline(w, inp)
        result["parity"] = parity_field(y_bl, oy, 1e-5, "y of one pass of %d s5_step calls "
                                        "from the zero state, all %d sequences, against the "
                                        "float64 oracle" % (w.L, w.B))
    print(json.dumps(result), flush=True)
    if dist:
        dist.destroy_process_group()
    return result


# ---------------------------------------------------------------------------
STACK_METRIC = "S5 stack training step (fwd+bwd) tokens/s"


def stack_flops(B, L, H, P, nl):
    """Dense flops of one forward + backward step (the bf16 GEMMs): per layer
    forward Bu and the readout (two of 2T*H*2P) and the gate's W h (2T*H*H);
    backward W^T act and dW (two of 2T*H*H) and x_hat, zbar, dB_bar, dC~
    (four of 2T*H*2P): nine products."""
    T = B * L
    mode_gemm, gate_gemm = 2 * T * H * 2 * P, 2 * T * H * H
    forward = 2 * mode_gemm + gate_gemm
    backward = 4 * mode_gemm + 2 * gate_gemm
    return nl * (forward + backward)


def run_stack(args):
    import numpy as np
    import torch

    from diagonal_state_space_gb300.stack import S5Stack
    from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = WORKLOADS["stack6"]
    inp = make_inputs(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    u0, G = dev(inp["u0"]), dev(inp["G"])
    st = S5Stack(inp["params"], w.B, w.L)
    stream = torch.cuda.current_stream()

    def step():
        st.forward(u0)
        st.backward(G)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # The K timed steps are captured once into a CUDA graph and replayed once
    # between events (the step is ~140 launches; replaying them from a graph
    # takes the host's per-call work out of the timed region, as a training
    # loop that captures its step would).  Eager timing if capture fails.
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                step()
        graph.replay()   # one untimed replay: the graph's first launch uploads it
        torch.cuda.synchronize()
    except Exception as exc:  # noqa: BLE001
        print("bench: stack graph capture failed (%s); timing eagerly" % exc, file=sys.stderr)
        graph = None
    sampler = ClockSampler(gpu_uuid(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(args.steps):
            step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, dist)
    tokens = w.B * w.L
    # end to end: u0 and G from pinned host memory, du0 back, every step.  Two
    # device sets and two copy streams let step i's copies overlap step
    # i-1's compute (du0 is staged on the device so that the next step's
    # backward may overwrite the stack's own buffer).
    u_host = torch.from_numpy(np.ascontiguousarray(inp["u0"])).pin_memory()
    g_host = torch.from_numpy(np.ascontiguousarray(inp["G"])).pin_memory()
    du_hosts = [torch.empty(u_host.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    u_in, g_in = [u0, torch.empty_like(u0)], [G, torch.empty_like(G)]
    du_stage = [torch.empty_like(st.ubar) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(ev_cmp[k])      # step i-2 has consumed set k
            u_in[k].copy_(u_host, non_blocking=True)
            g_in[k].copy_(g_host, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if used[k]:
            stream.wait_event(ev_out[k])        # du0 of step i-2 has been read back
        st.forward(u_in[k])
        st.backward(g_in[k])
        du_stage[k].copy_(st.ubar)
        ev_cmp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[k])
            du_hosts[k].copy_(du_stage[k], non_blocking=True)
            ev_out[k].record(s_out)
        used[k] = True

    e2e_steps = max(1, min(args.e2e_steps, 5))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    s_in.wait_event(a0)
    s_out.wait_event(a0)
    for i in range(2, 2 + e2e_steps):
        e2e_step(i)
    for ev in ev_out:
        stream.wait_event(ev)
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / e2e_steps
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None
    _, bf16_tf, peak_kind = load_peaks()
    flops = stack_flops(w.B, w.L, w.H, w.P, w.layers)
    achieved = flops / (ms / 1e3) / 1e12
    result = {
        "metric": STACK_METRIC, "value": job_throughput(tokens, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64 per layer)",
        "config": {"workload": "stack6: %d layers pre-LN -> S5 -> gate -> residual, forward + "
                               "backward, B=%d L=%d H=%d P=%d, bf16 GEMM operands, complex fp32 "
                               "scans" % (w.layers, w.B, w.L, w.H, w.P),
                   "global_batch": w.B * world, "seq_len": w.L,
                   "l2": "activations of %.1f GB per step, far above the 129 MB L2"
                         % (st.u.numel() * 4 * 7 / 1e9),
                   "timing": ("K steps captured in one CUDA graph, replayed once between events"
                              if graph is not None else "K steps launched eagerly between events"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "whole step (bf16 GEMMs + scans + elementwise)",
                     "achieved": achieved, "peak": bf16_tf, "unit": "TFLOP/s",
                     "frac": achieved / bf16_tf if bf16_tf else None,
                     "peak_source": "%s (MEASURED_PEAKS.json bf16_tflops)" % peak_kind,
                     "flops_per_step": flops, "traffic": None},
        "e2e": {"value": job_throughput(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * u_host.numel() * 4, "d2h_bytes_per_step": du_hosts[0].numel() * 4,
                "ms_per_step": e2e_ms},
        # per step one discretize of all layers' modes; per layer: forward weights,
        # LayerNorm, scan aggregates + apply, gate pre/post; backward gate pre/post,
        # scan aggregates + apply, LayerNorm, dD sum, ZOH chain, dC~; and the nine
        # tensor-core GEMMs (three forward, six backward)
        "gpu_launches": args.steps * (1 + w.layers * 23),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        # sequence 0's top-layer output and input gradient depend on that
        # sequence alone, so the oracle's one-sequence run checks them
        u_top = st.forward(u0)[0].float().cpu().numpy()
        du0 = st.backward(G)["du0"][0].float().cpu().numpy()
        torch.cuda.synchronize()
        result["cpu_baseline"], (ou, og) = stack_cpu_baseline(w, inp)
        result["parity"] = {
            "u_out": parity_field(u_top, ou[0], 2e-2, "sequence 0, top-layer output"),
            "du0": parity_field(du0, og["du0"][0], 2e-2, "sequence 0, input gradient"),
        }
    print(json.dumps(result), flush=True)
    if dist:
        dist.destroy_process_group()
    return result


def oracle_stack_run(inp, seqs):
    import oracle
    p = dict(inp["params"])
    p["lambda"] = p.pop("lambda_")
    return oracle.stack(p, inp["u0"][seqs], inp["G"][seqs])


def stack_cpu_baseline(w, inp):
    """The float64 oracle stack (forward + backward), single-threaded, on one
    sequence of the workload."""
    t0 = time.perf_counter()
    out = oracle_stack_run(inp, [0])
    dt = time.perf_counter() - t0
    rec = {"value": w.L / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": "1 sequence x %d tokens (of %d), %d layers forward + backward, %.1f s"
                     % (w.L, w.B, w.layers, dt), "host_cores_available": os.cpu_count()}
    return rec, out


def run_reference_stack(args):
    from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["stack6"]
    inp = make_inputs(w, B=1)
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_stack_run(inp, [0])
    dt = (time.perf_counter() - t0) / steps
    v = w.L / dt
    sample = "1 sequence x %d tokens per step (of %d sequences), %d layers fwd + bwd" % (
        w.L, w.B, w.layers)
    res = {"metric": STACK_METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": steps,
           "warmup": 0, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "P": w.P,
                      "layers": w.layers,
                      "reference": "float64 CPU oracle (oracle/s5_oracle.c), single thread"},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


def oracle_run(w, inp, seqs):
    import oracle
    if w.varying_dt:
        return oracle.forward_varying_dt(inp["lambda_"], inp["log_dt"], inp["b_tilde"],
                                         inp["c_tilde"], inp["d"], inp["g"][seqs], inp["u"][seqs])
    lb, bb = oracle.discretize_ex(inp["lambda_"], inp["log_dt"], inp["b_tilde"], method=w.method,
                                  clip_re=w.clip_re, dt_scale=w.dt_scale)
    if w.streaming:
        import numpy as np
        x = np.zeros((len(seqs), w.P), np.complex128)
        y = np.empty((len(seqs), w.L, w.H))
        for k in range(w.L):
            x, y[:, k] = oracle.step(lb, bb, inp["c_tilde"], inp["d"], x, inp["u"][seqs, k])
        return y
    if w.bidirectional:
        return oracle.forward_bidirectional(lb, bb, inp["c_tilde2"], inp["d"], inp["u"][seqs])
    return oracle.forward(lb, bb, inp["c_tilde"], inp["d"], inp["u"][seqs])


def cpu_baseline(w, inp):
    """The float64 oracle, as it stands, single-threaded on one host core.
    Returns the baseline record and the oracle's y (every sequence), against
    which the bench's own output is then compared."""
    seqs = list(range(w.B))
    t0 = time.perf_counter()
    out = oracle_run(w, inp, seqs)
    dt = time.perf_counter() - t0
    rec = {"value": len(seqs) * w.L / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": "the whole workload (%d sequences x %d tokens), one pass, %.1f s"
                     % (len(seqs), w.L, dt),
           "host_cores_available": os.cpu_count()}
    return rec, (out[0] if isinstance(out, tuple) else out)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    if args.workload == "stack6":
        return run_reference_stack(args)
    from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    steps = max(1, min(args.steps, 10))
    warm = max(1, min(args.warmup, 2))
    seqs = [0]          # one sequence per step keeps the run to a few minutes
    for _ in range(warm):
        oracle_run(w, inp, seqs)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_run(w, inp, seqs)
    dt = (time.perf_counter() - t0) / steps
    v = len(seqs) * w.L / dt
    sample = "%d sequence x %d tokens per step (of %d sequences)" % (len(seqs), w.L, w.B)
    res = {"metric": (BIDI_METRIC if w.bidirectional else STREAM_METRIC if w.streaming else METRIC),
           "value": v, "unit": "tokens/s",
           "n_gpus": world, "steps": steps,
           "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "P": w.P,
                      "reference": "float64 CPU oracle (oracle/s5_oracle.c), single thread"},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


def launch_replicas(args, argv):
    """``--gpus N``: inside a torchrun rank, WORLD_SIZE must equal N; run
    directly with N > 1, start N ranks of this script (one per GPU, replicas)
    under torch.distributed.run on 127.0.0.1 and return their exit status.
    Returns None when this process should run the bench itself."""
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is not None:
        if int(world_env) != args.gpus:
            sys.exit("bench.py: --gpus %d but WORLD_SIZE=%s; launch exactly --gpus ranks "
                     "(torchrun --nproc-per-node N bench.py --gpus N)" % (args.gpus, world_env))
        return None
    if args.gpus < 1:
        sys.exit("bench.py: --gpus must be at least 1")
    if args.gpus == 1:
        return None
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", str(args.gpus), "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    args = parse()
    rc = launch_replicas(args, sys.argv[1:])
    if rc is not None:
        sys.exit(rc)
    world, rank, _ = dist_env()
    if world > 1:
        print("bench: rank %d of %d" % (rank, world), file=sys.stderr, flush=True)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack6":
        run_stack(args)
    elif args.workload == "stream":
        run_stream(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
