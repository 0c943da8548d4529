#!/usr/bin/env python
"""Benchmark of the chunkwise gated delta rule on one GB300 (or N replicas).

One step = the forward pass and the complete backward pass of the KDA workload B=2, T=8192, H=32, dk=dv=128, bf16 I/O, per-channel gate
(the configuration the tokens/s headline is quoted on), synthetic seeded
inputs resident in HBM. Prints one JSON line. The policy decides what the
backward starts from: "save" (the default: the forward keeps its chunk
intermediates in a saved buffer, about 1.2 GB at this workload) or
"recompute" (the backward rebuilds them from the inputs, no saved buffer).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--policy save|recompute]

Under torchrun every rank runs its own replica (weak scaling, no data-path
collective); the elapsed time is the max over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA fwd+bwd tokens/s and TFLOP/s (% bf16 tensor peak), 1xGB300"
BT = 64
WORKLOAD_IDX = 4


def heads_subset(case, H):
    """The same workload restricted to its first H heads (profiling captures
    of a smaller device footprint)."""
    from workloads import Case

    def sl(x):
        return None if x is None else x[:, :, :H].contiguous()

    def st(x):
        return None if x is None else x[:, :H].contiguous()

    return Case(case.io, case.gate, case.B, case.T, H, case.K, case.V, case.scale, sl(case.q), sl(case.k),
                sl(case.v), sl(case.beta), sl(case.g), st(case.h0), sl(case.do), st(case.dht),
                case.cu_seqlens, case.name + f"_h{H}", dict(case.meta))


# ---------------------------------------------------------------- FLOP model
def chunk_lengths(case):
    out = []
    ss = case.seq_starts
    for n in range(case.N):
        L = ss[n + 1] - ss[n]
        out += [min(BT, L - a) for a in range(0, L, BT)]
    return out


def flops_model(case):
    """Algorithmic dense FLOPs (2 per multiply-add) per step, summed over
    chunk x head with the exact chunk length n and d = dk = dv:
    forward 10 n^2 d + 6 n d^2 + 2 n^3/3, backward 16 n^2 d + 12 n d^2,
    recompute 8 n^2 d + 4 n d^2 + 2 n^3/3."""
    d = case.K
    fwd = bwd = rec = 0.0
    for n in chunk_lengths(case):
        fwd += 10 * n * n * d + 6 * n * d * d + 2 * n ** 3 / 3
        bwd += 16 * n * n * d + 12 * n * d * d
        rec += 8 * n * n * d + 4 * n * d * d + 2 * n ** 3 / 3
    return fwd * case.H, bwd * case.H, rec * case.H


def kernel_work(case, save=False):
    """Work per launch of each library kernel: dense FLOPs (the products the
    kernel owns in the FLOP model) and STORED bytes (every tensor the kernel
    must read or write once at its stored precision, the chunk intermediates
    included), summed over chunk x head with the exact chunk length n
    (d = dk = dv). Under the save policy the forward prep also writes A for the
    backward and alpha with its two constants (per-channel gate: fp32 token rows
    and two rows of d; scalar gate: 80 floats), which the consumer reads in
    place of g. The roofline's algorithmic
    bytes (the operator's own inputs, outputs and states only) are in io_bytes."""
    d = case.K
    e = 2 if case.io == "bf16" else 4
    gb = {"channel": 4 * d, "scalar": 4, "none": 0}[case.gate]   # log-decay bytes per token
    # alpha saved for the consumer per chunk x head (fp32), in place of its g
    alpha = {"channel": 64 * d * 4 + 2 * d * 4, "scalar": 80 * 4, "none": 0}[case.gate]
    fl = dict(k_prep=0.0, k_fwd_scan=0.0, k_fwd_scan_recompute=0.0, k_bwd_scan=0.0,
              k_bwd_dstate=0.0, k_bwd_intra=0.0, k_prep_tc=0.0, k_fwd_scan_tc=0.0,
              k_fwd_scan_tc_recompute=0.0, k_fwd_scan_tc_save=0.0, k_bwd_scan_tc=0.0, k_bwd_consumer_tc=0.0)
    by = dict.fromkeys(fl, 0.0)
    for n in chunk_lengths(case):
        fl["k_prep"] += 8 * n * n * d + 2 * n ** 3 / 3
        fl["k_fwd_scan"] += 6 * n * d * d + 2 * n * n * d
        fl["k_fwd_scan_recompute"] += 4 * n * d * d
        fl["k_bwd_scan"] += 6 * n * d * d + 4 * n * n * d
        fl["k_bwd_dstate"] += 4 * n * n * d + 6 * n * d * d
        fl["k_bwd_intra"] += 8 * n * n * d
        fl["k_prep_tc"] += 8 * n * n * d + 2 * n ** 3 / 3
        fl["k_fwd_scan_tc"] += 6 * n * d * d + 2 * n * n * d
        fl["k_fwd_scan_tc_recompute"] += 4 * n * d * d
        fl["k_fwd_scan_tc_save"] += 4 * n * d * d
        fl["k_bwd_scan_tc"] += 6 * n * d * d + 4 * n * n * d
        fl["k_bwd_consumer_tc"] += 12 * n * n * d + 6 * n * d * d
        # tensor-core path: bf16 tiles W, U, F, Q_g, C_q, A, S, S+bar, R, P; fp32 G at the chunk end
        by["k_prep_tc"] += (3 * n * d * e + n * gb + n * e + 4 * n * d * 2 + n * n * 2 + d * 4
                            + ((n * n * 2 + alpha) if save else 0))
        by["k_fwd_scan_tc"] += 4 * n * d * 2 + n * n * 2 + d * 4 + n * d * e
        by["k_fwd_scan_tc_recompute"] += 3 * n * d * 2 + d * 4 + d * d * 2 + n * d * 2
        by["k_fwd_scan_tc_save"] += 3 * n * d * 2 + d * 4 + d * d * 2 + n * d * 2
        by["k_bwd_scan_tc"] += 3 * n * d * 2 + 2 * n * n * 2 + d * 4 + n * d * e + d * d * 2 + n * d * 2
        by["k_bwd_consumer_tc"] += (3 * n * d * 2 + 2 * d * d * 2 + 3 * n * d * e + alpha + n * e
                                    + 3 * n * d * e + n * e + n * gb)
    st = 2 * 4 * d * d * case.N   # initial/final state (or its adjoint) per sequence, read + write
    for kname in ("k_fwd_scan_tc", "k_bwd_scan_tc"):
        by[kname] += st
    # the joint schedule: the reverse scans and the consumer in one launch
    fl["k_bwd_joint_tc"] = fl["k_bwd_scan_tc"] + fl["k_bwd_consumer_tc"]
    by["k_bwd_joint_tc"] = by["k_bwd_scan_tc"] + by["k_bwd_consumer_tc"]
    return {k: (fl[k] * case.H, by[k] * case.H) for k in fl}


def io_bytes(case):
    """Algorithmic HBM bytes per launch of each library kernel: only the operator's own inputs,
    outputs and states that the kernel reads or writes (chunk intermediates excluded), summed over
    chunk x head with the exact chunk length n. The consumer reads q, k, v, dO, beta (the gate
    reaches it as the prep's alpha, an intermediate) and writes
    dq, dk, dv, dbeta, dg; the prep reads q, k, v, beta, g; the output scan writes o and reads h0,
    writes ht; the reverse scan reads dO and dht and writes dh0."""
    d = case.K
    e = 2 if case.io == "bf16" else 4
    gb = {"channel": 4 * d, "scalar": 4, "none": 0}[case.gate]
    tok = sum(chunk_lengths(case)) * case.H
    st = 4 * d * d * case.N * case.H
    by = {
        "k_prep_tc": tok * (3 * d * e + e + gb),
        "k_fwd_scan_tc": tok * d * e + 2 * st,
        "k_fwd_scan_tc_save": st,
        "k_fwd_scan_tc_recompute": st,
        "k_bwd_scan_tc": tok * d * e + 2 * st,
        "k_bwd_consumer_tc": tok * (4 * d * e + e + 3 * d * e + e + gb),
    }
    # the joint schedule: the consumer's inputs and outputs plus the reverse scan's states (dO once)
    by["k_bwd_joint_tc"] = by["k_bwd_consumer_tc"] + 2 * st
    for k in ("k_prep", "k_fwd_scan", "k_bwd_scan", "k_bwd_dstate", "k_bwd_intra"):
        by.setdefault(k, 0.0)
    by["k_prep"] = by["k_prep_tc"]
    by["k_fwd_scan"] = by["k_fwd_scan_tc"]
    by["k_bwd_scan"] = by["k_bwd_scan_tc"]
    by["k_bwd_dstate"] = tok * (2 * d * e + e + d * e)            # v, dO, beta in; dv out
    by["k_bwd_intra"] = tok * (3 * d * e + e + gb + 2 * d * e + e + gb)   # q, k, dO, beta, g in; dq, dk, dbeta, dg out
    return by


def token_bytes(case):
    """Algorithmic HBM bytes of one fwd+bwd step: every input read and every
    output written once (fwd: q,k,v,beta,g,h0 in, o,ht out; bwd: q,k,v,beta,g,
    h0,do,dht in, dq,dk,dv,dbeta,dg,dh0 out)."""
    e = 2 if case.io == "bf16" else 4
    T = case.B * case.T
    H, K, V = case.H, case.K, case.V
    gb = {"channel": 4 * K, "scalar": 4, "none": 0}[case.gate]
    st = 4 * K * V * case.N * H
    fwd = T * H * (e * (2 * K + V) + e + gb + e * V) + st * (2 if case.h0 is not None else 1)
    bwd = T * H * (e * (2 * K + 2 * V) + e + gb + e * (2 * K + V) + e + gb) + st * 3
    return fwd + bwd


# ------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_uuid=None, path=None):
        """path: where the raw samples go (kept); None: a temporary file, removed after parsing."""
        self.proc = None
        self.keep = bool(path)
        if not path:
            import tempfile
            fd, path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
            os.close(fd)
        self.path = path
        self.uuid = dev_uuid

    def start(self):
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.uuid:
                cmd += ["--id=" + self.uuid]
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max=2070.0, source="fallback")


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel's source file is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    srcdir = os.path.join(ROOT, "chunkwise_delta_rule_gb300", "csrc")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        if len(parts) < 4 or parts[0] != kernel:
            continue
        fname, digest, nbytes = parts[1], parts[2], parts[3]
        try:
            cur = hashlib.sha256(open(os.path.join(srcdir, fname), "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        if cur == digest:
            return float(nbytes)
    return None


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


def profile_begin(lib):
    lib.kda_profile_begin.restype = ctypes.c_int
    lib.kda_profile_begin()


def profile_end(lib):
    arr = (KernelTime * 32)()
    lib.kda_profile_end.argtypes = [ctypes.POINTER(KernelTime), ctypes.c_int]
    lib.kda_profile_end.restype = ctypes.c_int
    n = lib.kda_profile_end(arr, 32)
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(max(n, 0))}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device):
    """The largest x over all ranks (each rank passes its own step time); x itself
    with one rank. Works on any initialised backend (device: where the reduced
    tensor lives, a CUDA device for NCCL, the CPU for gloo)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ws, step_ms):
    """Weak scaling: every rank runs its own replica of the workload each step, so
    the job's rate is the units of all ranks over the slowest rank's step time."""
    return ws * units_per_rank / (step_ms * 1e-3)


# ----------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    from workloads import CONFIGS, make_config_case

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    cfg = CONFIGS[args.config]
    case_cpu = make_config_case(args.config)
    if args.kv:   # the same workload recipe at other key / value widths
        from workloads import make_case
        kk, vv = (int(x) for x in args.kv.split(","))
        c0 = case_cpu
        case_cpu = make_case(io=cfg["io"], gate=c0.gate, B=c0.B, T=c0.T, H=c0.H, K=kk, V=vv,
                             seed=cfg.get("seed", 3), h0=c0.h0 is not None, dht=c0.dht is not None)
    if args.heads:
        case_cpu = heads_subset(case_cpu, args.heads)
    pro = {}
    if args.prologue:
        case_cpu, pro = with_prologue(case_cpu)
        pro = {k: v.to(dev) for k, v in pro.items()}
    if args.gdn2:
        import torch as _t
        gen = _t.Generator().manual_seed(4242)
        pro["erase"] = (2.0 * _t.sigmoid(_t.randn(case_cpu.k.shape, generator=gen))).to(case_cpu.q.dtype).to(dev)
        pro["write"] = _t.sigmoid(_t.randn(case_cpu.v.shape, generator=gen)).to(case_cpu.q.dtype).to(dev)
    if args.gva > 1:   # grouped value heads: one q, k per group of value heads
        case_cpu.q = case_cpu.q[:, :, ::args.gva].contiguous()
        case_cpu.k = case_cpu.k[:, :, ::args.gva].contiguous()
    case = case_cpu.to(dev)
    lib = _lib.load()
    save = 1 if args.policy == "save" else 0
    p = kda.make_problem(case.q, case.k, case.v, case.g, None if args.gdn2 else case.beta, gate=case.gate,
                         scale=case.scale, initial_state=case.h0, cu_seqlens=case.cu_seqlens,
                         save_policy=save, qk_l2norm=bool(args.prologue), schedule=args.schedule, **pro)
    wf = torch.empty(kda.kda_workspace_size(p, False), dtype=torch.uint8, device=dev)
    wb = torch.empty(kda.kda_workspace_size(p, True), dtype=torch.uint8, device=dev)
    sv = torch.empty(kda.kda_saved_size(p), dtype=torch.uint8, device=dev) if save else None
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        kda.kda_chunk_fwd(p, workspace=wf, saved=sv)
        kda.kda_chunk_bwd(p, case.do, case.dht, workspace=wb, saved=sv)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid and not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid, args.clocks_csv) if rank == 0 else None
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # eager calls through the public API, every launch bracketed by the library's own events (the
    # per-kernel times and the roofline come from this region)
    profile_begin(lib)
    t_wall = time.perf_counter()
    for i in range(K):
        l2.zero_()                                  # flush L2 between timed steps
        ev[i][0].record()
        kda.kda_chunk_fwd(p, workspace=wf, saved=sv)
        ev[i][1].record()
        kda.kda_chunk_bwd(p, case.do, case.dht, workspace=wb, saved=sv)
        ev[i][2].record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier()
    kern = profile_end(lib)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    eager_ms = [f + b for f, b in zip(fwd_ms, bwd_ms)]
    # the same step captured once as a CUDA graph and replayed (the pages' timing protocol: graph
    # replays, medians), L2 flushed before every replay
    graph_ms = None
    if not args.no_graph:
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            step()
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step()
        for _ in range(args.warmup):
            gr.replay()
        torch.cuda.synchronize()
        barrier()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        tg = time.perf_counter()
        for i in range(K):
            l2.zero_()
            gev[i][0].record()
            gr.replay()
            gev[i][1].record()
        torch.cuda.synchronize()
        t_wall += time.perf_counter() - tg
        barrier()
        graph_ms = [a.elapsed_time(b) for a, b in gev]
        del gr
    clk = clocks.stop() if clocks else None
    eager_med = statistics.median(eager_ms)
    graph_med = statistics.median(graph_ms) if graph_ms else None
    # headline: the median step of the graph replays (eager median when graphs are off); max over ranks
    step_ms = max_over_ranks(graph_med if graph_med is not None else eager_med, ws, dev)

    tokens = case.B * case.T
    fl_f, fl_b, fl_r = flops_model(case)
    value = whole_job_rate(tokens, ws, step_ms)
    tflops = ws * (fl_f + fl_b) / (step_ms * 1e-3) / 1e12
    tflops_exec = ws * (fl_f + fl_b + (fl_r if args.policy == "recompute" else 0.0)) / (step_ms * 1e-3) / 1e12
    pk = peaks()
    launches = sum(v[0] for v in kern.values())
    # dominant kernel (largest total time per step) and its roofline. With a backward in P time
    # pieces the reverse scan and the consumer run P launches per step, each over 1/P of the units:
    # their per-launch work and traffic are a pass's divided by P.
    pieces = max(1, round(kern.get("k_bwd_consumer_tc", (K, 0.0))[0] / K))
    work = kernel_work(case, save=bool(save))
    iob = io_bytes(case)
    for kname in ("k_bwd_scan_tc", "k_bwd_consumer_tc"):
        if kname in work:
            work[kname] = (work[kname][0] / pieces, work[kname][1] / pieces)
            iob[kname] = iob[kname] / pieces

    def traffic_per_launch(kname):
        tr = traffic_for(kname)
        return None if tr is None else (tr / pieces if kname in ("k_bwd_scan_tc", "k_bwd_consumer_tc") else tr)

    dom = max(kern.items(), key=lambda kv: kv[1][1])[0] if kern else None
    roof = None
    if dom:
        n_l, tot = kern[dom]
        avg_ms = tot / n_l
        fl, stored = work.get(dom, (0.0, 0.0))
        by = iob.get(dom, 0.0)
        sm_mhz = clk["sm_mhz"] if clk else pk["sm_max"]
        if "_tc" in dom:
            # which roofline binds: compare the kernel's time at either peak (HBM: the algorithmic
            # bytes, the operator's own inputs and outputs; tensor: the algorithmic FLOPs)
            t_hbm = by / (pk["hbm"] * 1e9)
            t_tc = fl / (pk["bf16"] * 1e12)
            if t_hbm >= t_tc:
                achieved = by / (avg_ms * 1e-3) / 1e9
                roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"],
                        "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4)}
            else:
                achieved = fl / (avg_ms * 1e-3) / 1e12
                roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16"],
                        "unit": "TFLOP/s", "frac": round(achieved / pk["bf16"], 4)}
            stored_gbs = stored / (avg_ms * 1e-3) / 1e9
            roof.update({"traffic": traffic_per_launch(dom), "avg_launch_ms": round(avg_ms, 4),
                         "launches_per_step": round(n_l / K, 2),
                         "algorithmic_bytes": by, "algorithmic_flops": fl,
                         "bytes_note": "algorithmic bytes = the operator's own inputs, outputs and states this "
                                       "kernel reads or writes; stored bytes add the chunk intermediates",
                         "stored_bytes": stored, "stored_gbs": round(stored_gbs, 1),
                         "stored_frac": round(stored_gbs / pk["hbm"], 4),
                         "tensor_frac_of_bf16_peak": round(fl / (avg_ms * 1e-3) / 1e12 / pk["bf16"], 4),
                         "peak_source": pk["source"] + " (MEASURED_PEAKS.json, of measured)",
                         "sm_mhz_under_load": sm_mhz})
        else:
            alu_peak = 152 * 128 * 2 * pk["sm_max"] * 1e6 / 1e12   # FP32 FMA lanes x 2 x clock
            achieved = fl / (avg_ms * 1e-3) / 1e12
            roof = {"kernel": dom, "bound": "alu", "achieved": round(achieved, 3),
                    "peak": round(alu_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / alu_peak, 4),
                    "traffic": traffic_for(dom), "avg_launch_ms": round(avg_ms, 4),
                    "note": "fp32 CUDA-core FMA kernel; peak = 152 SMs x 128 FP32 lanes x 2 x max SM clock",
                    "sm_mhz_under_load": sm_mhz}
    kernels = {}
    for k, v in kern.items():
        rec = {"launches": v[0], "avg_ms": round(v[1] / v[0], 4),
               "share": round(v[1] / max(sum(x[1] for x in kern.values()), 1e-9), 4)}
        if k in work and work[k][1] > 0:
            t_l = v[1] / v[0] * 1e-3
            gbs = iob.get(k, 0.0) / t_l / 1e9
            sgbs = work[k][1] / t_l / 1e9
            rec.update({"algorithmic_gbs": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm"], 4),
                        "stored_gbs": round(sgbs, 1), "stored_frac": round(sgbs / pk["hbm"], 4),
                        "tflops": round(work[k][0] / t_l / 1e12, 2)})
        kernels[k] = rec

    e2e = None
    if not args.no_e2e and not args.prologue and not args.gdn2 and args.gva <= 1 and not args.kv:   # (the end-to-end and CPU legs time the headline problem)
        e2e = run_e2e(args, case_cpu, dev, kda, K)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu and not args.prologue and not args.gdn2 and args.gva <= 1 \
            and not args.kv:
        cpu = cpu_baseline(case_cpu)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg["io"] == "bf16" else "fp32",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": cfg["name"] + (f"_first{case.H}heads" if args.heads else ""), "B": case.B, "T": case.T, "H": case.H, "dk": case.K,
                       "dv": case.V, "gate": case.gate, "io": cfg["io"], "chunk": BT,
                       "policy": args.policy, "parallelism": f"replicas x{ws}",
                       "backward_pieces": pieces,
                       "prologue": ("raw gate activated in the operator (softplus form, A_log, dt_bias) and "
                                    "q/k L2-normalised in the operator") if args.prologue else "off",
                       "key_heads": case.q.shape[2],
                       "rule": ("GatedDeltaNet-2: erase b = 2 sigmoid(N(0,1)) per key channel, write w = "
                                "sigmoid(N(0,1)) per value channel") if args.gdn2
                       else "delta rule with beta",
                       "l2": "flushed by a 256 MiB write before every timed step (eager and graph)"},
            "tflops": round(tflops, 2), "tflops_executed": round(tflops_exec, 2),
            "frac_bf16_peak": round(tflops / pk["bf16"], 4),
            "frac_bf16_peak_sustained": round(tflops / pk["bf16_sus"], 4),
            "hbm_algorithmic_gbs": round(ws * token_bytes(case) / (step_ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(token_bytes(case) / (step_ms * 1e-3) / 1e9 / pk["hbm"], 4),
            "hbm_floor_ms": round(token_bytes(case) / (pk["hbm"] * 1e9) * 1e3, 4),
            "peaks_source": pk["source"],
            "timing": {"headline": "median of the CUDA-graph replays" if graph_med is not None
                       else "median of the eager steps",
                       "graph_median_ms": None if graph_med is None else round(graph_med, 4),
                       "eager_median_ms": round(eager_med, 4), "eager_mean_ms": round(sum(eager_ms) / K, 4),
                       "eager_min_ms": round(min(eager_ms), 4), "eager_max_ms": round(max(eager_ms), 4)},
            "fwd_ms": round(statistics.median(fwd_ms), 4), "bwd_ms": round(statistics.median(bwd_ms), 4),
            "roofline": roof, "kernels": kernels, "gpu_launches": launches,
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "wall_s": round(t_wall, 3),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def run_compare(args):
    """Schedules of the backward compared in one process, ABBA order: for each listed schedule the
    forward (save policy) runs once, then rounds of timed backward calls alternate A B B A ..., L2
    flushed before each call; prints one JSON line with the median backward time per schedule."""
    import torch

    import chunkwise_delta_rule_gb300 as kda
    from workloads import CONFIGS, make_config_case
    dev = torch.device("cuda", 0)
    cfg = CONFIGS[args.config]
    case = make_config_case(args.config).to(dev)
    scheds = [int(x) for x in args.compare.split(",")]
    probs = {}
    for sc in scheds:
        p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate=case.gate, scale=case.scale,
                             initial_state=case.h0, cu_seqlens=case.cu_seqlens, save_policy=1, schedule=sc)
        wf = torch.empty(kda.kda_workspace_size(p, False), dtype=torch.uint8, device=dev)
        wb = torch.empty(kda.kda_workspace_size(p, True), dtype=torch.uint8, device=dev)
        sv = torch.empty(kda.kda_saved_size(p), dtype=torch.uint8, device=dev)
        kda.kda_chunk_fwd(p, workspace=wf, saved=sv)
        probs[sc] = (p, wb, sv)
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def bwd(sc):
        p, wb, sv = probs[sc]
        kda.kda_chunk_bwd(p, case.do, case.dht, workspace=wb, saved=sv)

    for _ in range(max(args.warmup, 3)):
        for sc in scheds:
            bwd(sc)
    torch.cuda.synchronize()
    times = {sc: [] for sc in scheds}
    rounds = max(args.steps, 30)
    for r in range(rounds):
        order = scheds if r % 2 == 0 else scheds[::-1]
        for sc in order:
            l2.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            bwd(sc)
            b.record()
            times[sc].append((a, b))
    torch.cuda.synchronize()
    med = {sc: statistics.median(x.elapsed_time(y) for x, y in v) for sc, v in times.items()}
    names = {1: "one pass", 9: "joint"}
    print(json.dumps({"compare": "backward schedules, ABBA", "workload": cfg["name"], "observations": rounds,
                      "median_bwd_ms": {f"{sc} ({names.get(sc, f'{sc} pieces' if sc >= 2 else 'default')})":
                                        round(v, 4) for sc, v in med.items()}}), flush=True)


def run_e2e(args, case_cpu, dev, kda, K):
    """Same metric through the public API with host buffers: every step copies
    every input from pinned host memory, runs forward and backward, and reads
    every output back to pinned host memory. The batch runs as one piece per
    sequence (packed sequences: one piece), pipelined over three streams
    (inputs, compute, outputs) with double-buffered device inputs, so that one
    piece's copies overlap another piece's compute and the two copy directions
    overlap each other. The pieces' results are checked against one call on
    the whole batch first."""
    import torch
    names = ["q", "k", "v", "g", "beta", "h0", "do", "dht"]
    full = {n: getattr(case_cpu, n).pin_memory() for n in names if getattr(case_cpu, n) is not None}
    P = case_cpu.B if case_cpu.cu_seqlens is None else 1
    if P == 1:
        host = [full]
        if case_cpu.cu_seqlens is not None:
            host[0]["cu_seqlens"] = case_cpu.cu_seqlens.pin_memory()
    else:   # token tensors are [B, T, ...] and states [B, H, K, V]: sequence b is slice b
        host = [{n: t[b:b + 1] for n, t in full.items()} for b in range(P)]
    devt = [[{n: torch.empty_like(t, device=dev) for n, t in hp.items()} for hp in host] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for hp in host for t in hp.values())
    s_in, s_cp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(P)] for _ in range(2)]
    ev_used = [[torch.cuda.Event() for _ in range(P)] for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(P)]
    outs_host = [None] * P
    d2h = 0

    def run(d):
        p = kda.make_problem(d["q"], d["k"], d["v"], d.get("g"), d["beta"], gate=case_cpu.gate,
                             scale=case_cpu.scale, initial_state=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                             save_policy=1 if args.policy == "save" else 0,
                             schedule=args.schedule if args.e2e_schedule < 0 else args.e2e_schedule)
        o, ht, sv = kda.kda_chunk_fwd(p)
        grads = kda.kda_chunk_bwd(p, d["do"], d.get("dht"), saved=sv)
        return [o, ht] + [x for x in grads if x is not None]

    def step(st):
        nonlocal d2h
        buf = devt[st % 2]
        for b in range(P):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_used[st % 2][b])   # the compute that last read this buffer is done
                for n, t in host[b].items():
                    buf[b][n].copy_(t, non_blocking=True)
                ev_in[st % 2][b].record(s_in)
            with torch.cuda.stream(s_cp):
                s_cp.wait_event(ev_in[st % 2][b])
                res = run(buf[b])
                ev_used[st % 2][b].record(s_cp)
                ev_done[b].record(s_cp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                if outs_host[b] is None:
                    outs_host[b] = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in res]
                    d2h += sum(x.numel() * x.element_size() for x in res)
                for hbuf, x in zip(outs_host[b], res):
                    hbuf.copy_(x, non_blocking=True)
                    x.record_stream(s_out)

    def join():
        cur = torch.cuda.current_stream()
        for sx in (s_in, s_cp, s_out):
            cur.wait_stream(sx)

    for st in range(2):
        step(st)
    join()
    torch.cuda.synchronize()
    # the pieces against one call on the whole batch (device-resident inputs)
    ref = run({n: t.to(dev) for n, t in full.items()} | ({"cu_seqlens": host[0]["cu_seqlens"].to(dev)}
                                                          if "cu_seqlens" in host[0] else {}))
    torch.cuda.synchronize()
    worst = 0.0
    for b in range(P):
        for hx, rx in zip(outs_host[b], ref):
            r = rx.cpu() if P == 1 else rx[b:b + 1].cpu()
            if not torch.equal(hx, r):
                worst = max(worst, float((hx.double() - r.double()).abs().max()))
    del ref
    # three blocks of K steps; the median block is reported (the host link's copy rate varies from
    # process to process on this machine, and a block shows which mode a run is in)
    blocks = []
    for _ in range(3):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record()
        for sx in (s_in, s_cp, s_out):
            sx.wait_event(s0)
        for st in range(K):
            step(st)
        join()
        s1.record()
        torch.cuda.synchronize()
        blocks.append(s0.elapsed_time(s1) / K)
    ms = statistics.median(blocks)
    tokens = case_cpu.B * case_cpu.T
    return {"value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": f"{P} piece(s) (whole sequences), input/compute/output streams, double-buffered inputs",
            "block_ms": [round(b, 4) for b in blocks], "timing": f"median of 3 blocks of {K} steps",
            "pieces_vs_whole_batch": "bitwise equal" if worst == 0.0 else f"max abs diff {worst:.3e}"}


# ------------------------------------------------------ oracle (CPU) timing
def host_cores():
    """Host threads the oracle may use (the cores this process may run on)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(case_cpu):
    """The bounded sample both oracle legs time: whole (sequence, head) pairs of the workload, one
    per host core (all of them when the workload has fewer), spread over sequences and heads."""
    import math
    cores = host_cores()
    N, H = case_cpu.N, case_cpu.H
    total = N * H
    npairs = min(total, cores)
    step = max(1, total // npairs)
    while math.gcd(step, total) != 1:   # a stride coprime to the pair count visits distinct pairs
        step += 1
    pairs = []
    for j in range(npairs):
        i = (j * step) % total
        pairs.append((i % N, i // N))
    return pairs, cores


def time_oracle(case_cpu, pairs, threads, prepared=None):
    """Wall time of the FP64 oracle (recurrence + BPTT) on the sampled pairs with `threads` host
    threads; returns (tokens/s, seconds, token-heads). tokens/s = token-heads / H / seconds, the
    rate at which whole tokens of the workload (all H heads) would be processed."""
    from oracle.cases import pairs_arrays, run_pairs_arrays
    cat, starts = prepared if prepared is not None else pairs_arrays(case_cpu, pairs)
    t = time.perf_counter()
    run_pairs_arrays(case_cpu, cat, starts, backward=True, nthreads=threads)
    dt = time.perf_counter() - t
    ss = case_cpu.seq_starts
    tok_heads = sum(ss[n + 1] - ss[n] for n, _ in pairs)
    return tok_heads / case_cpu.H / dt, dt, tok_heads


def cpu_baseline(case_cpu):
    """The oracle on the host cores: one (sequence, head) pair per core, all cores; and one pair on
    one thread (the single-core figure)."""
    from oracle.cases import pairs_arrays
    pairs, cores = oracle_sample(case_cpu)
    prep = pairs_arrays(case_cpu, pairs)
    v, dt, th = time_oracle(case_cpu, pairs, cores, prep)
    v1, dt1, th1 = time_oracle(case_cpu, pairs[:1], 1)
    return {"value": round(v, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(pairs)} whole (sequence, head) pairs (one per host core) = {th} token-heads, fp64 "
                      f"recurrence + BPTT, {dt:.2f} s wall on {cores} threads; tokens/s = token-heads / H / wall",
            "value_1thread": round(v1, 2),
            "sample_1thread": f"1 pair = {th1} token-heads on 1 thread, {dt1:.2f} s wall"}


def with_prologue(case):
    """The workload with raw inputs for the in-operator prologue: q, k times a
    per-(token, head) norm in [0.5, 3], a raw gate ~ N(0, 1), A_log = log U(1, 4)
    per head and dt_bias = the softplus inverse of dt ~ logU(1e-3, 1e-1)."""
    import math

    import torch
    gen = torch.Generator().manual_seed(12345)
    B, T, H, K = case.q.shape
    qn = torch.rand(B, T, H, 1, generator=gen) * 2.5 + 0.5
    kn = torch.rand(B, T, H, 1, generator=gen) * 2.5 + 0.5
    case.q = (case.q.float() * qn).to(case.q.dtype)
    case.k = (case.k.float() * kn).to(case.k.dtype)
    case.g = torch.randn(case.g.shape, generator=gen)
    dt = torch.exp(torch.rand((H, K) if case.gate == "channel" else (H,), generator=gen)
                   * (math.log(0.1) - math.log(1e-3)) + math.log(1e-3))
    return case, dict(A_log=torch.log(torch.rand(H, generator=gen) * 3 + 1), dt_bias=dt + torch.log(-torch.expm1(-dt)))


DECODE = dict(name="kda_decode_bf16", B=64, H=32, K=128, V=128)


def run_decode(args):
    """Decoding: one token for each of B sequences through the token-by-token
    forward, the fp32 states updated in place (the serving step). The state
    traffic (read + write, 128 KB per (sequence, head)) dominates; L2 is
    flushed before every timed step."""
    import torch

    import chunkwise_delta_rule_gb300 as kda
    from chunkwise_delta_rule_gb300 import _lib
    from workloads import make_case

    dev = torch.device("cuda", 0)
    cfg = DECODE
    case = make_case(io="bf16", gate="channel", B=cfg["B"], T=1, H=cfg["H"], K=cfg["K"], V=cfg["V"],
                     seed=7).to(dev)
    state = case.h0.clone()
    p = kda.make_problem(case.q, case.k, case.v, case.g, case.beta, gate="channel", scale=case.scale,
                         initial_state=state)
    lib = _lib.load()
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        kda.kda_recurrent_fwd(p, ht=state)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(None, args.clocks_csv)
    clocks.start()
    time.sleep(0.3)
    profile_begin(lib)
    for i in range(K):
        l2.zero_()
        ev[i][0].record()
        kda.kda_recurrent_fwd(p, ht=state)
        ev[i][1].record()
    torch.cuda.synchronize()
    kern = profile_end(lib)
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    B, H, D = cfg["B"], cfg["H"], cfg["K"]
    by = B * H * (D * D * 4 * 2 + 2 * D * 2 + D * 4 + D * 2 + 2 + D * 2)   # state in/out; q, k; g; v; beta; o
    n_l, tot = kern.get("k_recurrent", (K, ms * K))
    avg = tot / max(n_l, 1)
    pk = peaks()
    ach = by / (avg * 1e-3) / 1e9
    line = {"metric": "KDA decode tokens/s (token-by-token forward, in-place state), 1xGB300",
            "value": round(B / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": cfg["name"], "B": B, "T": 1, "H": H, "dk": D, "dv": D, "gate": "channel",
                       "io": "bf16", "state": "fp32, updated in place",
                       "l2": "flushed by a 256 MiB write before every timed step"},
            "roofline": {"kernel": "k_recurrent", "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(ach / pk["hbm"], 4), "traffic": None,
                         "avg_launch_ms": round(avg, 5), "algorithmic_bytes": by,
                         "peak_source": pk["source"] + " (MEASURED_PEAKS.json)"},
            "gpu_launches": sum(v[0] for v in kern.values()), "clocks": clk}
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the FP64 oracle (the only reference there is), timed on the host cores.
    Each step runs the same bounded sample as the CPU-baseline leg (one whole (sequence, head)
    pair per core); ms_per_step is that sample's measured wall time."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle.cases import pairs_arrays
    from workloads import CONFIGS, make_config_case
    cfg = CONFIGS[args.config]
    case_cpu = make_config_case(args.config)
    pairs, cores = oracle_sample(case_cpu)
    prep = pairs_arrays(case_cpu, pairs)
    for _ in range(args.warmup):
        time_oracle(case_cpu, pairs, cores, prep)
    vals, dts, th = [], [], 0
    for _ in range(args.steps):
        v, dt, th = time_oracle(case_cpu, pairs, cores, prep)
        vals.append(v)
        dts.append(dt)
    dt_med = statistics.median(dts)
    value = th / case_cpu.H / dt_med
    v1, dt1, th1 = time_oracle(case_cpu, pairs[:1], 1)
    sample = (f"{len(pairs)} whole (sequence, head) pairs per step (one per host core) = {th} token-heads of "
              f"the workload, fp64 recurrence + BPTT on {cores} host threads; ms_per_step = the sample's "
              f"median wall time; tokens/s = token-heads / H / wall")
    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt_med, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": cfg["name"], "B": case_cpu.B, "T": case_cpu.T, "H": case_cpu.H,
                       "dk": case_cpu.K, "dv": case_cpu.V, "gate": case_cpu.gate, "io": cfg["io"]},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample, "value_1thread": round(v1, 2),
                             "sample_1thread": f"1 pair = {th1} token-heads on 1 thread, {dt1:.2f} s wall"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls only (no CUDA-graph replay leg)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=WORKLOAD_IDX)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--schedule", type=int, default=0,
                    help="backward schedule: 0 the library's choice, 1 one pass, 2..8 time pieces, 9 joint")
    ap.add_argument("--e2e-schedule", type=int, default=-1,
                    help="backward schedule of the end-to-end leg (default: the same as --schedule)")
    ap.add_argument("--clocks-csv", default="",
                    help="keep the raw nvidia-smi clock samples of the timed region in this file")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--heads", type=int, default=0, help="restrict the workload to its first H heads (profiling)")
    ap.add_argument("--kv", default="", help="key,value widths (e.g. 80,112) for the same workload recipe")
    ap.add_argument("--gva", type=int, default=1,
                    help="grouped value heads: this many value heads per key head")
    ap.add_argument("--gdn2", action="store_true",
                    help="the GatedDeltaNet-2 rule (erase/write vectors in place of beta)")
    ap.add_argument("--prologue", action="store_true",
                    help="raw gate and unnormalised q, k: activation and L2 norm inside the operator")
    ap.add_argument("--decode", action="store_true",
                    help="time the token-by-token forward on a decoding step instead of the headline")
    ap.add_argument("--compare", default="",
                    help="comma-separated backward schedules (e.g. 9,3,1) timed against each other in ABBA order")
    ap.add_argument("--policy", choices=["save", "recompute"], default="save",
                    help="save: the forward keeps its intermediates for the backward; recompute: the backward rebuilds them")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.compare:
        run_compare(args)
    elif args.decode:
        run_decode(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
