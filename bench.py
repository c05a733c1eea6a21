#!/usr/bin/env python
"""Benchmark of the DeltaNet delta-rule operator on one GB300 (per rank).

Headline (``value``): chunkwise forward tokens/s on the 1.3B-layer shape
(B8 H16 T2048 dk=dv=128, C=64, bf16 I/O, fp32 state, zero initial state).
One step = one ``dn_chunk_fwd`` over that batch.  Beside it, in the same
run: the fused decoding step (B256 H16 dk=dv=128, fp32 state, bf16 inputs,
beta in (0,2)) over 1024 chained steps with fresh inputs, reported as
tokens/s and achieved HBM GB/s; the headline measured end to end through the
public API from pinned host buffers; and the fp64 oracle on a bounded sample
of the headline workload on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same per-GPU workload on its own GPU (the
operator shards over independent (batch, head) pairs, no collective): weak
scaling, ``value`` = all ranks' tokens / the slowest rank's time.  The
reference arm (``--impl reference``) times the fp64 CPU oracle, rank 0 only.
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "delta-rule chunk fwd tokens/s on 1 GB300 + % roofline; decode step HBM GB/s"
HEADLINE = "layer1p3b_bf16"
DECODE = "decode_bf16"
# nominal dense tf32 / bf16 tensor rates (1.1 / 2.25 PFLOP/s): the peak of a tf32
# contraction, scaled from the measured bf16 one
TF32_PER_BF16_NOMINAL = 1.1 / 2.25
LONG = "long_prefill_bf16"
E_SLICES = 4  # batch slices of the pipelined end-to-end leg
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2**20


def chunk_flops_per_token_head(C, dk, dv):
    """Algorithmic FLOPs of the chunkwise WY form per token and head, with the
    triangular halves skipped: C(3dk + 2dv) + 6 dk dv + C^2/3."""
    return C * (3 * dk + 2 * dv) + 6 * dk * dv + C * C / 3.0


def chunk_dense_flops_per_token_head(C, dk, dv):
    """The same products counted as full tiles (the triangles not skipped),
    as tensor cores execute them: 2C(3dk + 2dv) + 6 dk dv + C^2/3."""
    return 2 * C * (3 * dk + 2 * dv) + 6 * dk * dv + C * C / 3.0


def bwd_flops_per_chunk(C, dk, dv):
    """FLOPs the chunkwise backward executes per (batch, head, chunk), dense
    tiles as the three kernels form them (the forward recompute of the chunk
    states included, as the method recomputes by design):
    2 (9 C^2 dk + 10 C dk dv + 8 C^2 dv + 2.5 C^3)."""
    return 2.0 * (9 * C * C * dk + 10 * C * dk * dv + 8 * C * C * dv + 2.5 * C ** 3)


def fp32_alu_tflops(sm_mhz, sms=152, lanes=128):
    """FP32 CUDA-core peak: SMs x FP32 lanes per SM x 2 FLOP (FMA) x clock."""
    return sms * lanes * 2 * sm_mhz * 1e6 / 1e12



def chunk_bytes(B, H, T, dk, dv, esize, with_s0, with_st):
    """Algorithmic HBM bytes of one chunk forward: q, k, v, beta read, o
    written, plus the fp32 states read / written once per head."""
    b = B * H * T * (2 * dk + 2 * dv + 1) * esize
    b += B * H * dk * dv * 4 * (int(with_s0) + int(with_st))
    return b


def decode_bytes(B, H, dk, dv, esize):
    """Algorithmic HBM bytes of one decoding step: the fp32 state read and
    written once, q, k, v, beta read and o written."""
    return B * H * (2 * dk * dv * 4 + (2 * dk + 2 * dv + 1) * esize)


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_traffic(names, source: str):
    """DRAM bytes per call (summed over the named kernels) from the committed
    ncu summary, or None when the kernel source changed since the capture."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    table = json.loads(p.read_text())
    src = ROOT / "delta_rule_recurrent_gb300" / "csrc" / source
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    total = 0.0
    for name in ([names] if isinstance(names, str) else names):
        entry = table.get(name)
        if not entry or entry.get("source_sha") != sha:
            return None
        total += entry["bytes_per_launch"]
    return total


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({names[i] for r in busy for i, flag in enumerate(r[3]) if flag == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": seen, "samples": len(busy)}


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(n: int, argv, script: str | None = None) -> int:
    """Runs `script` (this file by default; the script that was started, from
    main) as n ranks of one node under torchrun, one process per GPU,
    rendezvous on 127.0.0.1; returns torchrun's exit code.  `python bench.py
    --gpus N` without a torchrun environment goes through here, so it runs
    the same replicas a torchrun launch of it does."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={free_port()}",
           script or str(Path(__file__).resolve()), *argv]
    return subprocess.call(cmd)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the slowest rank's time): an all-reduce
    on the process group's device (NCCL: the GPU, gloo: host memory)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput of weak-scaling replicas: every rank processes the
    same units, and the job takes as long as its slowest rank."""
    return world * units_per_rank / seconds


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def timed_loop(fn, steps, stream, world):
    """Runs fn `steps` times between a barrier + synchronize on both sides;
    returns (wall seconds of the whole region, per-launch event ms list)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        fn(i)
        ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    region_s = e0.elapsed_time(e1) / 1e3
    return region_s, [s.elapsed_time(e) for s, e in zip(starts, ends)]


def timed_region(fn, steps, stream, world):
    """Runs fn `steps` times back to back between a barrier + synchronize on
    both sides, with CUDA events only at the region's ends (none between the
    steps, so launches that overlap their predecessor's tail can); returns
    the region's seconds."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3


def graph_decode(step, nsteps, stream, world):
    """Captures step(0..nsteps-1) into one CUDA graph, replays it once to
    warm up, then times one replay; returns (seconds, None) or (None, error)."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for i in range(nsteps):
                step(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(torch.cuda.current_stream())
        g.replay()
        e1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / 1e3, world), None
    except Exception as exc:  # reported in the JSON line, the eager numbers stand
        return None, f"{type(exc).__name__}: {exc}"


def cpu_oracle_sample(inp, budget_s=10.0, max_passes=50):
    """Times the fp64 oracle on whole batch elements of the workload (all H
    heads, all T tokens each), pass after pass, until `budget_s` has passed;
    returns tokens/s of the workload, the batch elements done and the cores
    used."""
    import oracle
    cores = oracle.host_cores()
    B, H, T, _, _ = inp.shape
    done, t0 = 0, time.perf_counter()
    while done < B * max_passes:
        b = done % B
        sl = slice(b, b + 1)
        oracle.forward(inp.q[sl], inp.k[sl], inp.v[sl], inp.beta[sl],
                       None if inp.S0 is None else inp.S0[sl], nthreads=cores)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return done * T / el, done, cores, el


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle on the headline workload."""
    if rank != 0:
        return
    import workloads
    w = workloads.WORKLOADS[HEADLINE]
    inp = workloads.workload_inputs(HEADLINE)
    B, H, T, dk, dv = inp.shape
    import oracle
    cores = oracle.host_cores()
    def one(i):
        b = i % B
        sl = slice(b, b + 1)
        oracle.forward(inp.q[sl], inp.k[sl], inp.v[sl], inp.beta[sl], None, nthreads=cores)
    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(args.warmup + i)
    el = time.perf_counter() - t0
    value = args.steps * T / el
    sample = f"per step one batch element of {HEADLINE} (H={H} heads x T={T} tokens), fp64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": HEADLINE, "B": B, "H": H, "T": T, "dk": dk, "dv": dv,
                   "C": w["C"], "io_dtype": w["dtype"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    import delta_rule_recurrent_gb300 as dn
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    # ---------------- headline: chunk forward, 1.3B-layer shape -------------
    w = workloads.WORKLOADS[HEADLINE]
    inp = workloads.workload_inputs(HEADLINE)
    B, H, T, dk, dv = inp.shape
    C = w["C"]
    q, k, v, beta = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta))
    o = torch.empty(B, H, T, dv, dtype=q.dtype, device=dev)
    S_T = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    algo = args.algo
    lib = dn.load()
    tc = algo in ("auto", "tcgen05") and _tc_used(lib, dk, dv, q.dtype)
    # The two-pass tensor-core path takes a workspace (one [PT; T] tile per
    # chunk), allocated once here, outside the timed region.
    ws_bytes = 0 if args.no_workspace else lib.dn_chunk_fwd_workspace_bytes(
        B, H, T, dk, dv, C, 1 if q.dtype == torch.bfloat16 else 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    split = tc and ws is not None
    launches_per_call = 2 if split else 1

    def chunk_step(_i):
        dn.chunk_fwd(q, k, v, beta, out=o, final_state=S_T, algo=algo, workspace=ws)

    for i in range(args.warmup):
        chunk_step(i)
    torch.cuda.synchronize()

    gpu_index = _physical_gpu_index(local)
    with ClockSampler(gpu_index) as clocks:
        region_s, per_launch = timed_loop(chunk_step, args.steps, stream, world)
        region_s = max_over_ranks(region_s, world)

        # ---------------- decode: fused recurrent step ----------------------
        wd = workloads.WORKLOADS[DECODE]
        Bd, Hd, dkd, dvd = wd["B"], wd["H"], wd["dk"], wd["dv"]
        nsteps = args.decode_steps
        dq, dkk, dvv, db = workloads.decode_inputs_on_device(
            Bd, Hd, dkd, dvd, nsteps + args.warmup, dtype=wd["dtype"], seed=wd["seed"],
            beta_scale=wd["beta_scale"], device=dev)
        Sd = (torch.randn(Bd, Hd, dkd, dvd, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(wd["seed"]))
              * wd["s0_std"])
        od = torch.empty(Bd, Hd, dvd, dtype=dq.dtype, device=dev)

        def decode_step(i):
            dn.recurrent_step(dq[i], dkk[i], dvv[i], db[i], Sd, out=od)

        for i in range(args.warmup):
            decode_step(nsteps + i)
        torch.cuda.synchronize()
        # Consecutive steps overlap their launches (programmatic dependent
        # launch), which an event between two steps would prevent: the steps
        # run back to back and the region's time over the steps is the mean
        # launch duration; the per-step events of timed_loop give the steps in
        # isolation beside it.
        dec_region_s = max_over_ranks(timed_region(decode_step, nsteps, stream, world), world)
        _, dec_launch = timed_loop(decode_step, nsteps, stream, world)

        # The same steps captured once into a CUDA graph and replayed as one
        # launch (no per-step host overhead); the state keeps evolving.
        dec_graph = graph_decode(decode_step, nsteps, stream, world)

        # ---------------- backward: gradients of the chunk forward ----------
        d_o, d_S = workloads.grad_inputs(B, H, T, dv, dk, dtype=w["dtype"], seed=w["seed"],
                                         ds_std=0.1)
        d_o, d_S = d_o.to(dev), d_S.to(dev)
        bws = torch.empty(lib.dn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, C, 1 if tc else 0),
                          dtype=torch.uint8, device=dev)

        def bwd_step(_i):
            dn.chunk_bwd(q, k, v, beta, d_o, d_final_state=d_S, workspace=bws)

        bwd_steps = max(1, min(args.steps, 10))
        for i in range(min(args.warmup, 3)):
            bwd_step(i)
        torch.cuda.synchronize()
        bwd_region_s, bwd_launch = timed_loop(bwd_step, bwd_steps, stream, world)
        bwd_region_s = max_over_ranks(bwd_region_s, world)
        del d_o, d_S, bws

        # ---------------- varlen: the same tokens as 64 packed sequences ------
        vl_lens = workloads.varlen_lengths(64, B * T, seed=w["seed"])
        vl_cu = [0]
        for ln in vl_lens:
            vl_cu.append(vl_cu[-1] + ln)
        # q, k, v, beta re-read as [H, B*T, d]: head-major packing of the same values
        vq, vk, vv = (x.transpose(0, 1).reshape(H, B * T, -1).contiguous() for x in (q, k, v))
        vb = beta.transpose(0, 1).reshape(H, B * T).contiguous()
        vws = None

        def varlen_step(_i):
            dn.chunk_fwd_varlen(vq, vk, vv, vb, vl_cu, workspace=vws)

        import ctypes
        cu_arr = (ctypes.c_int * len(vl_cu))(*vl_cu)
        vneed = lib.dn_chunk_fwd_varlen_workspace_bytes(cu_arr, 64, H, dk, dv, C, 1 if tc else 0)
        vws = torch.empty(vneed, dtype=torch.uint8, device=dev) if vneed else None
        vsteps = max(1, min(args.steps, 20))
        for i in range(min(args.warmup, 3)):
            varlen_step(i)
        torch.cuda.synchronize()
        vl_region_s, vl_launch = timed_loop(varlen_step, vsteps, stream, world)
        vl_region_s = max_over_ranks(vl_region_s, world)
        del vq, vk, vv, vb, vws

        # ---------------- q/k preparation: L2 norm + query scale ------------
        qc, kc = q.clone(), k.clone()

        def prep_step(_i):  # in place: idempotent once normalised, same traffic
            dn.qk_prepare(qc, kc, scale=dk ** -0.5, l2norm=True, inplace=True)

        psteps = max(1, min(args.steps, 20))
        for i in range(min(args.warmup, 3)):
            prep_step(i)
        torch.cuda.synchronize()
        pr_region_s, pr_launch = timed_loop(prep_step, psteps, stream, world)
        pr_region_s = max_over_ranks(pr_region_s, world)
        del qc, kc

        # ---------------- the same call on raw q, k, prepared in its kernels --
        raw = workloads.workload_inputs(HEADLINE, normalize=False)
        rq, rk = raw.q.to(dev), raw.k.to(dev)
        del raw

        def fused_prep_step(_i):
            dn.chunk_fwd(rq, rk, v, beta, out=o, final_state=S_T, algo=algo, workspace=ws,
                         qk_l2norm=True, scale=dk ** -0.5)

        for i in range(min(args.warmup, 3)):
            fused_prep_step(i)
        torch.cuda.synchronize()
        fp_region_s, fp_launch = timed_loop(fused_prep_step, psteps, stream, world)
        fp_region_s = max_over_ranks(fp_region_s, world)
        del rq, rk

        # ---------------- Gated DeltaNet: chunk forward and decode step -----
        gate = workloads.gate_inputs(B, H, T, seed=w["seed"]).to(dev)
        og = torch.empty_like(o)
        Sg = torch.empty_like(S_T)
        gneed = lib.dn_chunk_fwd_gated_workspace_bytes(B, H, T, dk, dv, C, 1 if tc else 0)
        gws = torch.empty(gneed, dtype=torch.uint8, device=dev) if gneed else None

        def gated_step(_i):  # the tcgen05 form where it applies
            dn.chunk_fwd_gated(q, k, v, beta, gate, out=og, final_state=Sg, workspace=gws)

        def gated_simt_step(_i):
            dn.chunk_fwd_gated(q, k, v, beta, gate, out=og, final_state=Sg, workspace=None)

        gsteps = max(1, min(args.steps, 10))
        for i in range(min(args.warmup, 3)):
            gated_step(i)
        torch.cuda.synchronize()
        g_region_s, g_launch = timed_loop(gated_step, gsteps, stream, world)
        g_region_s = max_over_ranks(g_region_s, world)
        for i in range(min(args.warmup, 3)):
            gated_simt_step(i)
        torch.cuda.synchronize()
        gs_region_s, gs_launch = timed_loop(gated_simt_step, gsteps, stream, world)
        gs_region_s = max_over_ranks(gs_region_s, world)
        del gate, og, Sg, gws

        dgate = workloads.gate_inputs(Bd, Hd, seed=wd["seed"]).to(dev)
        Sdg = Sd.clone()

        def gated_decode_step(i):
            dn.recurrent_step_gated(dq[i], dkk[i], dvv[i], db[i], dgate, Sdg, out=od)

        for i in range(args.warmup):
            gated_decode_step(nsteps + i)
        torch.cuda.synchronize()
        gd_region_s = timed_region(gated_decode_step, nsteps, stream, world)
        _, gd_launch = timed_loop(gated_decode_step, nsteps, stream, world)
        gd_region_s = max_over_ranks(gd_region_s, world)
        del dgate, Sdg

        # ---------------- KDA: per-key-channel decay, chunk forward and step --
        kgate = workloads.gate_inputs(B, H, T, seed=w["seed"], channels=dk).to(dev)
        ok_, Sk_ = torch.empty_like(o), torch.empty_like(S_T)
        kneed = lib.dn_chunk_fwd_kda_workspace_bytes(B, H, T, dk, dv, C, 1 if tc else 0)
        kws = torch.empty(kneed, dtype=torch.uint8, device=dev) if kneed else None

        def kda_step(_i):  # the tcgen05 form where it applies
            dn.chunk_fwd_kda(q, k, v, beta, kgate, out=ok_, final_state=Sk_, workspace=kws)

        def kda_simt_step(_i):
            dn.chunk_fwd_kda(q, k, v, beta, kgate, out=ok_, final_state=Sk_, workspace=None)

        for i in range(min(args.warmup, 3)):
            kda_step(i)
        torch.cuda.synchronize()
        k_region_s, k_launch = timed_loop(kda_step, gsteps, stream, world)
        k_region_s = max_over_ranks(k_region_s, world)
        ksteps = max(1, min(args.steps, 3))
        kda_simt_step(0)
        torch.cuda.synchronize()
        ks_region_s, ks_launch = timed_loop(kda_simt_step, ksteps, stream, world)
        ks_region_s = max_over_ranks(ks_region_s, world)
        del kgate, ok_, Sk_, kws

        dkgate = workloads.gate_inputs(Bd, Hd, seed=wd["seed"], channels=dkd).to(dev)
        Sdk = Sd.clone()

        def kda_decode_step(i):
            dn.recurrent_step_kda(dq[i], dkk[i], dvv[i], db[i], dkgate, Sdk, out=od)

        for i in range(args.warmup):
            kda_decode_step(nsteps + i)
        torch.cuda.synchronize()
        kd_region_s = timed_region(kda_decode_step, nsteps, stream, world)
        _, kd_launch = timed_loop(kda_decode_step, nsteps, stream, world)
        kd_region_s = max_over_ranks(kd_region_s, world)
        del dkgate, Sdk

        # ---------------- the decayed backwards: Gated DeltaNet and KDA ---------
        d_o, d_S = workloads.grad_inputs(B, H, T, dv, dk, dtype=w["dtype"], seed=w["seed"],
                                         ds_std=0.1)
        d_o, d_S = d_o.to(dev), d_S.to(dev)
        dec_bwd = {}
        for form, gshape, fn, wsfn in (
                ("gated", None, dn.chunk_bwd_gated, lib.dn_chunk_bwd_gated_workspace_bytes),
                ("kda", dk, dn.chunk_bwd_kda, lib.dn_chunk_bwd_kda_workspace_bytes)):
            gg = workloads.gate_inputs(B, H, T, seed=w["seed"], channels=gshape).to(dev)
            gws_b = torch.empty(wsfn(B, H, T, dk, dv, C, 1 if tc else 0), dtype=torch.uint8,
                                device=dev)

            def dec_bwd_step(_i, fn=fn, gg=gg, gws_b=gws_b):
                fn(q, k, v, beta, gg, d_o, d_final_state=d_S, workspace=gws_b)

            dsteps = max(1, min(args.steps, 3))
            dec_bwd_step(0)
            torch.cuda.synchronize()
            r_s, r_launch = timed_loop(dec_bwd_step, dsteps, stream, world)
            dec_bwd[form] = (max_over_ranks(r_s, world), r_launch, dsteps)
            del gg, gws_b
        del d_o, d_S

        # ---------------- long prefill: one long sequence per head, carried state --
        wl = workloads.WORKLOADS[LONG]
        lp = workloads.workload_inputs(LONG)
        Bl, Hl, Tl, dkl, dvl = lp.shape
        lq, lk, lv, lb = (x.to(dev) for x in (lp.q, lp.k, lp.v, lp.beta))
        lS0 = lp.S0.to(dev)
        lo = torch.empty(Bl, Hl, Tl, dvl, dtype=lq.dtype, device=dev)
        lST = torch.empty(Bl, Hl, dkl, dvl, dtype=torch.float32, device=dev)
        ldt = 1 if lq.dtype == torch.bfloat16 else 0
        lneed = lib.dn_chunk_fwd_workspace_bytes(Bl, Hl, Tl, dkl, dvl, wl["C"], ldt)
        lws = torch.empty(lneed, dtype=torch.uint8, device=dev) if lneed else None
        # The sequence split (dn_chunk_fwd_split) where the tensor cores cover
        # the shape: each sequence cut into as many runs as fill the GPU once.
        sneed = lib.dn_chunk_fwd_split_workspace_bytes(Bl, Hl, Tl, dkl, dvl, wl["C"], ldt, 0)
        lsplit = tc and sneed > 0
        sws = torch.empty(sneed, dtype=torch.uint8, device=dev) if lsplit else None
        nchl = (Tl + wl["C"] - 1) // wl["C"]
        runs = min(max(1, torch.cuda.get_device_properties(dev).multi_processor_count
                       // (Bl * Hl)), nchl, 1024)
        runs = -(-nchl // -(-nchl // runs))  # runs of whole chunks, none empty
        long_launches = (6 if runs > 1 else 2) if lsplit else launches_per_call

        def long_plain(_i):
            dn.chunk_fwd(lq, lk, lv, lb, initial_state=lS0, out=lo, final_state=lST, algo=algo,
                         workspace=lws)

        def long_step(_i):
            if not lsplit:
                return long_plain(_i)
            dn.chunk_fwd_split(lq, lk, lv, lb, initial_state=lS0, out=lo, final_state=lST,
                               segments=0, workspace=sws)

        lsteps = max(1, min(args.steps, 10))
        for i in range(min(args.warmup, 3)):
            long_step(i)
            long_plain(i)
        torch.cuda.synchronize()
        lp_region_s, lp_launch = timed_loop(long_step, lsteps, stream, world)
        lp_region_s = max_over_ranks(lp_region_s, world)
        _, lp_plain_launch = timed_loop(long_plain, lsteps, stream, world)
        del lp, lq, lk, lv, lb, lS0, lo, lST, lws, sws
    clk = clocks.summary()
    del dq, dkk, dvv, db

    # ---------------- e2e: public API from pinned host buffers --------------
    # The batch in E_SLICES slices: slice i's inputs go host -> device on one
    # copy stream, its forward runs on the compute stream once they are in,
    # and its outputs (o and the final state) go device -> host on a second
    # copy stream, so the copies of one slice overlap the compute and the
    # copies of the others.  Every copy is one cudaMemcpyAsync of a
    # contiguous slice.  Consecutive steps use two device buffer sets in
    # turn, so a step's uploads overlap the previous step's last forward and
    # downloads; a set is refilled only after the forward that read it (two
    # steps back) is done, and its outputs overwritten only after they were
    # read back.
    hq, hk, hv, hb = (x.pin_memory() for x in (inp.q, inp.k, inp.v, inp.beta))
    ho = torch.empty(B, H, T, dv, dtype=q.dtype).pin_memory()
    hS = torch.empty(B, H, dk, dv, dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hb))
    d2h = ho.numel() * ho.element_size() + hS.numel() * hS.element_size()
    n_sl = E_SLICES if B % E_SLICES == 0 else 1
    bs = B // n_sl
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sl_ws = []
    for i in range(n_sl):
        need = lib.dn_chunk_fwd_workspace_bytes(bs, H, T, dk, dv, C,
                                                1 if q.dtype == torch.bfloat16 else 0)
        sl_ws.append(torch.empty(need, dtype=torch.uint8, device=dev) if need else None)
    e_sets = [{"t": (q, k, v, beta, o, S_T)},
              {"t": tuple(torch.empty_like(x) for x in (q, k, v, beta, o, S_T))}]
    for st in e_sets:
        st["fwd_done"], st["d2h_done"], st["used"] = torch.cuda.Event(), torch.cuda.Event(), False

    def e2e_step(i, final=False):
        st = e_sets[i & 1]
        eq, ek, ev, eb, eo, eS = st["t"]
        arrived, done = [], []
        if i == 0:  # the first step's uploads start after the region's start event
            go = torch.cuda.Event()
            go.record(stream)
            up.wait_event(go)
        if st["used"]:
            up.wait_event(st["fwd_done"])      # the forward two steps back has read the set
            stream.wait_event(st["d2h_done"])  # and its outputs are back on the host
        for j in range(n_sl):
            sl = slice(j * bs, (j + 1) * bs)
            with torch.cuda.stream(up):
                for dst, src in ((eq, hq), (ek, hk), (ev, hv), (eb, hb)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                arrived.append(torch.cuda.Event())
                arrived[-1].record(up)
        for j in range(n_sl):
            sl = slice(j * bs, (j + 1) * bs)
            stream.wait_event(arrived[j])
            dn.chunk_fwd(eq[sl], ek[sl], ev[sl], eb[sl], out=eo[sl], final_state=eS[sl],
                         algo=algo, workspace=sl_ws[j])
            done.append(torch.cuda.Event())
            done[-1].record(stream)
        st["fwd_done"].record(stream)
        with torch.cuda.stream(down):
            for j in range(n_sl):
                sl = slice(j * bs, (j + 1) * bs)
                down.wait_event(done[j])
                ho[sl].copy_(eo[sl], non_blocking=True)
                hS[sl].copy_(eS[sl], non_blocking=True)
            st["d2h_done"].record(down)
        st["used"] = True
        if final:  # the region ends when every result is on the host
            stream.wait_stream(down)
            stream.wait_stream(up)

    for i in range(min(args.warmup, 3)):
        e2e_step(i, final=True)
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 50))
    e2e_s, _ = timed_loop(lambda i: e2e_step(i, final=i == e2e_steps - 1), e2e_steps, stream,
                          world)
    e2e_s = max_over_ranks(e2e_s, world)
    # link rates seen by the copies alone (same buffers, same streams)
    torch.cuda.synchronize()
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(up)
    with torch.cuda.stream(up):
        for dst, src in ((q, hq), (k, hk), (v, hv), (beta, hb)):
            dst.copy_(src, non_blocking=True)
    c1.record(up)
    down.wait_event(c1)
    with torch.cuda.stream(down):
        ho.copy_(o, non_blocking=True)
        hS.copy_(S_T, non_blocking=True)
    c2.record(down)
    torch.cuda.synchronize()
    h2d_gbs = h2d / (c0.elapsed_time(c1) / 1e3) / 1e9
    d2h_gbs = d2h / (c1.elapsed_time(c2) / 1e3) / 1e9

    # ---------------- numbers ----------------------------------------------
    tokens = B * T
    value = job_throughput(world, tokens * args.steps, region_s)
    launch_s = statistics.mean(per_launch) / 1e3
    flops = chunk_flops_per_token_head(C, dk, dv) * B * H * T
    dflops = chunk_dense_flops_per_token_head(C, dk, dv) * B * H * T
    cbytes = chunk_bytes(B, H, T, dk, dv, q.element_size(), False, True)
    tflops = flops / launch_s / 1e12
    # A "launch" here is one dn_chunk_fwd call; on the two-pass path that is
    # the prepare kernel and the sequence kernel back to back.
    if split:
        kname, knames = "chunk_prep + chunk_scan (two passes)", ["chunk_prep", "chunk_scan"]
    elif tc:
        kname, knames = "chunk_tc (fused)", ["chunk_tc_fused"]
    else:
        kname, knames = "chunk_simt", ["chunk_simt"]
    # The chunk forward's arithmetic intensity (about 133 flop/B on the
    # 1.3B-layer shape) is below the ridge of the measured peaks (about 285
    # flop/B), so HBM is the roof that bounds it; the tensor-peak fraction of
    # the algorithmic FLOPs is reported beside it.
    roofline = {
        "bound": "hbm", "achieved": cbytes / launch_s / 1e9, "peak": peaks["hbm_gbs"],
        "unit": "GB/s", "frac": cbytes / launch_s / 1e9 / peaks["hbm_gbs"],
        "traffic": kernel_traffic(knames, "chunk_tc.cu" if tc else "chunk_simt.cu"),
        "peak_source": f"{peak_src} (copy bandwidth)", "kernel": kname,
        "launches_per_call": launches_per_call, "bytes_per_launch": cbytes,
        "launch_us": launch_s * 1e6,
        "tensor": {"achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": tflops / peaks["bf16_tflops"], "flops_per_launch": flops,
                   "dense_tile_flops_per_launch": dflops,
                   "dense_tile_frac": dflops / launch_s / 1e12 / peaks["bf16_tflops"],
                   "peak_source": f"{peak_src} (bf16 dense burst)"},
    }
    dbytes = decode_bytes(Bd, Hd, dkd, dvd, 2)
    dec_launch_s = dec_region_s / nsteps  # back to back (see timed_region)
    dec_iso_s = statistics.mean(dec_launch) / 1e3
    dec_gbs = dbytes / dec_launch_s / 1e9
    decode = {
        "workload": DECODE, "steps": nsteps, "value": world * Bd * nsteps / dec_region_s,
        "unit": "tokens/s", "ms_per_step": 1e3 * dec_region_s / nsteps,
        "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                     "traffic": kernel_traffic("recurrent_step", "decode.cu"),
                     "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": dbytes,
                     "launch_us": dec_launch_s * 1e6,
                     "launch_us_isolated": dec_iso_s * 1e6,
                     "timing": "steps back to back, events at the region's ends (consecutive "
                               "launches overlap); launch_us_isolated: events around each step"},
        "graph": ({"value": world * Bd * nsteps / dec_graph[0], "unit": "tokens/s",
                   "ms_per_step": 1e3 * dec_graph[0] / nsteps,
                   "hbm_gbs": dbytes * nsteps / dec_graph[0] / 1e9,
                   "frac": dbytes * nsteps / dec_graph[0] / 1e9 / peaks["hbm_gbs"],
                   "launches": nsteps, "note": "all steps in one CUDA graph, one replay"}
                  if dec_graph[0] else {"unavailable": dec_graph[1]}),
        "config": {"B": Bd, "H": Hd, "dk": dkd, "dv": dvd, "state": "fp32",
                   "io_dtype": wd["dtype"], "beta": "2*sigmoid(N(0,1))",
                   "l2": "state 537 MB per step > L2"},
    }
    nchunks = -(-T // C)
    bflops = bwd_flops_per_chunk(C, dk, dv) * B * H * nchunks
    bwd_launch_s = statistics.mean(bwd_launch) / 1e3
    # The backward picks its own path (the tensor-core recompute and chain for bf16,
    # d = 128), whatever --algo says for the forward.
    bwd_tc = _tc_used(lib, dk, dv, q.dtype)
    if bwd_tc:  # bf16 I/O: recompute, chain and gradients on tcgen05 (the solve on CUDA cores)
        bpeak = peaks["bf16_tflops"]
        bbound = "tensor"
        barith = ("tcgen05 bf16 MMAs, fp32 accumulation; states and state gradients "
                  "carried as bf16 hi/lo tile pairs")
        bsrc = f"{peak_src} (bf16 dense burst)"
    else:
        bpeak, bbound, barith = fp32_alu_tflops(2070.0), "alu", "fp32 CUDA cores"
        bsrc = "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz"
    backward = {
        "workload": HEADLINE, "steps": bwd_steps, "value": world * tokens * bwd_steps / bwd_region_s,
        "unit": "tokens/s", "ms_per_step": 1e3 * bwd_region_s / bwd_steps,
        "arith": barith, "launches_per_call": 4 if bwd_tc else 3,
        "roofline": {"bound": bbound, "achieved": bflops / bwd_launch_s / 1e12, "peak": bpeak,
                     "unit": "TFLOP/s", "frac": bflops / bwd_launch_s / 1e12 / bpeak,
                     "traffic": kernel_traffic("chunk_bwd_grads_tc", "chunk_tc.cu") if bwd_tc else None,
                     "traffic_kernel": "chunk_bwd_grads_tc (the dominant kernel)" if bwd_tc else None,
                     "peak_source": bsrc,
                     "flops_per_launch": bflops, "launch_us": bwd_launch_s * 1e6},
        "config": {"d_o": "N(0,1)", "d_S_T": "N(0,0.1^2)", "S0": "none"},
    }
    vl_launch_s = statistics.mean(vl_launch) / 1e3
    # q, k, v, beta, o of the same tokens plus one fp32 final state per (sequence, head)
    vbytes = chunk_bytes(1, H, B * T, dk, dv, q.element_size(), False, False) + 64 * H * dk * dv * 4
    varlen = {
        "workload": f"{HEADLINE} tokens as 64 packed sequences (lengths {min(vl_lens)}-{max(vl_lens)})",
        "steps": vsteps, "value": world * tokens * vsteps / vl_region_s, "unit": "tokens/s",
        "ms_per_step": 1e3 * vl_region_s / vsteps,
        "roofline": {"bound": "hbm", "achieved": vbytes / vl_launch_s / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": vbytes / vl_launch_s / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": vbytes,
                     "launch_us": vl_launch_s * 1e6,
                     "tensor": {"achieved": flops / vl_launch_s / 1e12, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s",
                                "frac": flops / vl_launch_s / 1e12 / peaks["bf16_tflops"]}},
    }
    pr_launch_s = statistics.mean(pr_launch) / 1e3
    pbytes = 4 * B * H * T * dk * q.element_size()  # q and k read once and written once
    qk_prep = {
        "workload": HEADLINE, "steps": psteps, "value": world * tokens * psteps / pr_region_s,
        "unit": "tokens/s", "ms_per_step": 1e3 * pr_region_s / psteps,
        "op": "q, k <- x / sqrt(sum x^2 + 1e-6) per row; q *= dk^-0.5 (in place)",
        "roofline": {"bound": "hbm", "achieved": pbytes / pr_launch_s / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": pbytes / pr_launch_s / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": pbytes,
                     "launch_us": pr_launch_s * 1e6},
    }
    fp_launch_s = statistics.mean(fp_launch) / 1e3
    qk_prep["in_kernel"] = {
        "op": "the headline chunk forward on raw q, k with qk_l2norm=True, scale=dk^-0.5 "
              "(normalised and scaled as the kernels load them)",
        "steps": psteps, "value": world * tokens * psteps / fp_region_s, "unit": "tokens/s",
        "ms_per_step": 1e3 * fp_region_s / psteps, "launch_us": fp_launch_s * 1e6,
        "vs_plain_call": fp_launch_s / launch_s,
        "roofline": {"bound": "hbm", "achieved": cbytes / fp_launch_s / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": cbytes / fp_launch_s / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": cbytes},
    }
    lp_launch_s = statistics.mean(lp_launch) / 1e3
    lbytes = chunk_bytes(Bl, Hl, Tl, dkl, dvl, 2, True, True)
    lflops = chunk_flops_per_token_head(wl["C"], dkl, dvl) * Bl * Hl * Tl
    long_prefill = {
        "workload": LONG, "steps": lsteps, "value": world * Bl * Tl * lsteps / lp_region_s,
        "unit": "tokens/s", "ms_per_step": 1e3 * lp_region_s / lsteps,
        "config": {"B": Bl, "H": Hl, "T": Tl, "dk": dkl, "dv": dvl, "S0": "N(0, 0.1^2) fp32"},
        "path": (f"dn_chunk_fwd_split: {runs} runs per sequence scanned in parallel, "
                 "joined through their transitions" if lsplit else "dn_chunk_fwd"),
        "plain_call_us": 1e3 * statistics.mean(lp_plain_launch),
        "roofline": {"bound": "hbm", "achieved": lbytes / lp_launch_s / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": lbytes / lp_launch_s / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": lbytes,
                     "launch_us": lp_launch_s * 1e6,
                     "tensor": {"achieved": lflops / lp_launch_s / 1e12,
                                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": lflops / lp_launch_s / 1e12 / peaks["bf16_tflops"],
                                "flops_per_launch": lflops}},
    }
    g_launch_s = statistics.mean(g_launch) / 1e3
    gs_launch_s = statistics.mean(gs_launch) / 1e3
    gflops = chunk_flops_per_token_head(C, dk, dv) * B * H * T
    alu_peak = fp32_alu_tflops(2070.0)
    alu_src = "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz"
    gbytes = cbytes + B * H * T * 4  # plus the fp32 log keep rate per token and head
    if gneed:
        g_arith = "tcgen05 bf16 MMAs, fp32 accumulation (two passes)"
        g_roof = {"bound": "hbm", "achieved": gbytes / g_launch_s / 1e9, "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": gbytes / g_launch_s / 1e9 / peaks["hbm_gbs"],
                  "traffic": kernel_traffic(["chunk_prep_gated", "chunk_scan_gated"], "chunk_tc.cu"),
                  "peak_source": f"{peak_src} (copy bandwidth)", "bytes_per_launch": gbytes,
                  "launch_us": g_launch_s * 1e6,
                  "tensor": {"achieved": gflops / g_launch_s / 1e12, "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s",
                             "frac": gflops / g_launch_s / 1e12 / peaks["bf16_tflops"],
                             "flops_per_launch": gflops}}
    else:
        g_arith = "fp32 CUDA cores"
        g_roof = {"bound": "alu", "achieved": gflops / g_launch_s / 1e12, "peak": alu_peak,
                  "unit": "TFLOP/s", "frac": gflops / g_launch_s / 1e12 / alu_peak,
                  "traffic": None, "peak_source": alu_src, "flops_per_launch": gflops,
                  "launch_us": g_launch_s * 1e6}
    gd_launch_s = gd_region_s / nsteps  # back to back, as the plain step
    gdbytes = dbytes + Bd * Hd * 4  # plus the fp32 log keep rate per head
    gated = {
        "chunk": {"workload": HEADLINE, "steps": gsteps,
                  "value": world * tokens * gsteps / g_region_s, "unit": "tokens/s",
                  "ms_per_step": 1e3 * g_region_s / gsteps, "arith": g_arith,
                  "gate": "alpha ~ U(0.9, 1)", "workspace_bytes": gneed,
                  "launches_per_call": 2 if gneed else 1, "roofline": g_roof},
        "chunk_cuda_cores": {"workload": HEADLINE, "steps": gsteps,
                             "value": world * tokens * gsteps / gs_region_s, "unit": "tokens/s",
                             "ms_per_step": 1e3 * gs_region_s / gsteps, "arith": "fp32 CUDA cores",
                             "note": "the same call with no workspace",
                             "roofline": {"bound": "alu", "achieved": gflops / gs_launch_s / 1e12,
                                          "peak": alu_peak, "unit": "TFLOP/s",
                                          "frac": gflops / gs_launch_s / 1e12 / alu_peak,
                                          "traffic": None, "peak_source": alu_src,
                                          "flops_per_launch": gflops,
                                          "launch_us": gs_launch_s * 1e6}},
        "decode": {"workload": DECODE, "steps": nsteps,
                   "value": world * Bd * nsteps / gd_region_s, "unit": "tokens/s",
                   "ms_per_step": 1e3 * gd_region_s / nsteps,
                   "roofline": {"bound": "hbm", "achieved": gdbytes / gd_launch_s / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": gdbytes / gd_launch_s / 1e9 / peaks["hbm_gbs"],
                                "traffic": None, "peak_source": f"{peak_src} (copy bandwidth)",
                                "bytes_per_launch": gdbytes, "launch_us": gd_launch_s * 1e6}},
    }
    k_launch_s = statistics.mean(k_launch) / 1e3
    kd_launch_s = kd_region_s / nsteps  # back to back, as the plain step
    kdbytes = dbytes + Bd * Hd * dkd * 4  # plus the fp32 per-channel log keep rates
    ks_launch_s = statistics.mean(ks_launch) / 1e3
    kbytes = cbytes + B * H * T * dk * 4  # plus the fp32 log keep rate per token, head and channel
    if kneed:
        k_arith = "tcgen05 bf16 MMAs, fp32 accumulation (decayed operands, two passes)"
        k_roof = {"bound": "hbm", "achieved": kbytes / k_launch_s / 1e9, "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": kbytes / k_launch_s / 1e9 / peaks["hbm_gbs"],
                  "traffic": None, "peak_source": f"{peak_src} (copy bandwidth)",
                  "bytes_per_launch": kbytes, "launch_us": k_launch_s * 1e6,
                  "tensor": {"achieved": gflops / k_launch_s / 1e12, "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s",
                             "frac": gflops / k_launch_s / 1e12 / peaks["bf16_tflops"],
                             "flops_per_launch": gflops}}
    else:
        k_arith = "fp32 CUDA cores"
        k_roof = {"bound": "alu", "achieved": gflops / k_launch_s / 1e12, "peak": alu_peak,
                  "unit": "TFLOP/s", "frac": gflops / k_launch_s / 1e12 / alu_peak,
                  "traffic": None, "peak_source": alu_src, "flops_per_launch": gflops,
                  "launch_us": k_launch_s * 1e6}
    kda = {
        "chunk": {"workload": HEADLINE, "steps": gsteps,
                  "value": world * tokens * gsteps / k_region_s, "unit": "tokens/s",
                  "ms_per_step": 1e3 * k_region_s / gsteps, "arith": k_arith,
                  "gate": "alpha ~ U(0.9, 1) per key channel", "workspace_bytes": kneed,
                  "launches_per_call": 4 if kneed else 1, "vs_plain_call": k_launch_s / launch_s,
                  "roofline": k_roof},
        "chunk_cuda_cores": {"workload": HEADLINE, "steps": ksteps,
                             "value": world * tokens * ksteps / ks_region_s, "unit": "tokens/s",
                             "ms_per_step": 1e3 * ks_region_s / ksteps, "arith": "fp32 CUDA cores",
                             "note": "the same call with no workspace",
                             "roofline": {"bound": "alu", "achieved": gflops / ks_launch_s / 1e12,
                                          "peak": alu_peak, "unit": "TFLOP/s",
                                          "frac": gflops / ks_launch_s / 1e12 / alu_peak,
                                          "traffic": None, "peak_source": alu_src,
                                          "flops_per_launch": gflops,
                                          "launch_us": ks_launch_s * 1e6}},
        "decode": {"workload": DECODE, "steps": nsteps,
                   "value": world * Bd * nsteps / kd_region_s, "unit": "tokens/s",
                   "ms_per_step": 1e3 * kd_region_s / nsteps,
                   "roofline": {"bound": "hbm", "achieved": kdbytes / kd_launch_s / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": kdbytes / kd_launch_s / 1e9 / peaks["hbm_gbs"],
                                "traffic": None, "peak_source": f"{peak_src} (copy bandwidth)",
                                "bytes_per_launch": kdbytes, "launch_us": kd_launch_s * 1e6}},
    }
    # The decayed backwards: recompute on tcgen05 (bf16, d = 128), chain and
    # per-chunk gradients on tf32 mma.sync (bf16) or fp32 CUDA cores (fp32).
    dec_tc = _tc_used(lib, dk, dv, q.dtype)
    if dec_tc:
        dpeak = peaks["bf16_tflops"] * TF32_PER_BF16_NOMINAL
        dsrc = (f"{peak_src} bf16 dense burst x {TF32_PER_BF16_NOMINAL:.3f} "
                "(nominal tf32 / bf16, 1.1 / 2.25 PFLOP/s)")
        dbound, darith = "tensor", ("states recomputed on tcgen05; chain and per-chunk gradients "
                                    "on tf32 mma.sync, fp32 accumulation")
    else:
        dpeak, dsrc = fp32_alu_tflops(2070.0), "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz"
        dbound, darith = "alu", "fp32 CUDA cores"
    decayed_backward = {}
    for form, (r_s, r_launch, dsteps) in dec_bwd.items():
        ls = statistics.mean(r_launch) / 1e3
        decayed_backward[form] = {
            "workload": HEADLINE, "steps": dsteps, "value": world * tokens * dsteps / r_s,
            "unit": "tokens/s", "ms_per_step": 1e3 * r_s / dsteps, "arith": darith,
            "gate": "alpha ~ U(0.9, 1)" + (" per key channel" if form == "kda" else ""),
            "vs_plain_backward": ls / bwd_launch_s,
            "roofline": {"bound": dbound, "achieved": bflops / ls / 1e12, "peak": dpeak,
                         "unit": "TFLOP/s", "frac": bflops / ls / 1e12 / dpeak, "traffic": None,
                         "peak_source": dsrc, "flops_per_launch": bflops,
                         "flops_note": "the plain backward's products (the decay's elementwise "
                                       "work not counted)",
                         "launch_us": ls * 1e6}}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * region_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if tc else "f32", "data": "synthetic (seeded)",
        "config": {"workload": HEADLINE, "B": B, "H": H, "T": T, "dk": dk, "dv": dv, "C": C,
                   "io_dtype": w["dtype"], "state": "fp32", "algo": kname,
                   "workspace_bytes": ws_bytes,
                   "l2": f"inputs {(3 * B * H * T * dk * 2) >> 20} MB > L2 (129 MB), no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "decode": decode,
        "backward": backward,
        "varlen": varlen,
        "qk_prepare": qk_prep,
        "gated": gated,
        "kda": kda,
        "decayed_backward": decayed_backward,
        "e2e": {"value": world * tokens * e2e_steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1e3 * e2e_s / e2e_steps,
                "pipeline": f"{n_sl} batch slices: host->device copies, forward and "
                            "device->host copies (o and the final state) on three streams; "
                            "two device buffer sets in turn, so consecutive steps overlap",
                "copy_only_ms": 1e3 * (h2d / h2d_gbs + d2h / d2h_gbs) / 1e9,
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs},
        "long_prefill": long_prefill,
        "gpu_launches": (launches_per_call * (args.steps + n_sl * e2e_steps)  # chunk fwd, e2e
                         + (long_launches + launches_per_call) * lsteps  # long prefill: split, plain
                         + 2 * nsteps + (nsteps if dec_graph[0] else 0)  # decode (back to back,
                         # then isolated), graph replay
                         + (4 if bwd_tc else 3) * bwd_steps             # recompute, chain, grads
                         + launches_per_call * vsteps                   # varlen
                         + psteps                                       # q/k preparation
                         + launches_per_call * psteps                   # forward preparing q, k
                         + (2 if gneed else 1) * gsteps + gsteps + 2 * nsteps  # gated: both forms, decode
                         + (4 if kneed else 1) * gsteps + ksteps + 2 * nsteps   # KDA: both forms, decode
                         # decayed backwards: recompute (2 or 4 launches on tcgen05, else 1),
                         # chain, gradients
                         + sum((2 + ((4 if f == "kda" else 2) if dec_tc else 1)) * d[2]
                               for f, d in dec_bwd.items())),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, done, cores, el = cpu_oracle_sample(inp, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {
            "value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} batch elements of {HEADLINE} ({done / B:.1f} passes over its {B}; "
                      f"all {H} heads x {T} tokens each), fp64, {el:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def _tc_used(lib, dk, dv, dtype):
    import torch
    # the AUTO policy: tensor cores whenever the tcgen05 path covers the case
    code = 1 if dtype == torch.bfloat16 else 0
    return lib.dn_chunk_fwd_algo(None, None, None, None, None, None, None, 0, 0, 0, dk, dv, 64,
                                 code, None, 0, None, 2) == 0


def _physical_gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", choices=["auto", "simt", "tcgen05"], default="auto")
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workspace", action="store_true",
                    help="tensor-core path without a workspace (the fused kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, sys.argv[1:], script=sys.argv[0]))
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
