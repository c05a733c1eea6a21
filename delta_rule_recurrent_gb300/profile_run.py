"""Runs one workload a few times through the public API, for profiler captures.

    python -m delta_rule_recurrent_gb300.profile_run chunk [--B 8] [--T 2048] [--algo auto] [--reps 3] [--no-workspace] [--qk-l2norm]
    python -m delta_rule_recurrent_gb300.profile_run decode [--B 256] [--steps 4]
    python -m delta_rule_recurrent_gb300.profile_run bwd [--B 8] [--T 2048] [--reps 2]
    python -m delta_rule_recurrent_gb300.profile_run gated [--B 8] [--T 2048] [--reps 3] [--no-workspace]
    python -m delta_rule_recurrent_gb300.profile_run kda [--B 8] [--T 2048] [--reps 3]
    python -m delta_rule_recurrent_gb300.profile_run long [--T 32768] [--reps 2] [--segments 0]
    python -m delta_rule_recurrent_gb300.profile_run gbwd [--B 8] [--T 2048] [--reps 2]
    python -m delta_rule_recurrent_gb300.profile_run kbwd [--B 8] [--T 2048] [--reps 2]

`chunk` runs the chunkwise forward on the 1.3B-layer shape (B8 H16 T2048
dk=dv=128, bf16; B and T can be reduced; the tensor-core path runs in two
passes unless --no-workspace selects its fused kernel); `decode` runs consecutive decoding
steps on the decode workload's shape (B256 H16 dk=dv=128, fp32 state); `bwd`
runs the chunkwise backward (dn_chunk_bwd) on the 1.3B-layer shape; `gated`
runs the Gated DeltaNet chunkwise forward there (keep rates U(0.9, 1); two
tcgen05 passes, or the CUDA-core kernel with --no-workspace); `kda` runs the
KDA chunkwise forward there (per-channel keep rates U(0.9, 1)); `long` runs
the long-prefill shape (B1 H16 T32768, fp32 initial state) through the
sequence split (dn_chunk_fwd_split; --segments 0 fills the GPU once);
`gbwd` and `kbwd` run the Gated DeltaNet and KDA backwards on the 1.3B-layer
shape (keep rates U(0.9, 1), per token or per key channel).
Inputs come from the seeded generators in `workloads`.
"""
from __future__ import annotations

import argparse
import sys
from pathlib import Path

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))


def main(argv=None):
    import torch

    import delta_rule_recurrent_gb300 as dn
    import workloads

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("what", choices=["chunk", "decode", "bwd", "gated", "kda", "long", "gbwd", "kbwd"])
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--algo", default="auto", choices=list(dn.ALGOS))
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--no-workspace", action="store_true")
    ap.add_argument("--segments", type=int, default=0, help="long: runs per sequence")
    ap.add_argument("--qk-l2norm", action="store_true",
                    help="chunk: raw q, k normalised and scaled inside the kernels")
    a = ap.parse_args(argv)
    dev = torch.device("cuda:0")
    if a.what == "chunk":
        over = {k: v for k, v in (("B", a.B), ("T", a.T)) if v is not None}
        inp = workloads.workload_inputs("layer1p3b_bf16", normalize=not a.qk_l2norm, **over)
        q, k, v, b = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta))
        prep = dict(qk_l2norm=True, scale=inp.q.shape[-1] ** -0.5) if a.qk_l2norm else {}
        for _ in range(a.reps):
            o, _ = dn.chunk_fwd(q, k, v, b, algo=a.algo,
                                workspace=None if a.no_workspace else "auto", **prep)
    elif a.what == "gated":
        over = {k: v for k, v in (("B", a.B), ("T", a.T)) if v is not None}
        inp = workloads.workload_inputs("layer1p3b_bf16", **over)
        B, H, T, d = inp.q.shape
        q, k, v, b = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta))
        g = workloads.gate_inputs(B, H, T, seed=7).to(dev)
        for _ in range(a.reps):
            o, _ = dn.chunk_fwd_gated(q, k, v, b, g, workspace=None if a.no_workspace else "auto")
    elif a.what == "kda":
        over = {k: v for k, v in (("B", a.B), ("T", a.T)) if v is not None}
        inp = workloads.workload_inputs("layer1p3b_bf16", **over)
        B, H, T, d = inp.q.shape
        q, k, v, b = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta))
        g = workloads.gate_inputs(B, H, T, seed=7, channels=d).to(dev)
        for _ in range(a.reps):
            o, _ = dn.chunk_fwd_kda(q, k, v, b, g)
    elif a.what == "long":
        over = {"T": a.T} if a.T is not None else {}
        inp = workloads.workload_inputs("long_prefill_bf16", **over)
        q, k, v, b, S0 = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
        for _ in range(a.reps):
            o, _ = dn.chunk_fwd_split(q, k, v, b, initial_state=S0, segments=a.segments)
    elif a.what in ("gbwd", "kbwd"):
        over = {k: v for k, v in (("B", a.B), ("T", a.T)) if v is not None}
        inp = workloads.workload_inputs("layer1p3b_bf16", **over)
        B, H, T, d = inp.q.shape
        d_o, d_S = workloads.grad_inputs(B, H, T, d, d, dtype="bf16", seed=2, ds_std=0.1)
        q, k, v, b, g_o, gS = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta, d_o, d_S))
        kda = a.what == "kbwd"
        g = workloads.gate_inputs(B, H, T, seed=7, channels=d if kda else None).to(dev)
        fn = dn.chunk_bwd_kda if kda else dn.chunk_bwd_gated
        for _ in range(a.reps):
            o = fn(q, k, v, b, g, g_o, d_final_state=gS)[0]
    elif a.what == "bwd":
        over = {k: v for k, v in (("B", a.B), ("T", a.T)) if v is not None}
        inp = workloads.workload_inputs("layer1p3b_bf16", **over)
        B, H, T, d = inp.q.shape
        d_o, d_S = workloads.grad_inputs(B, H, T, d, d, dtype="bf16", seed=2, ds_std=0.1)
        q, k, v, b, g, gS = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.beta, d_o, d_S))
        for _ in range(a.reps):
            o = dn.chunk_bwd(q, k, v, b, g, d_final_state=gS)[0]
    else:
        w = workloads.WORKLOADS["decode_bf16"]
        B = a.B or w["B"]
        q, k, v, b = workloads.decode_inputs_on_device(B, w["H"], w["dk"], w["dv"], a.steps,
                                                       seed=3, device=dev)
        S = torch.randn(B, w["H"], w["dk"], w["dv"], device=dev) * w["s0_std"]
        for i in range(a.steps):
            o = dn.recurrent_step(q[i], k[i], v[i], b[i], S)
    torch.cuda.synchronize()
    print("ok", float(o.float().abs().mean()))


if __name__ == "__main__":
    main()
