"""Benchmark: gated-subspace linear maps of a 6B-class decoder layer at batch 1.

Workload (one "step"): the four projections of a 6B-class layer (fused QKV
12288x4096, output 4096x4096, MLP up 16384x4096, MLP down 4096x16384), bf16
weights, k = 256, eps = 0.05, and 256 sequential single-token decode steps;
each decode step runs the gated map over the four projections in order
(gsi_stack with T = 1), so one step is 1024 gated-map calls.  Per map, exactly
26 of the 256 tokens (10%) have rho >= eps (two-level noise mixture).

Weights rotate over R replicas of the layer (distinct device copies) so the
working set of consecutive decode steps does not sit in L2: 8 replicas put
~269 MB of fast-path weights (V, Gram, M) and ~3.2 GB of W behind the 129 MB
L2, as the 28 distinct layers of a real model would.

Printed: one JSON line with tokens/s (the whole step: 256 tokens through the
layer's four maps), the achieved HBM bandwidth of the step and of the
dominant kernel against the measured peak, an end-to-end figure through the
public API with host buffers, and the float64 oracle timed on the host cores.
`--impl reference` times the oracle alone on the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import synth  # noqa: E402

T_TOKENS = 256
EPS = synth.EPS
K_RANK = 256
N_SLOW = 26


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s, burst): measured, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_inputs():
    """The four 6B maps with their 256 tokens each (CPU, storage dtype)."""
    return [synth.map_6b(role, T=T_TOKENS, n_slow=N_SLOW, k=K_RANK) for role in synth.ROLES]


def map_bytes(m):
    es = 2
    return dict(V=m.d * m.k * es, gram=m.k * m.k * 4, M=m.d_out * m.k * es, W=m.d_out * m.d * es,
                x=m.d * es, y=m.d_out * 4)


def algorithmic_bytes(maps_in, flags_np):
    """Bytes the method must move for the whole step (the algorithmic model):
    per call |V| + |Gram| + x + y + flag, plus |M| if fast or |W| if slow."""
    total = fast_apply = slow_apply = gate = 0
    n_fast = n_slow = 0
    for m, f in zip(maps_in, flags_np):
        b = map_bytes(m)
        ns = int(f.sum())
        nf = len(f) - ns
        g = b["V"] + b["gram"] + b["x"] + m.k * 4 + 4 + 1
        gate += g * len(f)
        fast_apply += nf * (b["M"] + m.k * 4 + b["y"])
        slow_apply += ns * (b["W"] + b["x"] + b["y"])
        n_fast += nf
        n_slow += ns
    total = gate + fast_apply + slow_apply
    dense = sum((map_bytes(m)["W"] + map_bytes(m)["x"] + map_bytes(m)["y"]) * len(f)
                for m, f in zip(maps_in, flags_np))
    return dict(total=total, gate=gate, fast=fast_apply, slow=slow_apply, dense=dense,
                n_fast=n_fast, n_slow=n_slow)


# ---------------------------------------------------------------------------- oracle (CPU)
def oracle_step(maps64, tokens, eps):
    """The float64 oracle over `tokens` decode steps through the four maps."""
    from oracle import gsi_oracle as orc

    for t in tokens:
        for (W, M, V, X) in maps64:
            orc.gsi_linear(W, M, V, X[t:t + 1], eps)


def oracle_maps(maps_in, M_list=None):
    from oracle import gsi_oracle as orc

    out = []
    for i, m in enumerate(maps_in):
        W, V, X = synth.widen(m.W), synth.widen(m.V), synth.widen(m.X)
        M = synth.widen(M_list[i]) if M_list is not None else orc.image(W, V)
        out.append((W, M, V, X))
    return out


def time_oracle(maps64, eps, min_seconds):
    """Repeat full 256-token passes of the oracle until min_seconds have passed."""
    toks = list(range(T_TOKENS))
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(maps64, toks, eps)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return passes * T_TOKENS / dt, dt, passes


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def combine_ranks(ms, world, dist=None, device=None):
    """The whole job's step time and throughput: every rank runs its own
    replica of the workload (no data-path collective), so the job's step
    takes the slowest rank's time (all-reduce MAX) and the job processes
    T_TOKENS tokens per rank per step.  Returns (ms, tokens per second)."""
    if dist is not None and world > 1:
        t = torch.tensor([float(ms)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, T_TOKENS * world / (ms / 1e3)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    maps_in = make_inputs()
    maps64 = oracle_maps(maps_in)
    n_tok = args.ref_tokens
    for _ in range(args.warmup):
        oracle_step(maps64, range(min(4, n_tok)), EPS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(maps64, range(n_tok), EPS)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    line = {
        "impl": "reference", "metric": "gsi_linear_tokens_per_s_batch1", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "6B-class layer linears (qkv/out/up/down), bf16 stored, batch-1 decode, "
                               f"k={K_RANK}, eps={EPS}, 10% slow tokens",
                   "tokens_per_step": n_tok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"{n_tok} of the 256 decode tokens per step, all four maps, "
                                   "float64 numpy oracle on host cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------- GPU
# DRAM bytes per launch of the step's kernel (decode_kernel, one launch per
# gated-map call), from one ncu capture of `bench.py --kernel-traffic`
# (dram__bytes_read.sum + dram__bytes_write.sum over decode_kernel launches
# 1-1024, i.e. exactly the step's calls, with --cache-control none so that
# the L2 prefetch of the next map serves the next launch as in the live
# step): valid only for the kernel source it was taken on (first 16 hex
# digits of the SHA-256 of csrc/gsi_decode.cu followed by csrc/gsi_plan.h);
# otherwise the roofline reports traffic null.
KERNEL_TRAFFIC = {"src_sha256": "26891ad75c152d51", "bytes_per_launch": 19428989.5}
TRAFFIC_SOURCES = ("gsi_decode.cu", "gsi_plan.h")


def kernel_source_hash():
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gated_rank_subspace_gb300", "csrc")
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic():
    return KERNEL_TRAFFIC["bytes_per_launch"] if kernel_source_hash() == KERNEL_TRAFFIC["src_sha256"] else None


def call_bytes(d, d_out, k, T, n_fast, n_slow, es=2):
    """Algorithmic bytes of one gated-map call of T tokens: V_k and its Gram,
    M if any token is fast, W if any is slow, and per token x in, y out,
    g and rho and the flag: |V| + |Gram| + [n_f > 0] |M| + [n_s > 0] |W|
    + T (d s_x + d_out 4 + k 4 + 5)."""
    return (d * k * es + k * k * 4 + (d_out * k * es if n_fast else 0) + (d_out * d * es if n_slow else 0)
            + T * (d * es + d_out * 4 + k * 4 + 5))


def dense_bytes(d, d_out, T, es=2):
    """The dense map's bytes for the same call: W once, x in, y out."""
    return d_out * d * es + T * (d * es + d_out * 4)


def graph_time_ms(fn, stream, reps, warm=2):
    """Mean time of one call of fn, captured in a CUDA graph, over reps replays."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / reps


def run_config3(gsi, dev, stream, hbm_peak, steps=64, reps=2):
    """The 28-layer linear-only stack of the 6B shapes (depth-coherent bases,
    per-layer slow fraction 5-15%): `steps` single-token decode steps, each one
    gsi_stack call over the 112 maps (one decode launch per map), all steps in
    one CUDA graph.  Tokens/s counts one token per 28-layer step."""
    L = 28
    bases, fr, base_W, tokens = synth.stack_config3(L, steps)
    maps, Xs = [], []
    for role in synth.ROLES:
        base_W[role] = base_W[role].to(dev)
    for l in range(L):
        for role in synth.ROLES:
            d_out, d = synth.SHAPES_6B[role]
            perm, signs = synth.layer_weight_rows(3, l, synth.ROLE_ID[role], d_out)
            W = (base_W[role][torch.from_numpy(perm).to(dev)] *
                 torch.from_numpy(signs).to(dev, torch.bfloat16)[:, None]).contiguous()
            maps.append(gsi.make_map(W, synth.storage(bases[role][l], torch.bfloat16).to(dev)))
            Xs.append(tokens[(l, role)].to(dev))
    del base_W
    Ys = [torch.zeros(steps, m.d_out, device=dev) for m in maps]
    Fs = [torch.zeros(steps, dtype=torch.uint8, device=dev) for _ in maps]
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, 1), dev)
    args = [gsi.stack_args(maps, [X[t:t + 1] for X in Xs], [Y[t:t + 1] for Y in Ys], [F[t:t + 1] for F in Fs])
            for t in range(steps)]
    torch.cuda.synchronize()

    def run():
        for a in args:
            gsi.stack_raw(a, len(maps), 1, EPS, ws, stream=stream)

    ms = graph_time_ms(run, stream, reps)
    assert gsi.workspace_status(ws, stream=stream) == 0
    flags = [F.cpu().numpy().astype(bool) for F in Fs]
    nbytes = dense = 0
    for m, f in zip(maps, flags):
        for t in range(steps):
            nbytes += call_bytes(m.d, m.d_out, m.k, 1, int(not f[t]), int(f[t]))
            dense += dense_bytes(m.d, m.d_out, 1)
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {"workload": "28-layer linear-only stack, 6B shapes, depth-coherent bases, k=256, eps=0.05, "
                       f"{steps} single-token decode steps (one gsi_stack call of 112 maps per step)",
           "tokens_per_s": steps / (ms * 1e-3), "ms_per_token": ms / steps, "achieved_gbs": gbs,
           "frac_of_hbm_peak": gbs / hbm_peak, "bytes_saved_vs_dense": dense / nbytes,
           "slow_fraction": float(np.mean([f.mean() for f in flags])),
           "kernel": "decode_kernel (one launch per gated-map call, 112 per step)"}
    del maps, Xs, Ys, Fs, args, ws
    torch.cuda.empty_cache()
    return out


def config4_maps(gsi, dev, L=40):
    """The 40-layer 13B stack on the device (layer weights and bases derived
    from per-role base draws, see synth.stack_config4); returns (maps, pools)."""
    base_W, V64, rows, cols, pools = synth.stack_config4(L)
    maps = []
    for role in synth.ROLES:
        base_W[role] = base_W[role].to(dev)
    Vb = {r: synth.storage(V64[r], torch.bfloat16).to(dev) for r in synth.ROLES}
    for l in range(L):
        for role in synth.ROLES:
            perm, signs = rows[(l, role)]
            W = (base_W[role][torch.from_numpy(perm).to(dev)] *
                 torch.from_numpy(signs).to(dev, torch.bfloat16)[:, None]).contiguous()
            V = Vb[role][:, torch.from_numpy(cols[(l, role)]).to(dev)].contiguous()
            maps.append(gsi.make_map(W, V))
    return maps, pools


def run_config4(gsi, dev, stream, hbm_peak, reps=2):
    """13B linears, 40 layers, k=320, small-batch decode: T in {1, 4, 16}
    tokens per call, slow fraction f in {0, 5, 25, 100}% (per-token Bernoulli
    labels); every decode step is one gsi_stack call over the 160 maps.  Per
    point: tokens/s of the 40-layer model, GB/s of the algorithmic bytes, and
    the bytes saved against dense W x (a call reads W when any of its T
    tokens is slow)."""
    L = 40
    maps, pools = config4_maps(gsi, dev, L)
    ws = gsi.new_workspace(max(gsi.stack_workspace_size(maps, T) for T in (1, 4, 16)), dev)
    points = []
    for T, steps in ((1, 16), (4, 8), (16, 4)):
        for f in (0.0, 0.05, 0.25, 1.0):
            n = T * steps
            Xs, Ys, Fs = [], [], []
            for l in range(L):
                for role in synth.ROLES:
                    Xs.append(synth.pool_tokens(pools, role, l, n, f, salt=int(T * 100 + f * 100)).to(dev))
            for m in maps:
                Ys.append(torch.zeros(n, m.d_out, device=dev))
                Fs.append(torch.zeros(n, dtype=torch.uint8, device=dev))
            args = [gsi.stack_args(maps, [X[s * T:(s + 1) * T] for X in Xs], [Y[s * T:(s + 1) * T] for Y in Ys],
                                   [F[s * T:(s + 1) * T] for F in Fs]) for s in range(steps)]

            def run():
                for a in args:
                    gsi.stack_raw(a, len(maps), T, EPS, ws, stream=stream)

            ms = graph_time_ms(run, stream, reps)
            assert gsi.workspace_status(ws, stream=stream) == 0
            nbytes = dense = 0
            n_slow = 0
            for m, F in zip(maps, Fs):
                fl = F.cpu().numpy().astype(bool).reshape(steps, T)
                n_slow += int(fl.sum())
                for s in range(steps):
                    ns = int(fl[s].sum())
                    nbytes += call_bytes(m.d, m.d_out, m.k, T, T - ns, ns)
                    dense += dense_bytes(m.d, m.d_out, T)
            gbs = nbytes / (ms * 1e-3) / 1e9
            points.append({"T": T, "f": f, "tokens_per_s": n / (ms * 1e-3), "ms_per_step": ms / steps,
                           "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
                           "bytes_saved_vs_dense": dense / nbytes,
                           "slow_fraction": n_slow / (n * len(maps))})
            del Xs, Ys, Fs, args
    out = {"workload": "13B-class linears (qkv 15360x5120, out 5120^2, up 13824x5120, down 5120x13824), "
                       "40 layers, bf16, k=320, eps=0.05; each decode step one gsi_stack call over the 160 maps",
           "points": points,
           "kernels": "T=1: decode_kernel per map; T=4, 16: batch_decode_kernel (small-batch decode) per map"}
    del maps, ws
    torch.cuda.empty_cache()
    return out


def run_config5(gsi, dev, stream, hbm_peak, tflops_peak, reps=20, R=2):
    """The prefill-sized map (T=2048, d=4096, d_out=16384, k=256, 410 slow
    tokens) on the tensor-core path, calls alternating over R weight
    replicas."""
    m_in = synth.config5()
    base = gsi.make_map(m_in.W.to(dev), m_in.V.to(dev))
    reps_m = [base] + [gsi.Map(base.W.clone(), base.V.clone(), base.M.clone(), base.gram.clone())
                       for _ in range(R - 1)]
    X = m_in.X.to(dev)
    T = X.shape[0]
    Y = torch.zeros(T, base.d_out, device=dev)
    F = torch.zeros(T, dtype=torch.uint8, device=dev)
    ws = gsi.new_workspace(gsi.workspace_size(base, T, "auto"), dev)

    def run():
        for m in reps_m:
            gsi.linear(m, X, EPS, Y=Y, flags=F, workspace=ws, want_rho=False, stream=stream)

    ms = graph_time_ms(run, stream, reps) / R
    assert gsi.workspace_status(ws, stream=stream) == 0
    ns = int(F.sum())
    nf = T - ns
    d, d_out, k = base.d, base.d_out, base.k
    flop = 2 * (T * d * k + nf * d_out * k + ns * d_out * d)
    nbytes = call_bytes(d, d_out, k, T, nf, ns)
    out = {"workload": "prefill-sized map: T=2048, d=4096, d_out=16384, k=256, 410 slow tokens, bf16, "
                       "tensor-core path (gsi_linear AUTO)",
           "tokens_per_s": T / (ms * 1e-3), "us_per_call": ms * 1e3,
           "tflops": flop / (ms * 1e-3) / 1e12, "frac_of_bf16_peak": flop / (ms * 1e-3) / 1e12 / tflops_peak,
           "achieved_gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
           "gflop_per_call": flop / 1e9, "dense_gflop_per_call": 2 * T * d_out * d / 1e9, "n_slow": ns}
    del reps_m, base, X, Y, F, ws
    torch.cuda.empty_cache()
    return out


SWEEP_EPS = [0.0, 0.0125, 0.025, 0.05, 0.1, 0.2, 0.4, float("inf")]


def run_sweep():
    """The gate's trade-off across thresholds (eps = inf: static projection)
    on configs 2-4, from the library's gsi_path_errors and gsi_eps_sweep:
    slow fraction, relative output error against dense W x, modelled bytes
    per token (W read by a call when any of its tokens is slow) and effective
    parameters per token.  Prints one JSON line."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    dev = torch.device("cuda")
    n_eps = len(SWEEP_EPS)

    def one_map(W, V, X, tpc):
        gm = gsi.make_map(W.to(dev), V.to(dev))
        Xd = X.to(dev)
        _, _, rho, err, ynorm = gsi.path_errors(gm, Xd)
        ns, nc, _ = gsi.eps_sweep(rho, err, ynorm, SWEEP_EPS, tpc)
        T, (d_out, d), k = X.shape[0], W.shape, V.shape[1]
        es = W.element_size()
        r = rho.cpu().numpy()
        n_calls = (T + tpc - 1) // tpc
        fast_calls = [sum(bool((r[c:c + tpc] < e).any()) for c in range(0, T, tpc)) for e in SWEEP_EPS]
        fixed = n_calls * (d * k * es + k * k * 4) + T * (d * es + d_out * 4)
        nbytes = [fixed + fc * d_out * k * es + sc * d_out * d * es for fc, sc in zip(fast_calls, nc.cpu().tolist())]
        dense = n_calls * d_out * d * es + T * (d * es + d_out * 4)
        e2 = (err.double() ** 2).cpu().numpy()
        e2_fast = [float(e2[r < e].sum()) for e in SWEEP_EPS]  # fast tokens (NaN: slow)
        out = dict(T=T, ns=ns.cpu().tolist(), e2=e2_fast, y2=float((ynorm.double() ** 2).sum()), bytes=nbytes,
                   dense=dense, params=(d_out * k, d_out * d))
        del gm, Xd, rho, err, ynorm
        return out

    def summarize(parts, tokens):
        y2 = sum(p["y2"] for p in parts)
        rows = []
        for i in range(n_eps):
            slow = sum(p["ns"][i] for p in parts) / sum(p["T"] for p in parts)
            eff = sum(((p["T"] - p["ns"][i]) * p["params"][0] + p["ns"][i] * p["params"][1]) / p["T"] for p in parts)
            b = sum(p["bytes"][i] for p in parts) / tokens
            rows.append({"eps": SWEEP_EPS[i] if math.isfinite(SWEEP_EPS[i]) else "inf",
                         "slow_fraction": slow,
                         "rel_err": math.sqrt(sum(p["e2"][i] for p in parts) / y2),
                         "max_map_rel_err": max(math.sqrt(p["e2"][i] / p["y2"]) for p in parts),
                         "MB_per_token": b / 1e6,
                         "saved_vs_dense": sum(p["dense"] for p in parts) / tokens / b,
                         "effective_params_per_token": eff})
        return rows

    report = {"metric": "gsi_eps_sweep", "data": "synthetic", "rows_per_config": {}}
    # config 2: the bench's 6B layer maps, 256 single-token calls each
    parts = [one_map(m.W, m.V, m.X, 1) for m in make_inputs()]
    report["rows_per_config"]["cfg2 6B layer, 256 tokens, T=1 calls"] = summarize(parts, T_TOKENS)
    # config 3: the first 4 layers of the depth-coherent 28-layer stack, 64 steps
    bases, fr, base_W, tokens = synth.stack_config3(n_layers=4, steps=64)
    parts = []
    for l in range(4):
        for role in synth.ROLES:
            perm, signs = synth.layer_weight_rows(3, l, synth.ROLE_ID[role], base_W[role].shape[0])
            W = (base_W[role][torch.from_numpy(perm)] * torch.from_numpy(signs).to(torch.bfloat16)[:, None]).contiguous()
            parts.append(one_map(W, synth.storage(bases[role][l], torch.bfloat16), tokens[(l, role)], 1))
    report["rows_per_config"]["cfg3 stack layers 0-3, 64 steps, T=1 calls"] = summarize(parts, 64)
    # config 4: 13B maps (k = 320), calls of 16 tokens, Bernoulli slow labels
    for f in (0.0, 0.05, 0.25, 1.0):
        parts = []
        for role in synth.ROLES:
            d_out, d = synth.SHAPES_13B[role]
            r = synth.ROLE_ID[role]
            V64 = synth.orthonormal_basis(synth.rng(4, 0, r, 1), d, 320)
            W = synth.storage(synth.gaussian_weight(synth.rng(4, 0, r, 2), d_out, d), torch.bfloat16)
            X = synth.map_tokens(4, 0, r, V64, 64, f, bernoulli=True)
            parts.append(one_map(W, synth.storage(V64, torch.bfloat16), X, 16))
        report["rows_per_config"][f"cfg4 13B layer, f={f}, 64 tokens, T=16 calls"] = summarize(parts, 64)
    print(json.dumps(report))


def run_cascade(n_layers=4, d=4096, m=512, k=256, T=2048, target=0.999, ref_steps=100, cap=100):
    """Basis construction on depth-coherent calibration blocks (bf16, 6B
    width, spectrum 0.995^i with a gap of 0.5 at k): for each layer, the
    steps until the basis is within `target` coherence of that layer's
    converged basis (`ref_steps` steps from a random start), from a random
    start and from the previous layer's basis (the cascade); the depth
    coherence of consecutive layers' bases.  Prints one JSON line."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    dev = torch.device("cuda")
    U, blocks = synth.calibration_stream(6, n_layers, d=d, m=m, T=T, decay=0.995, gap_at=k, gap=0.5)
    Xs = [synth.storage(b, torch.bfloat16).to(dev) for b in blocks]
    work = gsi.new_workspace(int(gsi.lib().gsi_basis_step_work_bytes(T, d, k)), dev)

    def start(l, salt):
        Vt = torch.tensor(synth.random_basis_t(6, k, d, salt=100 * l + salt), dtype=torch.float32, device=dev)
        gsi.basis_orthonormalize(Vt)
        return Vt

    def steps_to(X, Vt, ref):
        c = gsi.basis_coherence(Vt, ref).item()
        n = 0
        while c < target and n < cap:
            gsi.basis_step(X, Vt, work)
            n += 1
            c = gsi.basis_coherence(Vt, ref).item()
        return n, c

    # time of one step (two contractions of 2 T d k flop each, then DGKS)
    Vt = start(0, 9)
    for _ in range(2):
        gsi.basis_step(Xs[0], Vt, work)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        gsi.basis_step(Xs[0], Vt, work)
    e1.record()
    torch.cuda.synchronize()
    step_ms = e0.elapsed_time(e1) / 5
    layers, prev = [], None
    for l in range(n_layers):
        ref = start(l, 1)
        for _ in range(ref_steps):
            gsi.basis_step(Xs[l], ref, work)
        n_cold, c_cold = steps_to(Xs[l], start(l, 2), ref)
        row = {"layer": l, "cold_steps": n_cold, "cold_coherence": c_cold}
        if prev is not None:
            warm = prev.clone()
            row["start_coherence"] = gsi.basis_coherence(warm, ref).item()
            n_warm, c_warm = steps_to(Xs[l], warm, ref)
            row.update(warm_steps=n_warm, warm_coherence=c_warm,
                       saving=1 - n_warm / n_cold if n_cold else 0.0,
                       depth_coherence=gsi.basis_coherence(prev, ref).item())
        layers.append(row)
        prev = ref
    report = {"metric": "gsi_basis_cascade", "data": "synthetic",
              "config": {"d": d, "k": k, "calibration_tokens": T, "dtype": "bf16 tokens, f32 basis",
                         "spectrum": f"0.995^i over {m} directions, x0.5 from direction {k} on",
                         "chain": "U(l+1) = orth(U(l) + 0.1 N/sqrt(d))",
                         "target": f"coherence >= {target} with the layer's basis after {ref_steps} steps"},
              "step_ms": step_ms, "step_gflop": 4 * T * d * k / 1e9,
              "step_tflops": 4 * T * d * k / (step_ms * 1e-3) / 1e12, "layers": layers}
    print(json.dumps(report))


def run_per_call(R=4, n=32, reps_n=10):
    """Latency of one gated-map call per 6B map: a CUDA graph of n
    single-token calls (weights rotating over R device replicas, so W of a
    slow call comes from HBM), timed with CUDA events over reps_n replays,
    once with every token slow (eps = 0) and once with every token fast
    (eps = inf).  One JSON line per map."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    dev = torch.device("cuda", 0)
    for role in synth.ROLES:
        m_in = synth.map_6b(role, T=n, n_slow=0, k=K_RANK)
        base = gsi.make_map(m_in.W.to(dev), m_in.V.to(dev))
        reps = [base] + [gsi.Map(base.W.clone(), base.V.clone(), base.M.clone(), base.gram.clone())
                         for _ in range(R - 1)]
        X = m_in.X.to(dev)
        Y = torch.zeros(n, base.d_out, device=dev)
        F = torch.zeros(n, dtype=torch.uint8, device=dev)
        ws = gsi.new_workspace(gsi.stack_workspace_size([base], 1), dev)
        stream = torch.cuda.Stream(dev)
        args = [gsi.stack_args([reps[t % R]], [X[t:t + 1]], [Y[t:t + 1]], [F[t:t + 1]]) for t in range(n)]
        torch.cuda.synchronize()
        out = {"per_call": role, "calls": n, "replicas": R}
        for key, eps in (("slow", 0.0), ("fast", float("inf"))):
            def run():
                for a in args:
                    gsi.stack_raw(a, 1, 1, eps, ws, stream=stream)

            with torch.cuda.stream(stream):
                run()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                e0.record(stream)
                for _ in range(reps_n):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps_n * n)
            out[key + "_us"] = round(us, 2)
            mb = map_bytes(m_in)
            moved = mb["V"] + mb["gram"] + (mb["W"] if key == "slow" else mb["M"]) + mb["x"] + mb["y"]
            out[key + "_gbs"] = round(moved / (us * 1e-6) / 1e9, 1)
        assert int(F.sum()) == 0 and gsi.workspace_status(ws, stream=stream) == 0
        print(json.dumps(out))


def probe_stack(n_tokens=16, R=2):
    """A small case of the bench step for ncu: the four 6B maps over 2 device
    replicas (about 1 GB of weights), n_tokens decode steps, each one
    gsi_stack call (one decode_kernel launch per map), run once.  Prints the
    algorithmic bytes of every launch in launch order (JSON line) so that an
    ncu capture of a few of them can be compared with what they had to
    move."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    dev = torch.device("cuda", 0)
    maps_in = [synth.map_6b(role, T=n_tokens, n_slow=max(1, n_tokens // 8), k=K_RANK) for role in synth.ROLES]
    base = [gsi.make_map(m.W.to(dev), m.V.to(dev)) for m in maps_in]
    reps = [base] + [[gsi.Map(b.W.clone(), b.V.clone(), b.M.clone(), b.gram.clone()) for b in base]
                     for _ in range(R - 1)]
    Xs = [m.X.to(dev) for m in maps_in]
    Ys = [torch.zeros(n_tokens, m.d_out, device=dev) for m in maps_in]
    Fs = [torch.zeros(n_tokens, dtype=torch.uint8, device=dev) for _ in maps_in]
    ws = gsi.new_workspace(gsi.stack_workspace_size(base, 1), dev)
    torch.cuda.synchronize()
    for t in range(n_tokens):
        gsi.stack(reps[t % R], [X[t:t + 1] for X in Xs], EPS, Ys=[Y[t:t + 1] for Y in Ys],
                  flags=[F[t:t + 1] for F in Fs], workspace=ws)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    flags = [F.cpu().numpy().astype(bool) for F in Fs]
    per_launch = [call_bytes(m.d, m.d_out, m.k, 1, int(not f[t]), int(f[t]))
                  for t in range(n_tokens) for m, f in zip(base, flags)]
    print(json.dumps({"probe_stack": n_tokens, "replicas": R, "algorithmic_bytes_per_launch": per_launch,
                      "slow_per_launch": [int(f[t]) for t in range(n_tokens) for f in flags]}))


def probe_batch(spec, L=2, steps=4):
    """A small case of the 13B small-batch stack for ncu: L layers of the
    four 13B maps (k=320, about 1 GB of weights per layer), `steps` decode
    steps of T tokens with slow fraction f (spec "T:f"), each step one
    gsi_stack call, run once.  Prints the algorithmic bytes of every call in
    call order (JSON line)."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    T, f = spec.split(":")
    T, f = int(T), float(f)
    dev = torch.device("cuda", 0)
    maps, pools = config4_maps(gsi, dev, L)
    n = T * steps
    Xs = [synth.pool_tokens(pools, role, l, n, f, salt=int(T * 100 + f * 100)).to(dev)
          for l in range(L) for role in synth.ROLES]
    Ys = [torch.zeros(n, m.d_out, device=dev) for m in maps]
    Fs = [torch.zeros(n, dtype=torch.uint8, device=dev) for _ in maps]
    ws = gsi.new_workspace(gsi.stack_workspace_size(maps, T), dev)
    torch.cuda.synchronize()
    for s in range(steps):
        a = gsi.stack_args(maps, [X[s * T:(s + 1) * T] for X in Xs], [Y[s * T:(s + 1) * T] for Y in Ys],
                           [F[s * T:(s + 1) * T] for F in Fs])
        gsi.stack_raw(a, len(maps), T, EPS, ws)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    fl = [F.cpu().numpy().astype(bool).reshape(steps, T) for F in Fs]
    per_call = [call_bytes(m.d, m.d_out, m.k, T, T - int(x[s].sum()), int(x[s].sum()))
                for s in range(steps) for m, x in zip(maps, fl)]
    print(json.dumps({"probe_batch": spec, "layers": L, "steps": steps, "algorithmic_bytes_per_call": per_call,
                      "slow_per_call": [int(x[s].sum()) for s in range(steps) for x in fl]}))


def probe_map(role, eps):
    """Eight one-token gsi_linear calls of one 6B map (default stream)."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    m_in = synth.map_6b(role, T=1, n_slow=0)
    m = gsi.make_map(m_in.W.cuda(), m_in.V.cuda())
    X = m_in.X.cuda()
    ws = gsi.new_workspace(gsi.workspace_size(m, 1))
    Y = torch.empty(1, m.d_out, device="cuda")
    F = torch.empty(1, dtype=torch.uint8, device="cuda")
    for _ in range(8):
        gsi.linear(m, X, eps, Y=Y, flags=F, workspace=ws, want_rho=False)
    torch.cuda.synchronize()
    print(json.dumps({"probe_map": role, "eps": eps, "flag": int(F[0])}))


def probe_prefill(calls=3):
    """A small case of the prefill map for ncu: `calls` gsi_linear calls of
    the T=2048 map (AUTO: the tensor-core path) on the default stream."""
    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    m_in = synth.config5()
    m = gsi.make_map(m_in.W.cuda(), m_in.V.cuda())
    X = m_in.X.cuda()
    T = X.shape[0]
    ws = gsi.new_workspace(gsi.workspace_size(m, T, "auto"))
    Y = torch.empty(T, m.d_out, device="cuda")
    F = torch.empty(T, dtype=torch.uint8, device="cuda")
    for _ in range(calls):
        gsi.linear(m, X, EPS, Y=Y, flags=F, workspace=ws, want_rho=False)
    torch.cuda.synchronize()
    assert gsi.workspace_status(ws) == 0
    print(json.dumps({"probe_prefill": calls, "n_slow": int(F.sum())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-traffic", action="store_true",
                    help="only run the step once eagerly (1024 decode_kernel launches), then its 1024 gate and "
                         "1024 apply launches, and print each decode launch's algorithmic bytes (the command an "
                         "ncu DRAM-byte capture of a few decode launches profiles)")
    ap.add_argument("--probe-map", choices=["qkv", "out", "up", "down"], default=None,
                    help="only run 8 one-token gsi_linear calls of this 6B map (a small case for ncu)")
    ap.add_argument("--probe-stack", type=int, default=0,
                    help="only run this many decode steps of the bench's four maps (2 weight replicas, one "
                         "decode_kernel launch per map) and print each launch's algorithmic bytes "
                         "(a small case for ncu)")
    ap.add_argument("--probe-batch", default=None, metavar="T:f",
                    help="only run 4 decode steps of T tokens (slow fraction f) through 2 layers of the 13B "
                         "maps and print each call's algorithmic bytes (a small case for ncu)")
    ap.add_argument("--probe-prefill", action="store_true",
                    help="only run 3 calls of the prefill map (T=2048, tensor-core path; a small case for ncu)")
    ap.add_argument("--probe-eps", type=float, default=0.0,
                    help="threshold of the --probe-map calls (0: every token slow)")
    ap.add_argument("--eps-sweep", action="store_true",
                    help="only report the threshold sweep on configs 2-4 (one JSON line)")
    ap.add_argument("--per-call", action="store_true",
                    help="only report one call's latency per 6B map, all tokens slow and all fast (JSON lines)")
    ap.add_argument("--cascade", action="store_true",
                    help="only report basis construction on depth-coherent calibration blocks (one JSON line)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (28-layer stack, 13B small-batch stack, prefill map)")
    ap.add_argument("--oracle-probe", action="store_true",
                    help="only time the oracle on the bench workload's tokens (JSON line; thread count from the "
                         "environment), as the single-thread leg of the CPU baseline")
    args = ap.parse_args()
    if args.oracle_probe:
        maps_in = make_inputs()
        v, dt, passes = time_oracle(oracle_maps(maps_in), EPS, args.cpu_seconds)
        print(json.dumps({"value": v, "seconds": dt, "passes": passes}))
        return
    if args.cascade:
        run_cascade()
        return
    if args.per_call:
        run_per_call()
        return
    if args.eps_sweep:
        run_sweep()
        return
    if args.probe_map:
        probe_map(args.probe_map, args.probe_eps)
        return
    if args.probe_stack:
        probe_stack(args.probe_stack)
        return
    if args.probe_batch:
        probe_batch(args.probe_batch)
        return
    if args.probe_prefill:
        probe_prefill()
        return
    if args.impl == "reference":
        run_reference(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod

    import __graft_entry__

    __graft_entry__.build()
    import gated_rank_subspace_gb300 as gsi

    dev = torch.device("cuda", local)
    maps_in = make_inputs()
    R = args.replicas
    # replicas: distinct device copies of every map's W, V, M, Gram
    base = []
    for m in maps_in:
        W, V = m.W.to(dev), m.V.to(dev)
        base.append(gsi.make_map(W, V))
    reps = [base]
    for _ in range(1, R):
        reps.append([gsi.Map(b.W.clone(), b.V.clone(), b.M.clone(), b.gram.clone()) for b in base])
    Xs = [m.X.to(dev) for m in maps_in]
    Ys = [torch.zeros(T_TOKENS, m.d_out, device=dev) for m in maps_in]
    Fs = [torch.zeros(T_TOKENS, dtype=torch.uint8, device=dev) for _ in maps_in]
    ws = gsi.new_workspace(gsi.stack_workspace_size(base, 1), dev)
    args_t = [gsi.stack_args(reps[t % R], [X[t:t + 1] for X in Xs], [Y[t:t + 1] for Y in Ys],
                             [F[t:t + 1] for F in Fs]) for t in range(T_TOKENS)]
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()  # uploads and the workspace zeroing ran on the default stream

    def step():
        for t in range(T_TOKENS):
            gsi.stack_raw(args_t[t], 4, 1, EPS, ws, stream=stream)

    # eager run once (validates the step), then capture the whole step
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    if not args.kernel_traffic:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                graph.replay()
        stream.synchronize()
        assert gsi.workspace_status(ws, stream=stream) == 0

        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks = sampler.stop()
        ms, tokens_per_s = combine_ranks(e0.elapsed_time(e1) / args.steps, world, dist, dev)

        flags_np = [F.cpu().numpy().astype(bool) for F in Fs]
        ab = algorithmic_bytes(maps_in, flags_np)
        step_gbs = ab["total"] / (ms * 1e-3) / 1e9
        hbm_peak, peak_kind = peaks()

    # launches per gated-map call: one on the single-launch decode (AUTO's
    # choice for one token where a slab of V fits), two on the streaming path
    per_call = []
    for b in base:
        try:
            gsi.workspace_size(b, 1, "fused")
            per_call.append(1)
        except gsi.GsiError:
            per_call.append(2)
    # ---- per-kernel timing: the same 1024 calls split into their two launches
    # (gsi_gate then gsi_apply, each call with its own workspace), and each
    # kernel's launches captured in a CUDA graph of their own so that they run
    # back to back as in the step; one graph for the gate launches, and one
    # graph each for the apply launches of fast and of slow calls.
    n_launch = T_TOKENS * 4
    ws_one = gsi.workspace_size(base[0], 1)
    for b in base[1:]:
        ws_one = max(ws_one, gsi.workspace_size(b, 1))
    ws_one = (ws_one + 255) // 256 * 256
    ws_all = gsi.new_workspace(ws_one * n_launch, dev)
    G_all = torch.empty(n_launch, K_RANK, device=dev)
    rho_all = torch.empty(n_launch, device=dev)
    Yk = [torch.empty_like(Y) for Y in Ys]
    Fk = [torch.empty_like(F) for F in Fs]
    torch.cuda.synchronize()
    calls = [(t, i) for t in range(T_TOKENS) for i in range(4)]

    def wsl(c):
        return ws_all[c * ws_one:(c + 1) * ws_one]

    def run_gates():
        for c, (t, i) in enumerate(calls):
            gsi.gate(reps[t % R][i], Xs[i][t:t + 1], EPS, workspace=wsl(c), G=G_all[c:c + 1],
                     rho=rho_all[c:c + 1], flags=Fk[i][t:t + 1], stream=stream)

    def run_applies(which):
        for c, (t, i) in enumerate(calls):
            if which is None or bool(flags_np[i][t]) == which:
                gsi.apply(reps[t % R][i], Xs[i][t:t + 1], G_all[c:c + 1], wsl(c), Y=Yk[i][t:t + 1],
                          stream=stream)

    def timed_graph(fn, reps_n):
        with torch.cuda.stream(stream):
            fn()  # eager once (sets kernel attributes outside capture)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(reps_n):
                g.replay()
            a1.record(stream)
        stream.synchronize()
        return a0.elapsed_time(a1) / reps_n

    if args.kernel_traffic:
        with torch.cuda.stream(stream):
            run_gates()
            run_applies(None)
        stream.synchronize()
        # the eager step's decode_kernel launches in launch order (token t,
        # then the four maps): their algorithmic bytes, to set beside an ncu
        # capture of a few of them
        fl = [F.cpu().numpy().astype(bool) for F in Fs]
        per_launch = [call_bytes(m.d, m.d_out, m.k, 1, int(not f[t]), int(f[t]))
                      for t in range(T_TOKENS) for m, f in zip(base, fl)]
        print(json.dumps({"kernel_traffic": "decode_kernel launches of the eager step",
                          "algorithmic_bytes_per_launch": per_launch,
                          "mean_algorithmic_bytes_per_launch": sum(per_launch) / len(per_launch)}))
        return
    t_gate = timed_graph(run_gates, args.steps)
    t_fast = timed_graph(lambda: run_applies(False), args.steps)
    t_slow = timed_graph(lambda: run_applies(True), args.steps)
    t_apply = timed_graph(lambda: run_applies(None), args.steps)
    for i in range(4):
        # the step ran the single-launch decode; the split calls run the
        # two-launch kernels, which add the same products in another order
        assert torch.equal(Fk[i], Fs[i]), "two-launch path's flags disagree with the step's"
        rel = float((Yk[i] - Ys[i]).norm() / Ys[i].norm())
        assert rel < 1e-4, f"two-launch path disagrees with the step's outputs (rel L2 {rel:.2e})"
    k_gate = ab["gate"] / (t_gate * 1e-3) / 1e9
    k_fast = ab["fast"] / (t_fast * 1e-3) / 1e9 if t_fast else None
    k_slow = ab["slow"] / (t_slow * 1e-3) / 1e9 if t_slow else None
    k_apply = (ab["fast"] + ab["slow"]) / (t_apply * 1e-3) / 1e9
    # The dominant kernel is decode_kernel, the step's only kernel: each
    # launch moves one call's algorithmic bytes, and its mean launch interval
    # over the timed replays (launch gaps included, so the achieved figure is
    # a lower bound) is ms / 1024.  On the two-launch path the dominant kernel
    # is decide_apply_kernel, whose stored-decision launches (gsi_apply) are
    # timed in a graph of their own.
    if sum(per_call) == 4:
        # the step's only kernel: one single-token decode launch per
        # gated-map call (gsi_stack runs the four maps one call each)
        dom = dict(name="decode_kernel (single-token decode: projection, gate, M g / W x in one launch)",
                   gbs=step_gbs, bytes_per_launch=ab["total"] / n_launch, ms=ms / n_launch,
                   timing="CUDA events over the timed region (graph replays of the step); "
                          "per-launch time = mean launch interval, gaps included")
    else:
        dom = dict(name="decide_apply_kernel (stored decision: y = M g fast, y = W x slow)", gbs=k_apply,
                   bytes_per_launch=(ab["fast"] + ab["slow"]) / n_launch, ms=t_apply / n_launch,
                   timing="CUDA events around a graph of this kernel's 1024 launches of one step")

    # ---- end to end: pinned host tokens in, outputs and flags out, every step
    Xh = [X.cpu().pin_memory() for X in Xs]
    Yh = [torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True) for Y in Ys]
    Fh = [torch.empty(F.shape, dtype=F.dtype, pin_memory=True) for F in Fs]
    h2d = sum(x.numel() * x.element_size() for x in Xh)
    d2h = sum(y.numel() * y.element_size() for y in Yh) + sum(f.numel() for f in Fh)

    def e2e_step():
        with torch.cuda.stream(stream):
            for xd, xh in zip(Xs, Xh):
                xd.copy_(xh, non_blocking=True)
            graph.replay()
            for yd, yh in zip(Ys, Yh):
                yh.copy_(yd, non_blocking=True)
            for fd, fh in zip(Fs, Fh):
                fh.copy_(fd, non_blocking=True)

    for _ in range(2):
        e2e_step()
    stream.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_tps = T_TOKENS * world / (e2e_ms / 1e3)

    # ---- oracle on the host cores (bounded sample of the same workload)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        maps64 = oracle_maps(maps_in, [b.M.cpu() for b in base])
        v, dt, passes = time_oracle(maps64, EPS, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"{passes} passes of the 256 decode tokens through all four maps "
                         f"({dt:.1f} s of float64 numpy; BLAS threads = host cores)"}

    if cpu is not None:
        # the same sample on one host thread (a fresh process whose BLAS
        # threads are set to one before numpy loads)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe", "--cpu-seconds",
                            str(args.cpu_seconds)], capture_output=True, text=True, env=env)
        try:
            one = json.loads(r.stdout.strip().splitlines()[-1])
            cpu["value_1_thread"] = one["value"]
            cpu["sample_1_thread"] = f"{one['passes']} passes ({one['seconds']:.1f} s) on one thread"
        except (ValueError, IndexError, KeyError):
            cpu["value_1_thread"] = None

    # ---- the gate's Gram form checked on the device against the explicit
    # residual x - V g (second pass over V) for the step's 1024 calls
    torch.cuda.synchronize()
    rho_dev = []
    for i, b in enumerate(base):
        G_i = G_all[i::4].contiguous()
        r_i = rho_all[i::4].contiguous()
        _, dv = gsi.residual_check(b, Xs[i], G_i, r_i)  # on the stream that made G_i and r_i
        rho_dev.append(dv)
    torch.cuda.synchronize()
    gate_check = {"max_abs_rho2_gram_minus_explicit": max(float(v.item()) for v in rho_dev),
                  "what": "largest |rho^2 (Gram form, gate kernels) - rho^2 (explicit x - V g, second pass)| "
                          "over the 1024 single-token calls of the step (gsi_residual_check)"}

    # the same step with the persistent stack kernel (one launch per decode
    # step over the four maps, grid barrier between maps), for comparison
    def step_persistent():
        for t in range(T_TOKENS):
            gsi.stack_raw(args_t[t], 4, 1, EPS, ws, stream=stream, mode="persistent")

    ms_pers = graph_time_ms(step_persistent, stream, args.steps)
    assert gsi.workspace_status(ws, stream=stream) == 0
    persistent = {"kernel": "stack_decode_kernel (one persistent launch per decode step over the four maps)",
                  "tokens_per_s": T_TOKENS * world / (ms_pers * 1e-3), "ms_per_step": ms_pers,
                  "achieved_gbs": ab["total"] / (ms_pers * 1e-3) / 1e9,
                  "frac_of_hbm_peak": ab["total"] / (ms_pers * 1e-3) / 1e9 / hbm_peak,
                  "us_per_map_call": ms_pers * 1e3 / n_launch}

    secondary = None
    if not args.no_secondary and world == 1:
        tf_peak, _ = bf16_peak()
        secondary = {"note": "further synthetic workloads, each timed on its own after the headline step"}
        for key, fn in (("cfg3_28_layer_stack", lambda: run_config3(gsi, dev, stream, hbm_peak)),
                        ("cfg4_13b_small_batch", lambda: run_config4(gsi, dev, stream, hbm_peak)),
                        ("cfg5_prefill", lambda: run_config5(gsi, dev, stream, hbm_peak, tf_peak))):
            try:
                secondary[key] = fn()
            except Exception as e:  # report and go on: the headline line still prints
                secondary[key] = {"error": f"{type(e).__name__}: {e}"}

    gpu_launches = args.steps * T_TOKENS * sum(per_call)
    line = {
        "metric": "gsi_linear_tokens_per_s_batch1",
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "6B-class decoder layer linears at batch 1: qkv 12288x4096, out 4096x4096, "
                        "up 16384x4096, down 4096x16384; bf16 W/V/M/x, fp32 accumulate and y; "
                        f"k={K_RANK}, eps={EPS}; 256 sequential single-token steps x 4 maps "
                        "(1024 gated-map calls) per step; 26/256 slow tokens per map",
            "l2": f"inputs larger than L2: weights rotate over {R} device replicas of the layer "
                  f"({R * sum(map_bytes(m)['V'] + map_bytes(m)['M'] + map_bytes(m)['gram'] for m in maps_in) / 1e6:.0f} MB "
                  "of fast-path weights, 129 MB L2)",
            "parallelism": "replicas only" if world > 1 else "single GPU",
            "graph": "whole step captured in one CUDA graph, programmatic dependent launch between kernels",
            "path": "single-token decode kernel, one launch per call (cluster projection for qkv, out and "
                    "up, grid projection for down)"
                    if sum(per_call) == 4 else "two-launch streaming kernels",
        },
        "achieved_step_gbs": step_gbs,
        "step_frac_of_hbm_peak": step_gbs / hbm_peak,
        "bytes_per_step": ab["total"],
        "dense_bytes_per_step": ab["dense"],
        "bytes_saved_vs_dense": ab["dense"] / ab["total"],
        "slow_fraction": ab["n_slow"] / (ab["n_slow"] + ab["n_fast"]),
        "kernels_gbs": {
            "gate (project_kernel + decide_apply_kernel decision-only, gsi_gate)": k_gate,
            "apply fast calls (decide_apply_kernel, gsi_apply)": k_fast,
            "apply slow calls (decide_apply_kernel, gsi_apply)": k_slow,
            "apply all calls": k_apply,
            "gate_ms_per_step": t_gate, "apply_fast_ms_per_step": t_fast,
            "apply_slow_ms_per_step": t_slow, "apply_ms_per_step": t_apply,
        },
        "roofline": {
            "kernel": dom["name"], "bound": "hbm", "achieved": dom["gbs"], "peak": hbm_peak,
            "unit": "GB/s", "frac": dom["gbs"] / hbm_peak, "traffic": kernel_traffic(),
            "peak_kind": peak_kind,
            "timing": dom["timing"],
            "bytes_per_launch": dom["bytes_per_launch"], "ms_per_launch": dom["ms"],
        },
        "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "gate_check": gate_check,
        "persistent_stack_same_step": persistent,
        "secondary": secondary,
    }
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
