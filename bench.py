"""Benchmark of the int4-gs64 MoE decode hot path on GB300.

Default workload (one step): the MoE decode micro-batch of 8 tokens, hidden
6144, 160 experts, expert intermediate 2048, top-8, router logits N(0,1) with
+2 on 16 seeded "hot" experts: routing and the expert FFN in one call
(moe_route_expert_ffn_int4: the grouping kernel routes and groups the
tokens, then fused gate+up+SiLU, down, weighted combine).
The metric is achieved HBM bandwidth over the algorithmic bytes of a step
(packed weights + scales of the experts the batch touches, plus activations
in and out). Inputs are synthetic and seeded (datagen); a step rotates over
8 seeded micro-batches, and every step reads ~0.6 GB of expert weights, far
more than the 129 MB L2, so no step is served from L2.

Also measured and reported under "rows" (not part of the step): the dense
int4-gs64 and int8-row GEMV 14336 x 4096 (16 / 8 rotating weight copies) and
the 1-token MoE layer H 2048 / E 256 / I 512 (8 rotating routings).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs N independent replicas under torchrun (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "int4-gs64 MoE expert GEMV HBM GB/s and % of 8 TB/s; µs/decode-token layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
EXPERT_BYTES = lambda H, I: 3 * H * I // 2 + 3 * H * I // 64 * 4  # noqa: E731
W3 = dict(H=6144, E=160, I=2048, k=8, T=8, hot=16)
W2 = dict(H=2048, E=256, I=512, k=8, T=1, hot=0)
ROTATE = 8


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ workload

def w3_batches(wl, n):
    """n seeded micro-batches: x, logits, and the oracle-independent union size."""
    import datagen
    out = []
    for b in range(n):
        x, logits = datagen.moe_inputs(wl["T"], wl["E"], wl["H"], hot=wl["hot"],
                                       token_start=b * wl["T"])
        top = np.argsort(-logits, axis=1, kind="stable")[:, : wl["k"]]
        out.append(dict(x=x, logits=logits, U=len(np.unique(top))))
    return out


def step_bytes(wl, U):
    act = wl["T"] * wl["H"] * 4 * 2 + wl["T"] * wl["E"] * 4 + wl["T"] * wl["k"] * 8
    return U * EXPERT_BYTES(wl["H"], wl["I"]) + act


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"qmv_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU baseline (oracle)

def cpu_baseline(wl, batch, budget_s: float = 15.0):
    """The fp64 oracle, as it stands, on the host cores: routing of the whole
    batch, then the FFN of as many tokens as fit in ~budget_s, scaled to the
    whole micro-batch."""
    import datagen
    import oracle
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    x, logits = batch["x"], batch["logits"]
    t0 = time.perf_counter()
    ids, w = oracle.route_topk(logits, wl["k"])
    t_route = time.perf_counter() - t0
    n_tok, t_ffn = 0, 0.0
    while n_tok < wl["T"] and (n_tok == 0 or t_ffn * (n_tok + 1) / n_tok < budget_s):
        t = n_tok
        touched = np.unique(ids[t])
        sub = datagen.moe_weights(wl["E"], wl["H"], wl["I"], experts=touched)
        pos = {int(e): i for i, e in enumerate(touched)}
        mids = np.array([[pos[int(e)] for e in ids[t]]], np.int32)
        t1 = time.perf_counter()
        oracle.moe_ffn(sub, x[t:t + 1].astype(np.float64), mids, w[t:t + 1].astype(np.float32))
        t_ffn += time.perf_counter() - t1
        n_tok += 1
    t_step = t_route + t_ffn * wl["T"] / n_tok
    return dict(t_step=t_step, cores=oracle.get_threads(),
                sample=f"routing of all {wl['T']} tokens + expert FFN of {n_tok} of {wl['T']} "
                       f"tokens (8 experts each), scaled to the micro-batch")


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import datagen  # noqa: F401
    import oracle  # noqa: F401
    wl = W3
    batches = w3_batches(wl, 1)
    per = []
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state: untimed warm-up steps are skipped
    for s in range(args.steps):
        r = cpu_baseline(wl, batches[0], budget_s=max(2.0, 60.0 / max(args.steps, 1)))
        per.append(r)
    t = statistics.mean(r["t_step"] for r in per)
    B = step_bytes(wl, batches[0]["U"])
    value = B / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded datagen)",
        "config": bench_config(1, wl["T"]),
        "timing": "host wall clock of the fp64 oracle on the host cores (no GPU)",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": per[0]["cores"],
                         "kind": "oracle", "sample": per[0]["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU timing helpers

def graph_of(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm (also binds lazily-loaded state before capture)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def time_graphs(graphs, iters, stream):
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record(stream)
        for i in range(iters):
            graphs[i % len(graphs)].replay()
        e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) * 1e-3 / iters


def time_graphs_steps(graphs, iters, stream):
    """Like time_graphs, with an event after every replay: (mean seconds per
    replay over the whole region, per-replay seconds)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(iters):
            graphs[i % len(graphs)].replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) * 1e-3 for i in range(iters)]
    return ev[0].elapsed_time(ev[-1]) * 1e-3 / iters, per


def spread(xs, scale=1.0):
    """min / p10 / median / p90 / max of a list, times scale."""
    v = sorted(x * scale for x in xs)
    pick = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]  # noqa: E731
    return {"min": v[0], "p10": pick(0.1), "median": pick(0.5), "p90": pick(0.9), "max": v[-1]}


def bench_config(ws_n: int, T: int) -> dict:
    """The workload, as both arms print it."""
    return {"workload": "MoE decode H6144 E160 I2048 top8, 8 tokens, 16 hot experts",
            "global_batch": T * ws_n, "seq_len": 1, "parallelism": f"replicas x{ws_n}",
            "l2": "inputs larger than L2 (~0.6 GB of expert weights per step vs 129 MB L2); "
                  "8 rotating seeded micro-batches"}


def load_traffic(kernel: str, alg_bytes: float):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the
    source (the kernel's file and the headers holding its device code and sizes,
    hashed): the captured launch's dram read + write bytes, scaled to a launch of
    `alg_bytes` algorithmic bytes by the ratio of algorithmic bytes (the capture runs
    a smaller expert pool; traffic grows with the experts touched)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel]
    except Exception:
        return None
    h = hashlib.sha256()
    try:
        for f in sorted(d.get("sources", [])):
            h.update(open(os.path.join(ROOT, f), "rb").read())
    except OSError:
        return None  # a source it was measured on is gone: stale
    if h.hexdigest() != d.get("sha256"):
        return None
    return d["measured_bytes"] * alg_bytes / d["measured_algorithmic_bytes"]


# ------------------------------------------------------------------ profiling case

def run_profile_case(args):
    """Small case for ncu captures: the 8-token layer shape (H 6144, I 2048,
    top-8, 8 tokens) over a pool of only `--profile-experts` experts, run for
    `--steps` steps without timing. Inputs stay larger than L2 (about 21
    experts, 0.45 GB, are touched per step with 40 experts)."""
    import torch
    import datagen
    import int4_group_quantized_gs64_gb300 as q
    q.build()
    dev = torch.device("cuda")
    E, H, I, T, k = args.profile_experts, W3["H"], W3["I"], W3["T"], W3["k"]
    m = q.MoeInt4Weights.from_numpy(datagen.moe_weights(E, H, I), dev)
    x, logits = datagen.moe_inputs(T, E, H, hot=min(W3["hot"], E // 2))
    xd, ld = torch.from_numpy(x).to(dev), torch.from_numpy(logits).to(dev)
    ws = torch.empty(q.moe_workspace_bytes(m, T, k), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    for _ in range(args.steps):
        ids, w = q.moe_route_topk(ld, k)
        q.moe_expert_ffn_int4(m, xd, ids, w, out=out, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": f"MoE decode H{H} I{I} top{k}, {T} tokens, {E}-expert pool",
                      "experts_touched": int(len(np.unique(ids.cpu().numpy()))),
                      "steps": args.steps, "launches_per_step": 5}))
    return 0


def run_profile_dense(args):
    """ncu case for the dense GEMV: int4-gs64 14336 x 4096, one token, over 4
    rotating weight copies (132 MB, above L2), `--steps` launches each, no timing."""
    import torch
    import datagen
    import int4_group_quantized_gs64_gb300 as q
    q.build()
    dev = torch.device("cuda")
    N, K = 14336, 4096
    wq, sc, x = datagen.dense_int4(N, K, 1)
    ws_ = [torch.from_numpy(wq).to(dev) for _ in range(4)]
    ss_ = [torch.from_numpy(sc).to(dev) for _ in range(4)]
    xd = torch.from_numpy(x).to(dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    ws = torch.empty(q.qmv_gemv_workspace_bytes(K, 1), dtype=torch.uint8, device=dev)
    for i in range(args.steps * 4):
        q.qmv_int4_gs(ws_[i % 4], ss_[i % 4], xd, y=y, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": f"int4-gs64 GEMV {N}x{K}, 1 token, 4 weight copies",
                      "launches": args.steps * 4, "kernels_per_launch": 1}))
    return 0


def run_profile_int3(args):
    """ncu case for the int3-g64 GEMV: 14336 x 4096, one token, over 8 rotating
    weight and scale copies (206 MB, above L2), `--steps` launches each, no timing."""
    import torch
    import int4_group_quantized_gs64_gb300 as q
    q.build()
    dev = torch.device("cuda")
    N, K, C = 14336, 4096, 8
    rng = np.random.default_rng(3)
    w3 = [torch.from_numpy(rng.integers(0, 256, size=(N, K // 64 * 24), dtype=np.uint8)).to(dev)
          for _ in range(C)]
    s3 = [torch.from_numpy((np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4)
                           .astype(np.float32)).to(dev) for _ in range(C)]
    xd = torch.from_numpy(rng.normal(size=(1, K)).astype(np.float32)).to(dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    for i in range(args.steps * C):
        q.qmv_int3_gs(w3[i % C], s3[i % C], xd, y=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": f"int3-g64 GEMV {N}x{K}, 1 token, {C} weight copies",
                      "launches": args.steps * C, "kernels_per_launch": 1}))
    return 0


def run_profile_one(args):
    """ncu case for the one-token layer (H 2048, E 256, I 512, top-8; k_moe_one):
    8 seeded tokens in turn, `--steps` rounds, routing in-kernel, no timing."""
    import torch
    import datagen
    import int4_group_quantized_gs64_gb300 as q
    q.build()
    dev = torch.device("cuda")
    wl = W2
    m = q.MoeInt4Weights.from_numpy(datagen.moe_weights(wl["E"], wl["H"], wl["I"]), dev)
    bs = w3_batches(wl, 8)
    xs = [torch.from_numpy(b["x"]).to(dev) for b in bs]
    ls = [torch.from_numpy(b["logits"]).to(dev) for b in bs]
    ws = torch.empty(q.moe_workspace_bytes(m, 1, 8), dtype=torch.uint8, device=dev)
    out = torch.empty((1, wl["H"]), dtype=torch.float32, device=dev)
    for i in range(args.steps * len(bs)):
        q.moe_route_expert_ffn_int4(m, ls[i % len(bs)], xs[i % len(bs)], 8, out=out, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": "one-token MoE layer H2048 E256 I512 top8",
                      "calls": args.steps * len(bs), "one_kernel": q.moe_one_token_path(m, 8) == 1}))
    return 0


def run_profile_prefill(args):
    """ncu case for the prefill kernels: 512 tokens (H 6144, I 2048, top-8) over
    a pool of `--profile-prefill` experts, `--steps` calls, no timing."""
    import torch
    import datagen
    import int4_group_quantized_gs64_gb300 as q
    q.build()
    dev = torch.device("cuda")
    E, H, I, T, k = args.profile_prefill, W3["H"], W3["I"], 512, 8
    m = q.MoeInt4Weights.from_numpy(datagen.moe_weights(E, H, I), dev)
    xb, lg = datagen.moe_inputs(T, E, H, xdtype="bf16")
    xbd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    ids, w = q.moe_route_topk(torch.from_numpy(lg).to(dev), k)
    ws = torch.empty(q.moe_prefill_workspace_bytes(m, T, k), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    for _ in range(args.steps):
        q.moe_expert_ffn_int4_prefill(m, xbd, ids, w, out=out, ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": f"MoE prefill H{H} I{I} top{k}, {T} tokens, {E}-expert pool",
                      "steps": args.steps, "launches_per_step": 5}))
    return 0


# ------------------------------------------------------------------ ranks

def max_over_ranks(t_step: float, device=None) -> float:
    """The slowest rank's step time (every rank gets it); t_step itself on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t_step
    tt = torch.tensor([t_step], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_value(world_size: int, bytes_per_step: float, t_step: float) -> float:
    """Replicas each run the full step on their own micro-batches: the job moves
    world_size x bytes_per_step in the slowest rank's step time (GB/s)."""
    return world_size * bytes_per_step / t_step / 1e9


# ------------------------------------------------------------------ ours

def run_ours(args):
    import torch
    import datagen
    import int4_group_quantized_gs64_gb300 as q

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.build()
    q.lib()
    stream = torch.cuda.Stream(device=dev)
    wl = W3

    # ---- workload: all 160 experts resident (3.4 GB), 8 rotating micro-batches
    wts = datagen.moe_weights(wl["E"], wl["H"], wl["I"])
    m = q.MoeInt4Weights.from_numpy(wts, dev)
    del wts
    batches = w3_batches(wl, ROTATE)
    T, k = wl["T"], wl["k"]
    xs = [torch.from_numpy(b["x"]).to(dev) for b in batches]
    ls = [torch.from_numpy(b["logits"]).to(dev) for b in batches]
    ids = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in batches]
    wv = [torch.empty((T, k), dtype=torch.float32, device=dev) for _ in batches]
    outs = [torch.empty((T, wl["H"]), dtype=torch.float32, device=dev) for _ in batches]
    wsb = q.moe_workspace_bytes(m, T, k)
    wss = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in batches]
    B_mean = statistics.mean(step_bytes(wl, b["U"]) for b in batches)
    U_mean = statistics.mean(b["U"] for b in batches)

    def step(i):  # routing + expert FFN through the one-call entry point
        def f():
            q.moe_route_expert_ffn_int4(m, ls[i], xs[i], k, ids=ids[i], w=wv[i], out=outs[i],
                                        ws=wss[i], stream=stream)
        return f

    graphs = [graph_of(step(i), stream) for i in range(ROTATE)]
    launches_per_step = 4  # route+group+split, gate+up, down, combine

    # ---- warm-up, then a short untimed soak so the clock sampler sees the load
    clocks = ClockSampler(local)
    time_graphs(graphs, max(args.warmup, 3), stream)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.5:
        time_graphs(graphs, 64, stream)

    # ---- timed region: K steps, barrier + synchronize on both sides
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_step, step_times = time_graphs_steps(graphs, args.steps, stream)
    torch.cuda.synchronize()
    if ws_n > 1:
        t_step = max_over_ranks(t_step, dev)
        dist.barrier()
    clk = clocks.stop()

    # ---- the two FFN kernels alone (gate+up, the dominant one, and down), CUDA
    # events on the launching stream, over the 8 rotating micro-batches
    for i in range(ROTATE):
        with torch.cuda.stream(stream):
            q.moe_route_topk(ls[i], k, ids=ids[i], w=wv[i], stream=stream)
            q.moe_ffn_prepare(m, xs[i], ids[i], wss[i], stream=stream)
    gu_t, dn_t, gu_b, dn_b = [], [], [], []
    E_gu = 2 * wl["I"] * wl["H"] // 2 + 2 * wl["I"] * wl["H"] // 64 * 4
    E_dn = wl["H"] * wl["I"] // 2 + wl["H"] * wl["I"] // 64 * 4
    # every launch enqueued back to back and one synchronize at the end, so
    # the events measure the kernels, not the host's launch latency
    evs = []
    for rep in range(4):
        for i in range(ROTATE):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            with torch.cuda.stream(stream):
                ev[0].record(stream)
                q.moe_ffn_gate_up(m, T, k, wss[i], stream=stream)
                ev[1].record(stream)
                q.moe_ffn_down(m, T, k, wss[i], stream=stream)
                ev[2].record(stream)
            evs.append((rep, i, ev))
    torch.cuda.synchronize()
    for rep, i, ev in evs:
        if rep >= 1:
            gu_t.append(ev[0].elapsed_time(ev[1]) * 1e-3)
            dn_t.append(ev[1].elapsed_time(ev[2]) * 1e-3)
            U = batches[i]["U"]
            gu_b.append(U * E_gu + T * wl["H"] * 4 + T * k * wl["I"] * 4)
            dn_b.append(U * E_dn + T * k * wl["I"] * 4 + T * k * wl["H"] * 4)
    peak, peak_kind = peaks()
    gu_kernel = "k_moe_tma" if q.moe_weight_path(m) == 1 else "k_gate_up"
    gu_ach = sum(gu_b) / sum(gu_t) / 1e9
    dn_ach = sum(dn_b) / sum(dn_t) / 1e9
    roofline = {"bound": "hbm", "kernel": gu_kernel, "achieved": gu_ach,
                "peak": peak, "unit": "GB/s", "frac": gu_ach / peak,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "traffic": load_traffic(gu_kernel + " gate+up", statistics.mean(gu_b)),
                "bytes_per_launch": statistics.mean(gu_b),
                "us_per_launch": statistics.mean(gu_t) * 1e6,
                "us_per_launch_spread": spread(gu_t, 1e6), "launches_timed": len(gu_t),
                "down": {"kernel": gu_kernel, "achieved": dn_ach, "frac": dn_ach / peak,
                         "traffic": load_traffic(gu_kernel + " down", statistics.mean(dn_b)),
                         "bytes_per_launch": statistics.mean(dn_b),
                         "us_per_launch": statistics.mean(dn_t) * 1e6,
                         "us_per_launch_spread": spread(dn_t, 1e6)}}

    # ---- end to end through the public API with pinned host buffers
    hx = [torch.from_numpy(b["x"]).pin_memory() for b in batches]
    hl = [torch.from_numpy(b["logits"]).pin_memory() for b in batches]
    ho = [torch.empty((T, wl["H"]), dtype=torch.float32).pin_memory() for _ in batches]
    h2d = hx[0].numel() * 4 + hl[0].numel() * 4
    d2h = ho[0].numel() * 4
    for i in range(3):
        with torch.cuda.stream(stream):
            xs[i].copy_(hx[i], non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(args.steps, 10)
    # Copies run on their own streams so that step s+1's inputs travel while
    # step s computes; buffer i (of ROTATE) is reused only after the compute
    # and the read-back that used it before have finished. Every step's H2D
    # and D2H copies lie inside the timed region.
    st_h, st_d = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_h = [torch.cuda.Event() for _ in range(ROTATE)]
    ev_c = [torch.cuda.Event() for _ in range(ROTATE)]
    ev_d = [torch.cuda.Event() for _ in range(ROTATE)]
    e0.record(stream)
    st_h.wait_event(e0)
    st_d.wait_event(e0)
    for s in range(n_e2e):
        i = s % ROTATE
        if s >= ROTATE:
            st_h.wait_event(ev_c[i])  # the compute that read xs[i], ls[i] is done
        with torch.cuda.stream(st_h):
            xs[i].copy_(hx[i], non_blocking=True)
            ls[i].copy_(hl[i], non_blocking=True)
            ev_h[i].record(st_h)
        stream.wait_event(ev_h[i])
        if s >= ROTATE:
            stream.wait_event(ev_d[i])  # the read-back of outs[i] is done
        with torch.cuda.stream(stream):
            q.moe_route_expert_ffn_int4(m, ls[i], xs[i], k, ids=ids[i], w=wv[i], out=outs[i],
                                        ws=wss[i], stream=stream)
            ev_c[i].record(stream)
        st_d.wait_event(ev_c[i])
        with torch.cuda.stream(st_d):
            ho[i].copy_(outs[i], non_blocking=True)
            ev_d[i].record(st_d)
    for i in range(ROTATE):
        stream.wait_event(ev_d[i])
    e1.record(stream)
    e1.synchronize()
    t_e2e = e0.elapsed_time(e1) * 1e-3 / n_e2e
    if ws_n > 1:
        t_e2e = max_over_ranks(t_e2e, dev)

    rows = measure_rows(q, datagen, dev, stream, peak, m) if rank == 0 and not args.quick else {}

    if rank != 0:
        return 0
    value = whole_job_value(ws_n, B_mean, t_step)
    cpu = None
    if ws_n == 1 and not args.no_cpu:
        cb = cpu_baseline(wl, batches[0])
        cpu = {"value": step_bytes(wl, batches[0]["U"]) / cb["t_step"] / 1e9, "unit": "GB/s",
               "cores": cb["cores"], "kind": "oracle", "sample": cb["sample"]}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16x2-split MMA, fp32 accumulate",
        "data": "synthetic (seeded datagen, no trained weights)",
        "config": bench_config(ws_n, T),
        "experts_touched_mean": U_mean, "bytes_per_step_mean": B_mean,
        "timing": "CUDA graph replay of K steps between CUDA events, an event after every step",
        "ms_per_step_spread": spread(step_times, 1e3),
        "pct_of_8TBs": value / ws_n / NOMINAL_HBM_GBS * 100,
        "us_per_layer": t_step * 1e6, "us_per_decode_token_layer": t_step * 1e6 / T,
        "token_eq_per_s": ws_n * T / t_step,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_value(ws_n, B_mean, t_e2e), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": t_e2e * 1e6},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "rows": rows,
    }
    print(json.dumps(line))
    if ws_n > 1:
        dist.destroy_process_group()
    return 0


def measure_rows(q, datagen, dev, stream, peak, pool):
    """Other rows of the hot path, each with its own roofline fraction."""
    import torch
    rows = {}
    # MoE prefill, 512 tokens on the tcgen05 path, same 160-expert pool
    wl4 = dict(H=6144, E=160, I=2048, k=8, T=512)
    xb, lg = datagen.moe_inputs(wl4["T"], wl4["E"], wl4["H"], xdtype="bf16")
    xbd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    lgd = torch.from_numpy(lg).to(dev)
    i4 = torch.empty((wl4["T"], 8), dtype=torch.int32, device=dev)
    w4 = torch.empty((wl4["T"], 8), dtype=torch.float32, device=dev)
    o4 = torch.empty((wl4["T"], wl4["H"]), dtype=torch.float32, device=dev)
    ws4 = torch.empty(q.moe_prefill_workspace_bytes(pool, wl4["T"], 8), dtype=torch.uint8,
                      device=dev)
    g4 = [graph_of(lambda: (q.moe_route_topk(lgd, 8, ids=i4, w=w4, stream=stream),
                            q.moe_expert_ffn_int4_prefill(pool, xbd, i4, w4, out=o4, ws=ws4,
                                                          stream=stream)), stream)]
    time_graphs(g4, 3, stream)
    t = time_graphs(g4, 10, stream)
    U4 = len(np.unique(np.argsort(-lg, axis=1, kind="stable")[:, :8]))
    B4 = U4 * EXPERT_BYTES(wl4["H"], wl4["I"]) + xb.nbytes + o4.numel() * 4
    F4 = 2 * wl4["T"] * 8 * 3 * wl4["H"] * wl4["I"]
    rows["moe_prefill_h6144_e160_i2048_512tok"] = {
        "us": t * 1e6, "GBs": B4 / t / 1e9, "frac": B4 / t / 1e9 / peak, "bytes": B4,
        "experts_touched": U4, "tflops": F4 / t / 1e12, "launches_per_call": 6,
        "path": "tcgen05 kind::f16 (bf16), A dequantized into TMEM"}
    del ws4, o4
    # dense int4-gs64 and int8-row GEMV, 14336 x 4096, one token
    N, K = 14336, 4096
    wq, sc, x = datagen.dense_int4(N, K, 1)
    C = 16
    wqs = [torch.from_numpy(wq).to(dev) for _ in range(C)]
    scs = [torch.from_numpy(sc).to(dev) for _ in range(C)]
    xd = torch.from_numpy(x).to(dev)
    y = torch.empty((1, N), device=dev)
    wsd = torch.empty(q.qmv_gemv_workspace_bytes(K, 1), dtype=torch.uint8, device=dev)
    # all C calls (rotating weight copies, 530 MB: above L2) in one graph, so
    # host-side graph launches do not leave the GPU idle between calls
    gs = [graph_of(lambda: [q.qmv_int4_gs(wqs[i], scs[i], xd, y=y, ws=wsd, stream=stream)
                            for i in range(C)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 32, stream) / C
    Bq = wq.nbytes + sc.nbytes + x.nbytes + N * 4
    rows["int4_gemv_14336x4096"] = {"us": t * 1e6, "GBs": Bq / t / 1e9, "frac": Bq / t / 1e9 / peak,
                                    "bytes": Bq, "launches_per_call": 1}
    # the same with the output rounded to bf16 (qmv_int4_gs_bf16)
    ybf = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
    gs = [graph_of(lambda: [q.qmv_int4_gs_bf16(wqs[i], scs[i], xd, y=ybf, ws=wsd, stream=stream)
                            for i in range(C)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 32, stream) / C
    Bqh = wq.nbytes + sc.nbytes + x.nbytes + N * 2
    rows["int4_gemv_14336x4096_bf16out"] = {"us": t * 1e6, "GBs": Bqh / t / 1e9,
                                            "frac": Bqh / t / 1e9 / peak, "bytes": Bqh,
                                            "launches_per_call": 1}
    del wqs, scs, gs
    w8, r8, x8 = datagen.dense_int8(N, K, 1)
    C8 = 8
    w8s = [torch.from_numpy(w8).to(dev) for _ in range(C8)]
    r8d = torch.from_numpy(r8).to(dev)
    gs = [graph_of(lambda: [q.qmv_int8_row(w8s[i], r8d, xd, y=y, ws=wsd, stream=stream)
                            for i in range(C8)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 64, stream) / C8
    B8 = w8.nbytes + r8.nbytes + x.nbytes + N * 4
    rows["int8_gemv_14336x4096"] = {"us": t * 1e6, "GBs": B8 / t / 1e9, "frac": B8 / t / 1e9 / peak,
                                    "bytes": B8, "launches_per_call": 1}
    gs = [graph_of(lambda: [q.qmv_int8_row_bf16(w8s[i], r8d, xd, y=ybf, ws=wsd, stream=stream)
                            for i in range(C8)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 64, stream) / C8
    B8h = w8.nbytes + r8.nbytes + x.nbytes + N * 2
    rows["int8_gemv_14336x4096_bf16out"] = {"us": t * 1e6, "GBs": B8h / t / 1e9,
                                            "frac": B8h / t / 1e9 / peak, "bytes": B8h,
                                            "launches_per_call": 1}
    del w8s, gs
    # int3-g64 two-plane GEMV, 14336 x 4096, one token (16 rotating copies, 410 MB)
    rng3 = np.random.default_rng(3)
    w3q = [torch.from_numpy(rng3.integers(0, 256, size=(N, K // 64 * 24), dtype=np.uint8)).to(dev)
           for _ in range(C)]
    s3 = [torch.from_numpy(sc).to(dev) for _ in range(C)]
    gs = [graph_of(lambda: [q.qmv_int3_gs(w3q[i], s3[i], xd, y=y, stream=stream)
                            for i in range(C)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 32, stream) / C
    B3q = N * K // 64 * 24 + sc.nbytes + x.nbytes + N * 4
    rows["int3_gemv_14336x4096"] = {"us": t * 1e6, "GBs": B3q / t / 1e9,
                                    "frac": B3q / t / 1e9 / peak, "bytes": B3q,
                                    "launches_per_call": 1,
                                    "path": "CUDA cores, warps walking rows, x staged in shared memory"}
    del w3q, s3, gs
    # small-S dense decode: 4 tokens against the 14336 x 4096 int4 matrix (weights read once)
    wqs = [torch.from_numpy(wq).to(dev) for _ in range(C)]
    x4 = torch.from_numpy(np.random.default_rng(11).normal(size=(4, K)).astype(np.float32)).to(dev)
    y4 = torch.empty((4, N), device=dev)
    ws4d = torch.empty(q.qmv_gemv_workspace_bytes(K, 4), dtype=torch.uint8, device=dev)
    scs = [torch.from_numpy(sc).to(dev) for _ in range(C)]
    gs = [graph_of(lambda: [q.qmv_int4_gs(wqs[i], scs[i], x4, y=y4, ws=ws4d, stream=stream)
                            for i in range(C)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 32, stream) / C
    Bq4 = wq.nbytes + sc.nbytes + x4.numel() * 4 + 4 * N * 4
    rows["int4_gemv_14336x4096_s4"] = {"us": t * 1e6, "GBs": Bq4 / t / 1e9,
                                       "frac": Bq4 / t / 1e9 / peak, "bytes": Bq4,
                                       "token_eq_per_s": 4 / t, "launches_per_call": 1}
    del wqs, scs, gs
    # pair of int4 GEMVs sharing x (q_a + kv_a shape 6144 -> (2048, 576)), one token;
    # 24 rotating weight copies (218 MB, above L2)
    K2, N0, N1, C2 = 6144, 2048, 576, 24
    pq = []
    for c in range(C2):
        rng = np.random.default_rng(100 + c)
        pm = []
        for N in (N0, N1):
            wq = rng.integers(0, 256, size=(N, K2 // 2), dtype=np.uint8)
            sc = (np.abs(rng.normal(0, 0.02, size=(N, K2 // 64))) + 1e-4).astype(np.float32)
            pm += [torch.from_numpy(wq).to(dev), torch.from_numpy(sc).to(dev)]
        pq.append(pm)
    xp = torch.from_numpy(np.random.default_rng(7).normal(size=(1, K2)).astype(np.float32)).to(dev)
    yp0 = torch.empty((1, N0), device=dev)
    yp1 = torch.empty((1, N1), device=dev)
    wsp = torch.empty(q.qmv_gemv_workspace_bytes(K2, 1), dtype=torch.uint8, device=dev)
    gs = [graph_of(lambda: [q.qmv_int4_gs_pair(*pq[i], xp, y0=yp0, y1=yp1, ws=wsp, stream=stream)
                            for i in range(C2)], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 32, stream) / C2
    gs = [graph_of(lambda: [(q.qmv_int4_gs(pq[i][0], pq[i][1], xp, y=yp0, ws=wsp, stream=stream),
                             q.qmv_int4_gs(pq[i][2], pq[i][3], xp, y=yp1, ws=wsp, stream=stream))
                            for i in range(C2)], stream)]
    time_graphs(gs, 4, stream)
    t2 = time_graphs(gs, 32, stream) / C2
    Bp = (N0 + N1) * (K2 // 2 + K2 // 64 * 4) + K2 * 4 + (N0 + N1) * 4
    rows["int4_gemv_pair_6144_2048_576"] = {"us": t * 1e6, "GBs": Bp / t / 1e9,
                                            "frac": Bp / t / 1e9 / peak, "bytes": Bp,
                                            "two_calls_us": t2 * 1e6, "launches_per_call": 1}
    del pq, gs
    # the 8-token layer with half of the 160 experts resident (served mask);
    # bytes: the served experts only
    wl = W3
    rmask = np.zeros(wl["E"], bool)
    rmask[np.random.default_rng(5).permutation(wl["E"])[: wl["E"] // 2]] = True
    words = np.zeros((wl["E"] + 31) // 32, np.uint32)
    for e in np.flatnonzero(rmask):
        words[e // 32] |= np.uint32(1) << np.uint32(e % 32)
    resd = torch.from_numpy(words.view(np.int32)).to(dev)
    bs3 = w3_batches(wl, ROTATE)
    T3, k3 = wl["T"], wl["k"]
    x3 = [torch.from_numpy(b["x"]).to(dev) for b in bs3]
    l3 = [torch.from_numpy(b["logits"]).to(dev) for b in bs3]
    i3 = [torch.empty((T3, k3), dtype=torch.int32, device=dev) for _ in bs3]
    w3 = [torch.empty((T3, k3), dtype=torch.float32, device=dev) for _ in bs3]
    o3 = [torch.empty((T3, wl["H"]), device=dev) for _ in bs3]
    sv3 = [torch.empty((T3, k3), dtype=torch.uint8, device=dev) for _ in bs3]
    ws3 = [torch.empty(q.moe_workspace_bytes(pool, T3, k3), dtype=torch.uint8, device=dev)
           for _ in bs3]

    def f3(i):
        return lambda: (q.moe_route_topk(l3[i], k3, ids=i3[i], w=w3[i], stream=stream),
                        q.moe_expert_ffn_int4_resident(pool, resd, x3[i], i3[i], w3[i], out=o3[i],
                                                       served=sv3[i], ws=ws3[i], stream=stream))
    gs = [graph_of(lambda: [f3(i)() for i in range(len(bs3))], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 16, stream) / len(bs3)
    U3 = []
    for b in bs3:
        top = np.argsort(-b["logits"], axis=1, kind="stable")[:, :k3]
        U3.append(int(rmask[np.unique(top)].sum()))
    B3 = statistics.mean(step_bytes(wl, u) for u in U3)
    rows["moe_decode_h6144_e160_i2048_8tok_resident_half"] = {
        "us": t * 1e6, "GBs": B3 / t / 1e9, "frac": B3 / t / 1e9 / peak, "bytes": B3,
        "served_experts_mean": statistics.mean(U3), "launches_per_call": 5}
    del ws3, gs
    # MoE decode, 1 token, H 2048 / E 256 / I 512 (pool 453 MB)
    wl = W2
    wts = datagen.moe_weights(wl["E"], wl["H"], wl["I"])
    m2 = q.MoeInt4Weights.from_numpy(wts, dev)
    del wts
    # 24 rotating micro-batches: ~140 distinct experts, ~250 MB, above L2
    bs = w3_batches(wl, 24)
    x2 = [torch.from_numpy(b["x"]).to(dev) for b in bs]
    l2 = [torch.from_numpy(b["logits"]).to(dev) for b in bs]
    i2 = [torch.empty((1, 8), dtype=torch.int32, device=dev) for _ in bs]
    w2 = [torch.empty((1, 8), dtype=torch.float32, device=dev) for _ in bs]
    o2 = [torch.empty((1, wl["H"]), device=dev) for _ in bs]
    ws2 = [torch.empty(q.moe_workspace_bytes(m2, 1, 8), dtype=torch.uint8, device=dev) for _ in bs]

    def f2(i):  # routing + FFN through the one-call entry point
        return lambda: q.moe_route_expert_ffn_int4(m2, l2[i], x2[i], 8, ids=i2[i], w=w2[i],
                                                   out=o2[i], ws=ws2[i], stream=stream)
    gs = [graph_of(lambda: [f2(i)() for i in range(len(bs))], stream)]
    time_graphs(gs, 4, stream)
    t = time_graphs(gs, 16, stream) / len(bs)
    B2 = statistics.mean(step_bytes(wl, b["U"]) for b in bs)
    one = q.moe_one_token_path(m2, 8) == 1
    rows["moe_decode_h2048_e256_i512_1tok"] = {
        "us": t * 1e6, "GBs": B2 / t / 1e9, "frac": B2 / t / 1e9 / peak, "bytes": B2,
        "launches_per_call": 1 if one else 5,
        "path": "one cooperative kernel routing the token and running the FFN (k_moe_one)"
                if one else "routing + grouped phases (k_moe_tma)"}
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the extra rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile-experts", type=int, default=0,
                    help="run the small ncu case with this many experts instead of the bench")
    ap.add_argument("--profile-dense", action="store_true",
                    help="run the small ncu case of the dense GEMV instead of the bench")
    ap.add_argument("--profile-one", action="store_true",
                    help="run the small ncu case of the one-token layer instead of the bench")
    ap.add_argument("--profile-int3", action="store_true",
                    help="run the small ncu case of the int3 GEMV instead of the bench")
    ap.add_argument("--profile-prefill", type=int, default=0,
                    help="run the small ncu case of the prefill with this many experts")
    args = ap.parse_args()
    if args.profile_prefill > 0:
        return run_profile_prefill(args)
    if args.profile_experts > 0:
        return run_profile_case(args)
    if args.profile_dense:
        return run_profile_dense(args)
    if args.profile_int3:
        return run_profile_int3(args)
    if args.profile_one:
        return run_profile_one(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
