"""Benchmark of one Medusa verify step (heads, tree packing, tree attention over
all layers, typical acceptance, KV compaction) on GB300.

Workload (default): the Vicuna-7B shape, bf16, batch 1, prefix 1024, 64-node
greedy sparse tree, T = 0.7, eps = 0.09, delta = 0.3; synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is verify steps/s of the whole job (N replicas,
one per GPU: the step does not shard, so N > 1 runs independent replicas).
The timed region holds exactly K steps, bracketed by a barrier and a device
synchronisation; per-step inputs (1.18 GB of head weights, 0.57 GB of KV cache)
are larger than L2, so no flush is needed between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "Medusa verify steps/s, accepted tok/s; tree-attn & head HBM GB/s vs peak (7B, 64 nodes)"
UNIT = "verify steps/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def workload_name(c):
    return (f"vicuna-7b-shape verify step: B={c['B']} H={c['H']} V={c['V']} K={c['K']} top-{c['topk']}, "
            f"{c['nl']} layers x {c['Hq']} heads x d{c['d']}, prefix {c['L']}, "
            f"{c['tree'][2]}-node greedy sparse tree, T={c['T']} eps={c['eps']} delta={c['delta']}")


def config_json(c, n_nodes):
    return {"workload": workload_name(c), "batch": c["B"], "hidden": c["H"], "vocab": c["V"], "heads": c["K"],
            "topk": c["topk"], "layers": c["nl"], "q_heads": c["Hq"], "kv_heads": c["Hkv"], "head_dim": c["d"],
            "prefix": c["L"], "tree_nodes": n_nodes, "temperature": c["T"], "eps": c["eps"], "delta": c["delta"],
            "l2": "inputs larger than L2 (1.18 GB head weights + 0.57 GB KV cache read per step), no flush",
            "parallelism": "replicas (one independent verify step per GPU)"}


def algorithmic_bytes(c, N):
    """Bytes each call must move at least once (reads + writes)."""
    B, H, V, K, topk = c["B"], c["H"], c["V"], c["K"], c["topk"]
    es = 2 if c["dtype"] == "bf16" else 4
    heads = K * (H * H + V * H) * es + B * H * es + B * K * topk * 8
    nl, Hq, Hkv, d, L = c["nl"], c["Hq"], c["Hkv"], c["d"], c["L"]
    attn = nl * B * (2 * L * Hkv * d + 2 * N * Hkv * d + 2 * N * Hq * d) * es + N * ((N + 31) // 32) * 4
    accept = B * N * V * 4 + B * N * 4
    # tree RoPE (outside the five-call step): q and tree K read and written once, positions read
    rope = 2 * nl * B * N * (Hq + Hkv) * d * es + B * N * 4
    return {"heads": heads, "attention": attn, "accept": accept, "rope": rope}


class ClockSampler:
    """nvidia-smi clock/throttle samples (200 ms) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def make_inputs(c, N, layers=None):
    inp = wl.step_inputs(c, N, layers=layers)
    return inp


def run_ours(args, c):
    import torch
    import torch.distributed as dist
    import medusa_head_speculative_heads_gb300 as mg
    from medusa_head_speculative_heads_gb300.build import build as build_lib
    from medusa_head_speculative_heads_gb300.step import VerifyStep

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build_lib()
    if world > 1:
        dist.barrier()
    mg.lib()

    topo = mg.Topology.greedy(np.array(wl.synthetic_accuracy(c["K"], c["tree"][1])), c["tree"][2])
    N = topo.n_nodes
    if args.profile:
        return run_profile(args, c, mg, topo, dev)
    tdev = lambda a: _to_dev(a, dev)  # noqa: E731
    inp = make_inputs(c, N)
    d = {k: tdev(inp[k]) for k in ("h", "w1", "w2", "root_tok", "prefix_len", "q", "kc", "vc", "kt", "vt", "logits")}
    vs = VerifyStep(B=c["B"], H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"], Hkv=c["Hkv"],
                    d=c["d"], Lmax=c["Lmax"], dtype=torch.bfloat16, topology=topo, temperature=c["T"],
                    eps=c["eps"], delta=c["delta"], device=dev)
    # Plant the synthetic backbone's agreement on this step's own tree tokens
    # (untimed set-up: the logits are an input of the step).
    vs.heads(d["h"], d["w1"], d["w2"])
    vs.tree(d["root_tok"], d["prefix_len"])
    torch.cuda.synchronize()
    tokens = vs.tokens.cpu().numpy()
    inp["logits"] = wl.plant(c, inp["logits"], tokens, topo.parent)
    d["logits"] = tdev(inp["logits"])
    stream = torch.cuda.current_stream(dev)

    def step():
        vs.run(d["h"], d["w1"], d["w2"], d["root_tok"], d["prefix_len"], d["q"], d["kc"], d["vc"], d["kt"],
               d["vt"], d["logits"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if vs.check() != 0:
        raise RuntimeError("device status set during warm-up")
    # The whole step as one CUDA graph (the five calls are stream-ordered with no
    # host synchronisation, so they capture as they are).
    graph = vs.capture(d["h"], d["w1"], d["w2"], d["root_tok"], d["prefix_len"], d["q"], d["kc"], d["vc"], d["kt"],
                       d["vt"], d["logits"])
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if vs.check() != 0:
        raise RuntimeError("device status set during graph warm-up")

    # ---- timed region: exactly K steps (graph replays), device events on the stream
    K = args.steps
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)

    # ---- per-call breakdown (separate eager pass, events between the calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for i in range(K):
        e = ev[i]
        e[0].record(stream)
        vs.heads(d["h"], d["w1"], d["w2"], stream)
        e[1].record(stream)
        vs.tree(d["root_tok"], d["prefix_len"], stream)
        e[2].record(stream)
        vs.attention(d["q"], d["kc"], d["vc"], d["kt"], d["vt"], d["prefix_len"], stream)
        e[3].record(stream)
        vs.accept(d["logits"], stream)
        e[4].record(stream)
        vs.compact(d["kc"], d["vc"], d["kt"], d["vt"], d["prefix_len"], stream)
        e[5].record(stream)
    torch.cuda.synchronize()
    names = ["heads", "tree_build", "attention", "accept", "compact"]
    per_call = {n: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) / K for j, n in enumerate(names)}
    accept_len = vs.accept_len.float().mean().item()
    assert vs.check() == 0
    # The tree RoPE that precedes attention in a verify pass (not part of the
    # five-call step): timed alone on copies of this workload's q and tree K.
    # Its 33.5 MB of bf16 q / K fit in L2, so every timed call follows an L2
    # flush (L2Flush) and a short GPU sleep (so the host's enqueue of the call
    # is not inside the events), and has its own events.
    rq, rk = d["q"].clone(), d["kt"].clone()
    flush = L2Flush(dev)
    for _ in range(3):
        mg.medusa_tree_rope(rq, rk, vs.pos, stream=stream)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush(i)
        torch.cuda._sleep(200000)  # ~0.1 ms of GPU time: the host enqueues the call before the start event fires
        rev[i][0].record(stream)
        mg.medusa_tree_rope(rq, rk, vs.pos, stream=stream)
        rev[i][1].record(stream)
    torch.cuda.synchronize()
    per_call["rope"] = sum(a.elapsed_time(b) for a, b in rev) / K
    del rq, rk, flush
    calib = time_calibration(mg, vs, c, N, K, stream, dev)
    linear = time_linear(mg, c, stream, dev, min(K, 50))
    linear_chain = time_linear_chain(mg, c, stream, dev)
    head_loss = time_head_loss(mg, stream, dev, min(K, 20))
    configs = None
    if args.configs != "none":
        configs = time_configs(mg, stream, dev, min(K, 20), None if args.configs == "all" else args.configs.split(","))

    ms_per_step = elapsed_ms / K
    value = job_steps_per_s(ms_per_step, world)
    hbm, tflops, peak_src = _peaks()
    ab = algorithmic_bytes(c, N)
    rooflines = {}
    for n in ("heads", "attention", "accept", "rope"):
        gbs = ab[n] / (per_call[n] * 1e-3) / 1e9
        rooflines[n] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbs / hbm, 4), "algorithmic_bytes": ab[n], "us": round(per_call[n] * 1e3, 2)}
    dominant = max(("heads", "attention"), key=lambda n: per_call[n])
    roof = dict(rooflines[dominant])
    roof["kernel"] = {"heads": "medusa_heads", "attention": "medusa_tree_attention"}[dominant]
    roof["peak_source"] = f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback 6.8 TB/s"
    roof["traffic"] = _traffic(roof["kernel"])

    e2e = run_e2e(args, c, vs, inp, d, dev, stream) if rank == 0 or world > 1 else None
    cpu = cpu_baseline(c, inp, topo) if (rank == 0 and world == 1 and not args.no_cpu) else None

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, model shapes)",
                "config": config_json(c, N),
                "accepted_tok_per_s": round(value * c["B"] * accept_len, 2), "mean_accept_len": accept_len,
                "per_call_us": {k: round(v * 1e3, 2) for k, v in per_call.items()},
                "roofline": roof, "rooflines": rooflines, "calibration": calib, "linear": linear, "linear_verify_pass": linear_chain,
                "head_loss": head_loss, "configs": configs, "e2e": e2e,
                "cpu_baseline": cpu,
                "gpu_launches": K * vs.launches_per_step(), "clocks": clocks}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_profile(args, c, mg, topo, dev):
    """Only the named call, `warmup` times and then `steps` times, on inputs
    drawn on the device (the per-layer tensors only when the call reads them),
    for profiler captures; prints no bench line.  Launches before the profiled
    calls: one heads call and one packing call (set-up), then `warmup` calls."""
    import torch
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    N = topo.n_nodes
    stream = torch.cuda.current_stream(dev)
    call = None
    if args.profile == "linear":  # the 8-layer verify pass (807 MB of weights) at 64 tree tokens
        lp = LinearPass(mg, c, dev)
        lp.tokens(64)
        call = lambda: lp.run(stream)  # noqa: E731
    elif args.profile == "head_loss":  # one sequence of 512 tokens: 262 MB of logits (above L2)
        lc, z, y = loss_inputs(dev, "f32", B=1, S=512)
        gz = torch.empty_like(z)
        call = lambda: mg.medusa_head_loss(z, y, lc["decay"], dlogits=gz, stream=stream)  # noqa: E731
    else:
        d = device_step_inputs(c, N, dev, layers=args.profile in ("attention", "rope"))
        vs = VerifyStep(B=c["B"], H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"],
                        Hkv=c["Hkv"], d=c["d"], Lmax=c["Lmax"], dtype=torch.bfloat16, topology=topo,
                        temperature=c["T"], eps=c["eps"], delta=c["delta"], device=dev)
        vs.heads(d["h"], d["w1"], d["w2"], stream)
        vs.tree(d["root_tok"], d["prefix_len"], stream)
        torch.cuda.synchronize()
        # The planting indexes the logits with the tree tokens on the device:
        # check them on the host first (an out-of-range index there is a
        # device-side assertion, not an exception).
        if vs.check() != 0 or not bool(((vs.tokens >= 0) & (vs.tokens < c["V"])).all()):
            raise RuntimeError("tree tokens outside the vocabulary")
        plant_on_device(c, d["logits"], vs.tokens, np.asarray(topo.parent))
        call = {"heads": lambda: vs.heads(d["h"], d["w1"], d["w2"], stream),
                "attention": lambda: vs.attention(d["q"], d["kc"], d["vc"], d["kt"], d["vt"], d["prefix_len"],
                                                  stream),
                "accept": lambda: vs.accept(d["logits"], stream),
                "rope": lambda: mg.medusa_tree_rope(d["q"], d["kt"], vs.pos, stream=stream)}[args.profile]
    for _ in range(args.warmup):
        call()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    if args.profile not in ("linear", "head_loss") and vs.check() != 0:
        raise RuntimeError("device status set")
    us = a.elapsed_time(b) / args.steps * 1e3
    line = {"profile": args.profile, "workload": f"{c['name']} B={c['B']} nodes={N} layers={c['nl']} heads={c['Hq']}/{c['Hkv']} prefix={c['L']}", "calls": args.steps,
            "us_per_call": round(us, 2)}
    if args.profile in ("heads", "attention"):
        hbm, tflops, _ = _peaks()
        nbytes = algorithmic_bytes(c, N)[args.profile]
        line["gbs"] = round(nbytes / us / 1e3, 1)
        line["hbm_frac"] = round(nbytes / us / 1e3 / hbm, 4)
    print(json.dumps(line))


def _capture(fn):
    """fn(s) (stream-ordered calls on stream s) captured into a CUDA graph on a
    side stream, after one eager run there outside capture; replay() launches
    it on the current stream."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_calibration(mg, vs, c, N, K, stream, dev):
    """Online tree calibration calls (outside the five-call step): this step's
    acceptance statistics, the accuracy-table update and a device rebuild of the
    greedy tree, each timed with CUDA events over K calls."""
    import torch
    R = c["topk"]
    Dmax = vs.path_nodes.shape[1] - 1
    tested = torch.zeros((Dmax, R), dtype=torch.int64, device=dev)
    accepted = torch.zeros_like(tested)
    acc = torch.tensor(wl.synthetic_accuracy(c["K"], c["tree"][1]), dtype=torch.float64, device=dev)
    calls = {
        "accept_stats": lambda s: mg.medusa_accept_stats(vs.path_nodes, vs.accept_len, vs.topo, R, tested, accepted,
                                                         stream=s),
        "acc_update": lambda s: mg.medusa_acc_update(acc[:Dmax], tested, accepted, 64.0, stream=s),
        "greedy_rebuild": lambda s: mg.medusa_topology_greedy_device(acc, N, stream=s),
    }
    out = {}
    for name, fn in calls.items():
        for _ in range(3):
            fn(stream)
        # K calls in one CUDA graph: the host's per-call cost (binding, launch)
        # stays out of the device time of these few-microsecond kernels.
        g = _capture(lambda s: [fn(s) for _ in range(K)])
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out[name + "_us"] = round(e0.elapsed_time(e1) / K * 1e3, 2)
        del g
    out["tree"] = f"{N} nodes from a {c['K']} x {c['tree'][1]} accuracy table"
    return out


class L2Flush:
    """Empties L2 before a timed call whose inputs would fit in it: a 256 MB
    write (the call's inputs leave L2), then a 256 MB read (the written lines
    are written back and replaced by clean ones), so the call starts with none
    of its inputs and none of another buffer's dirty lines in L2."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
        self.sink = None

    def __call__(self, i):
        self.w.fill_(i & 0xff)
        self.sink = self.r.max()


def time_linear(mg, c, stream, dev, reps):
    """The verify pass's linear layer (outside the five-call step) at the 7B
    hidden size, H x H weight, over 64 to 4096 tree tokens (B * N for B = 1 to
    64 at 64 nodes).  The weight fits in L2, so every call follows an L2 flush
    (L2Flush) and has its own events."""
    import torch
    H = c["H"]
    hbm, tflops, _ = _peaks()
    g = torch.Generator(device=dev).manual_seed(0)
    w = (torch.randn((H, H), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    flush = L2Flush(dev)
    out = {"weight": f"{H} x {H} bf16", "peak_tflops": tflops, "peak_gbs": hbm}
    for T in (64, 256, 1024, 4096):
        x = torch.randn((T, H), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = mg.lib().medusa_linear_workspace_size(T, H, H)
        wsb = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        for _ in range(3):
            mg.medusa_linear(x, w, y, ws=wsb, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            flush(i)
            torch.cuda._sleep(200000)  # the host's enqueue of the call is not timed
            ev[i][0].record(stream)
            mg.medusa_linear(x, w, y, ws=wsb, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        us = sum(a.elapsed_time(b) for a, b in ev) / reps * 1e3
        flops = 2.0 * T * H * H
        byts = 2.0 * (H * H + 2 * T * H)
        out[f"T{T}"] = {"us": round(us, 2), "tflops": round(flops / us / 1e6, 1),
                        "tensor_frac": round(flops / us / 1e6 / tflops, 4),
                        "gbs": round(byts / us / 1e3, 1), "hbm_frac": round(byts / us / 1e3 / hbm, 4)}
    del flush
    return out


class LinearPass:
    """The verify pass's linear layers of one Vicuna-7B-shape transformer layer
    (qkv 4096 -> 12288, o 4096 -> 4096, gate_up 4096 -> 22016, down 11008 -> 4096),
    two layers' worth of distinct weights (807 MB, above L2), run back to back as
    a verify pass runs them.  Weights are synthetic N(0, 0.02) bf16 drawn on the
    device from a seeded generator."""

    def __init__(self, mg, c, dev):
        import torch
        self.mg, self.dev = mg, dev
        H, I = c["H"], 11008
        self.shapes = [(H, 3 * H), (H, H), (H, 2 * I), (I, H)]
        self.g = torch.Generator(device=dev).manual_seed(1)
        self.layers = [(K, N, (torch.randn((N, K), generator=self.g, device=dev) * 0.02).to(torch.bfloat16))
                       for _ in range(2) for K, N in self.shapes]
        self.weight_bytes = sum(2 * K * N for K, N, _ in self.layers)

    def tokens(self, T):
        """Inputs, outputs and workspace for T tree tokens."""
        import torch
        self.T = T
        self.xs = {K: torch.randn((T, K), generator=self.g, device=self.dev).to(torch.bfloat16)
                   for K in {K for K, _ in self.shapes}}
        self.ys = {N: torch.empty((T, N), dtype=torch.bfloat16, device=self.dev) for _, N in self.shapes}
        self.ws = torch.empty(max(1, max(self.mg.lib().medusa_linear_workspace_size(T, K, N) for K, N in self.shapes)),
                              dtype=torch.uint8, device=self.dev)

    def run(self, s):
        for K, N, w in self.layers:
            self.mg.medusa_linear(self.xs[K], w, self.ys[N], ws=self.ws, stream=s)


def time_linear_chain(mg, c, stream, dev, reps=10):
    """LinearPass over the tree tokens of B = 1, 4 and 16 rows at 64 nodes."""
    import torch
    hbm, tflops, _ = _peaks()
    lp = LinearPass(mg, c, dev)
    wbytes = lp.weight_bytes
    out = {"layers": "qkv, o, gate_up, down x 2 (Vicuna-7B shapes)", "weight_bytes": wbytes}
    for B in (1, 4, 16):
        T = B * 64
        lp.tokens(T)
        for _ in range(3):
            lp.run(stream)
        # the 8 calls (up to 16 launches) as one CUDA graph, replayed back to
        # back: device time only, the host's per-call cost is not on the path
        gr = _capture(lp.run)
        for _ in range(3):
            gr.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / reps * 1e3
        flops = sum(2.0 * T * K * N for K, N, _ in lp.layers)
        out[f"T{T}"] = {"us_per_layer": round(us / len(lp.layers), 2), "weight_gbs": round(wbytes / us / 1e3, 1),
                        "hbm_frac": round(wbytes / us / 1e3 / hbm, 4), "tflops": round(flops / us / 1e6, 1),
                        "tensor_frac": round(flops / us / 1e6 / tflops, 4)}
        del gr
    del lp
    return out


def loss_inputs(dev, dtype="f32", **over):
    """The Medusa-1 training batch of the head loss (Vicuna-7B vocabulary, 4 heads,
    4 sequences of 2048 tokens unless overridden): logits ~ N(0, 2) drawn on the
    device from a seeded generator, target tokens from the seeded workload."""
    import torch
    lc = wl.loss_config("7b", **over)
    g = torch.Generator(device=dev).manual_seed(lc["cfg_id"])
    z = torch.randn((lc["K"], lc["B"], lc["S"], lc["V"]), generator=g, device=dev).mul_(2.0)
    if dtype == "bf16":
        z = z.to(torch.bfloat16)
    y = torch.from_numpy(wl.loss_tokens(lc)).to(dev)
    return lc, z, y


def time_head_loss(mg, stream, dev, reps):
    """Medusa-1 head loss + gradient over the whole training batch (outside the
    verify step): one read of the logits and one write of their gradient, both
    larger than L2, so no flush; fp32 and bf16 logits."""
    import torch
    hbm, _, _ = _peaks()
    out = {}
    for dt in ("f32", "bf16"):
        lc, z, y = loss_inputs(dev, dt)
        g = torch.empty_like(z)
        loss = torch.empty(lc["K"] + 1, dtype=torch.float32, device=dev)
        ws = torch.empty(mg.lib().medusa_head_loss_workspace_size(lc["K"], lc["B"], lc["S"]), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            mg.medusa_head_loss(z, y, lc["decay"], dlogits=g, loss=loss, ws=ws, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            torch.cuda._sleep(200000)  # the host's enqueue of the call is not timed
            ev[i][0].record(stream)
            mg.medusa_head_loss(z, y, lc["decay"], dlogits=g, loss=loss, ws=ws, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        us = sum(a.elapsed_time(b) for a, b in ev) / reps * 1e3
        byts = 2 * z.numel() * z.element_size() + y.numel() * 4
        out[dt] = {"us": round(us, 1), "algorithmic_bytes": byts, "gbs": round(byts / us / 1e3, 1),
                   "hbm_frac": round(byts / us / 1e3 / hbm, 4),
                   "loss": [round(float(v), 5) for v in loss.cpu()]}
        del z, g, y
    out["batch"] = f"{lc['K']} heads x {lc['B']} x {lc['S']} tokens x V {lc['V']}"
    out["peak_gbs"] = hbm
    return out


# The other workloads of the verify step, each timed as a whole step (the five
# calls in one CUDA graph): Vicuna-13B shape (batch 4, prefix 2048), the 7B-shape
# batch sweep (1 to 64 rows, prefix 1024, greedy acceptance) and the Vicuna-33B
# shape (prefix 4096) with the 64-node sparse and the 256-node dense tree.
CONFIG_RUNS = (("13b_b4", "13b", None, "tree"), ("sweep_b1", "sweep", 1, "tree"), ("sweep_b8", "sweep", 8, "tree"),
               ("sweep_b16", "sweep", 16, "tree"), ("sweep_b32", "sweep", 32, "tree"),
               ("sweep_b64", "sweep", 64, "tree"), ("33b_sparse64", "33b", None, "tree"),
               ("33b_dense256", "33b", None, "tree2"))


def lib_topology(mg, c, which="tree"):
    spec = c[which]
    if spec[0] == "dense":
        return mg.Topology.dense(list(spec[1]), spec[2])
    return mg.Topology.greedy(np.array(wl.synthetic_accuracy(c["K"], spec[1])), spec[2])


def device_step_inputs(c, N, dev, layers=True):
    """The workload's per-step inputs drawn on the device from a generator seeded
    with the configuration id (same distributions as the seeded host recipe:
    h, q, K, V ~ N(0, 1), weights ~ N(0, 0.02) in bf16, base logits ~ N(0, 2)
    in fp32, root tokens uniform); per-layer tensors are drawn layer by layer."""
    import torch
    g = torch.Generator(device=dev).manual_seed(1000 + c["cfg_id"])
    B, H, V, K, nl = c["B"], c["H"], c["V"], c["K"], c["nl"]
    bf = torch.bfloat16

    def normal(shape, std, out=None):
        x = torch.randn(shape, generator=g, device=dev)
        if std != 1.0:
            x.mul_(std)
        return x.to(bf) if out is None else out.copy_(x)

    d = {"h": normal((B, H), 1.0), "w1": torch.empty((K, H, H), dtype=bf, device=dev),
         "w2": torch.empty((K, V, H), dtype=bf, device=dev)}
    for k in range(K):
        normal((H, H), 0.02, d["w1"][k])
        normal((V, H), 0.02, d["w2"][k])
    shapes = {"q": (B, N, c["Hq"], c["d"]), "kc": (B, c["Lmax"], c["Hkv"], c["d"]),
              "vc": (B, c["Lmax"], c["Hkv"], c["d"]), "kt": (B, N, c["Hkv"], c["d"]), "vt": (B, N, c["Hkv"], c["d"])}
    for name, shp in (shapes.items() if layers else ()):
        d[name] = torch.empty((nl,) + shp, dtype=bf, device=dev)
        for l in range(nl):
            normal(shp, 1.0, d[name][l])
    d["logits"] = torch.randn((B, N, V), generator=g, device=dev).mul_(2.0)
    d["root_tok"] = torch.randint(0, V, (B,), generator=g, device=dev, dtype=torch.int32)
    d["prefix_len"] = torch.full((B,), c["L"], dtype=torch.int32, device=dev)
    return d


def plant_on_device(c, logits, tokens, parent):
    """The workload's planting (for every node with children, with probability
    p its first child's token gets the row maximum + 4), on device tensors; the
    per-node draws come from the same seeded generators as the host recipe."""
    import torch
    B, N, V = logits.shape
    first = np.full(N, -1)
    for n in range(N - 1, 0, -1):
        first[parent[n]] = n
    hit = np.zeros((B, N), bool)
    for b in range(B):
        u = wl.rng(c["cfg_id"], wl.T_PLANT, 0, b).random(N)
        hit[b] = (first >= 0) & (u < c["plant"])
    bi, ni = np.nonzero(hit)
    if len(bi) == 0:
        return
    bi_t = torch.from_numpy(bi).to(logits.device)
    ni_t = torch.from_numpy(ni).to(logits.device)
    ch_t = torch.from_numpy(first[ni]).to(logits.device)
    tok = tokens[bi_t, ch_t].long()
    if not bool(((tok >= 0) & (tok < V)).all()):
        raise RuntimeError("planting: tree tokens outside the vocabulary")
    rowmax = logits[bi_t, ni_t].amax(dim=1)
    logits[bi_t, ni_t, tok] = rowmax + 4.0


def config_algorithmic(c, N, mask_words):
    """Algorithmic bytes of heads and tree attention, and the attention's
    matrix-product flops over the visible keys (prefix + ancestors)."""
    ab = algorithmic_bytes(c, N)
    anc = sum(bin(int(w)).count("1") for w in np.asarray(mask_words, np.uint32).ravel())  # visible tree keys
    flops = 4.0 * c["nl"] * c["B"] * c["Hq"] * c["d"] * (N * c["L"] + anc)
    return ab["heads"], ab["attention"], flops


def time_configs(mg, stream, dev, steps, names=None):
    """Each workload of CONFIG_RUNS as a whole step: steps/s from graph replays
    (device events), mean accept length on planted logits, per-call times from
    an eager pass with events between the calls, and the heads / attention
    fractions of the measured peaks."""
    import torch
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    hbm, tflops, _ = _peaks()
    out = {}
    for key, name, B, which in CONFIG_RUNS:
        if names and key not in names:
            continue
        c = wl.config(name, **({} if B is None else {"B": B}))
        print(f"bench: workload {key}", file=sys.stderr, flush=True)
        topo = lib_topology(mg, c, which)
        N = topo.n_nodes
        d = device_step_inputs(c, N, dev)
        vs = VerifyStep(B=c["B"], H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"],
                        Hkv=c["Hkv"], d=c["d"], Lmax=c["Lmax"], dtype=torch.bfloat16, topology=topo,
                        temperature=c["T"], eps=c["eps"], delta=c["delta"], device=dev)
        vs.heads(d["h"], d["w1"], d["w2"], stream)
        vs.tree(d["root_tok"], d["prefix_len"], stream)
        torch.cuda.synchronize()
        if vs.check() != 0 or not bool(((vs.tokens >= 0) & (vs.tokens < c["V"])).all()):
            raise RuntimeError(f"{key}: tree tokens outside the vocabulary")
        plant_on_device(c, d["logits"], vs.tokens, np.asarray(topo.parent))
        args = (d["h"], d["w1"], d["w2"], d["root_tok"], d["prefix_len"], d["q"], d["kc"], d["vc"], d["kt"], d["vt"],
                d["logits"])
        graph = vs.capture(*args)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        if vs.check() != 0:
            raise RuntimeError(f"device status set in {key}")
        acc_len = vs.accept_len.float().mean().item()
        reps = max(3, min(steps, 10))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(reps)]
        for i in range(reps):
            e = ev[i]
            e[0].record(stream)
            vs.heads(d["h"], d["w1"], d["w2"], stream)
            e[1].record(stream)
            vs.tree(d["root_tok"], d["prefix_len"], stream)
            e[2].record(stream)
            vs.attention(d["q"], d["kc"], d["vc"], d["kt"], d["vt"], d["prefix_len"], stream)
            e[3].record(stream)
            vs.accept(d["logits"], stream)
            e[4].record(stream)
            vs.compact(d["kc"], d["vc"], d["kt"], d["vt"], d["prefix_len"], stream)
            e[5].record(stream)
        torch.cuda.synchronize()
        calls = ["heads", "tree_build", "attention", "accept", "compact"]
        us = {n: 1e3 * sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(reps)) / reps
              for j, n in enumerate(calls)}
        hb, atb, atf = config_algorithmic(c, N, vs.mask.cpu().numpy().view(np.uint32))
        heads_flops = 2.0 * c["B"] * c["K"] * (c["H"] * c["H"] + c["V"] * c["H"])
        out[key] = {
            "workload": f"{name} B={c['B']} H={c['H']} {c['nl']}x{c['Hq']}/{c['Hkv']}x{c['d']} prefix {c['L']} "
                        f"{N}-node {c[which][0]} tree T={c['T']}",
            "steps_per_s": round(1e3 / ms, 2), "ms_per_step": round(ms, 4),
            "accepted_tok_per_s": round(1e3 / ms * c["B"] * acc_len, 1), "mean_accept_len": round(acc_len, 3),
            "per_call_us": {k: round(v, 2) for k, v in us.items()},
            "heads": {"gbs": round(hb / us["heads"] / 1e3, 1), "hbm_frac": round(hb / us["heads"] / 1e3 / hbm, 4),
                      "tflops": round(heads_flops / us["heads"] / 1e6, 1)},
            "attention": {"gbs": round(atb / us["attention"] / 1e3, 1),
                          "hbm_frac": round(atb / us["attention"] / 1e3 / hbm, 4),
                          "tflops": round(atf / us["attention"] / 1e6, 1),
                          "tensor_frac": round(atf / us["attention"] / 1e6 / tflops, 4)},
            "step_gbs": round((hb + atb) / ms / 1e6, 1),
        }
        del graph, vs, d
        torch.cuda.empty_cache()
    out["inputs"] = ("drawn on the device from a seeded generator (the host recipe's distributions), logits planted "
                     "with the recipe's per-node draws; every input larger than L2, no flush")
    out["peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tflops}
    return out


def max_over_ranks(elapsed_ms: float, world: int, device) -> float:
    """The slowest rank's timed region (every rank gets it)."""
    if world <= 1:
        return elapsed_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_steps_per_s(ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank runs its own replica of the step, so the
    job completes `world` steps per (slowest-rank) step time."""
    return world / (ms_per_step / 1e3)


def _traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the source."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.md")) as f:
            rows = [ln.strip().strip("|").split("|") for ln in f if ln.startswith("| medusa_")]
        for r in rows:
            name, src, sha, nbytes = (x.strip() for x in r[:4])
            if name != kernel:
                continue
            path = os.path.join(ROOT, "medusa_head_speculative_heads_gb300", "csrc", src)
            if hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] != sha:
                return None
            return int(nbytes)
    except Exception:
        return None
    return None


def _to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


E2E_SETS = 2  # device input sets the end-to-end steps rotate through (three measured no faster)


def run_e2e(args, c, vs, inp, d, dev, stream):
    """Same step through the public calls with host buffers: every step copies
    its per-step inputs (hidden state, root token, prefix length, the verify
    pass's q and tree k/v, the base logits at the tree nodes) from pinned host
    memory and reads back the step's results (accept length, path, next token,
    new cache length).  Steps run through `PipelinedSteps`: the copy of step
    i + 1's inputs (into the second device input set) overlaps step i's
    kernels.  Weights and the KV cache stay resident (model state)."""
    import torch
    from medusa_head_speculative_heads_gb300.step import PipelinedSteps
    names = PipelinedSteps.names
    outs = [vs.accept_len, vs.path_nodes, vs.next_tok, vs.new_len]
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    pipe = PipelinedSteps(vs, {k: d[k] for k in names}, {k: d[k] for k in ("w1", "w2", "kc", "vc")}, outs, host_out,
                          n_sets=E2E_SETS)
    host, views = pipe.host_staging()  # the step's inputs staged in one pinned buffer: one upload per step
    for k in names:
        views[k].copy_(_to_dev(inp[k], "cpu"))
    for _ in range(max(3, args.warmup)):
        pipe.step(host)
    pipe.reset()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        pipe.step(host)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": round(world / (ms / 1e3), 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(pipe.bytes_h2d()), "d2h_bytes_per_step": int(pipe.bytes_d2h()),
            "overlap": f"host->device copies of the next steps' inputs (one transfer of a step's staged inputs "
                       f"each) overlap the kernels of step i ({E2E_SETS} device input sets)"}


def oracle_sample(c, inp, topo_o):
    """Times the float64 oracle on one whole verify step, every call in full
    (heads, packing, attention over all layers, acceptance, compaction over all
    layers): nothing extrapolated.  Returns (seconds, description)."""
    from oracle import step as ostep
    t0 = time.perf_counter()
    ostep.run_step(c, topo_o, inp, inp["logits"])
    work = time.perf_counter() - t0
    sample = (f"one whole verify step, nothing extrapolated: heads, tree packing, tree attention over all "
              f"{c['nl']} layers, typical acceptance, KV compaction over all layers; {work:.2f} s of CPU work, "
              f"single thread")
    return work, sample


def cpu_baseline(c, inp, topo):
    from oracle import topology as otopo
    topo_o = otopo.greedy(otopo.synthetic_accuracy(c["K"], c["tree"][1]), c["tree"][2])
    step_s, sample = oracle_sample(c, inp, topo_o)
    return {"value": round(1.0 / step_s, 6), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
            "host_cpus": os.cpu_count()}


def run_reference(args, c):
    """The oracle as it stands, timed on the host cores.

    Every step is one whole verify step of the workload (heads, tree packing,
    tree attention over all layers, typical acceptance, KV compaction over all
    layers), nothing sampled or extrapolated.  The oracle itself is
    single-threaded; independent steps run side by side on a pool of host
    threads (the C oracle releases the interpreter lock while it computes), one
    step per thread at a time.  value = steps / wall time of the timed steps."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import concurrent.futures as cf
    from oracle import step as ostep
    from oracle import topology as otopo
    import oracle
    oracle.build()
    oracle.oracle.lib()
    topo_o = otopo.greedy(otopo.synthetic_accuracy(c["K"], c["tree"][1]), c["tree"][2])
    inp = make_inputs(c, topo_o.n_nodes)
    inp["logits"] = wl.plant(c, inp["logits"], ostep.tree_tokens(c, topo_o, inp), topo_o.parent)
    threads = max(1, min(os.cpu_count() or 1, 16, args.steps))

    def one(_):
        ostep.run_step(c, topo_o, inp, inp["logits"])

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(args.warmup)))
        t0 = time.perf_counter()
        list(ex.map(one, range(args.steps)))
        wall = time.perf_counter() - t0
    ms = 1e3 * wall / args.steps
    value = args.steps / wall
    sample = (f"{args.steps} whole verify steps of the workload (heads, tree packing, tree attention over all "
              f"{c['nl']} layers, typical acceptance, KV compaction over all layers; nothing sampled or "
              f"extrapolated), each a single-thread float64 oracle step, {threads} steps at a time on "
              f"{threads} host threads; {wall:.1f} s wall")
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
                      "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic (seeded, model shapes)", "config": config_json(c, topo_o.n_nodes),
                      "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                                       "sample": sample, "host_cpus": os.cpu_count()},
                      "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--profile", choices=["heads", "attention", "accept", "rope", "linear", "head_loss"], default=None,
                    help="run only this call `steps` times after warm-up (profiler captures)")
    ap.add_argument("--configs", default="none",
                    help="other workloads timed as whole steps after the headline one: none (default), all, or a "
                         "comma list of " + ", ".join(k for k, *_ in CONFIG_RUNS))
    ap.add_argument("--profile-nodes", type=int, default=None,
                    help="with --profile: a greedy sparse tree of this many nodes instead of 64")
    ap.add_argument("--profile-batch", type=int, default=None,
                    help="with --profile: the 7B-shape batch-sweep workload at this batch instead of batch 1")
    ap.add_argument("--profile-shape", default=None,
                    help="with --profile: layers,q_heads,kv_heads,prefix of the workload (e.g. 1,8,2,32768: few "
                         "items with a long prefix)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if (args.profile_nodes is not None or args.profile_batch is not None or args.profile_shape) and not args.profile:
        ap.error("--profile-nodes / --profile-batch / --profile-shape apply to --profile runs only")
    c = wl.config("7b")
    if args.profile_batch is not None:
        c = wl.config("sweep", B=args.profile_batch)
    if args.profile_nodes is not None:
        c = wl.config(c["name"], B=c["B"], tree=(c["tree"][0], c["tree"][1], args.profile_nodes))
    if args.profile_shape:
        nl, hq, hkv, L = (int(v) for v in args.profile_shape.split(","))
        c = wl.config(c["name"], B=c["B"], tree=c["tree"], nl=nl, Hq=hq, Hkv=hkv, L=L)
    if args.impl == "reference":
        run_reference(args, c)
    else:
        run_ours(args, c)


if __name__ == "__main__":
    main()
