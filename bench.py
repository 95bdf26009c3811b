"""Benchmark of the MTP draft-layer forward on one GB300 (or N replicas).

Default workload: the Qwen-style dense draft layer (hidden 5120, 40/8 heads,
head 128, sigmoid-gated q, per-head q/k norm, 4096-token cache, SwiGLU 17408,
vocab 151936, affine 4-bit group-32 weights) at m = 1: one step = one full
draft forward (embedding gather through lm_head argmax).  Weights are 0.92 GB,
far above the 129 MB L2, so every step streams them from HBM.

``--config`` selects another workload: ``tiny_dense`` (microseconds per
draft; the 1.4 MB layer stays in L2, so it is latency-bound),
``mimo_chain`` (three chained layers of 4 rows each), ``moe`` (256 experts,
top 8 + shared; L2 flushed between steps) or ``qmatmul_sweep`` (the bare
projection at m in {1, 2, 4, 8, 16} over four shapes).

Each launch of a step is also timed alone (CUDA events recorded between the
library's launches on its stream, mtp_timing_begin/end), which gives the
roofline of the step's dominant launch.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
pages publish no runnable implementation of this path).
"""

from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MTP draft tokens/sec per layer (m=1) and HBM GB/s vs ~8 TB/s roofline"
UNIT = "draft tokens/s"
WORKLOAD = "qwen_dense"
CONFIG_CHOICES = ["tiny_dense", "qwen_dense", "mimo_chain", "moe", "qmatmul_sweep"]
DTYPE = ("int4-affine weights (f32 scales/biases); f32 activations split into f16 hi+lo parts "
         "for the tensor-core products; f32 accumulate")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD, choices=CONFIG_CHOICES)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16-stacks", action="store_true",
                    help="MoE workload: expert stacks with bfloat16 scales and biases")
    ap.add_argument("--seq", type=int, default=512, help="rows of the catch-up batch (--profile-kernel catch_up)")
    ap.add_argument("--profile-kernel", default=None,
                    choices=["lm_head", "ffn_down", "attention", "verify_head", "step", "catch_up"],
                    help="run only one entry point of the workload (small device footprint, for ncu)")
    return ap.parse_args()


# --------------------------------------------------------------- accounting
def aff(n, k):
    """Algorithmic bytes of an affine 4-bit group-32 weight [n, k]: 0.75 B per element."""
    return n * k * 3 // 4


def attn_keys(cfg):
    cached = min(cfg.cache_len, cfg.window - 1) if cfg.window > 0 else cfg.cache_len
    return cached + cfg.m


def aff_bf16(n, k):
    """An expert stack with bfloat16 scales and biases: 0.625 B per element."""
    return n * k // 2 + 2 * 2 * n * (k // 32)


def launch_plan(cfg, bf16_stacks=False):
    """(name, algorithmic HBM bytes) of each launch of one draft step, in the
    order the library enqueues them (weights at 0.75 B per element, the KV
    rows the attention reads, the activation rows read from memory)."""
    H, m = cfg.hidden, cfg.m
    nh, nkv, dq, dv = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v
    eh = aff(H, 2 * H) + 4 * (H + 2 * H * m)
    qkv = aff(cfg.q_rows + nkv * (dq + dv), H) + 4 * H * m
    attn = 4 * attn_keys(cfg) * nkv * (dq + dv)
    o = aff(H, nh * dv)
    lm = aff(cfg.vocab, H) + 4 * H
    if cfg.moe:
        E, Ie, k = cfg.n_experts, cfg.expert_intermediate, cfg.top_k
        ea = aff_bf16 if bf16_stacks else aff   # routed stacks; the shared expert is float32
        plan = [("launch A: embedding pack + eh_proj + q/k/v", eh + qkv), ("attention", attn),
                ("split merge + o_proj", o), ("router", 4 * E * H),
                ("expert gate/up + expert down + lm_head", k * 2 * ea(Ie, H) + 2 * aff(Ie, H)
                 + k * ea(H, Ie) + aff(H, Ie) + lm)]
        if H % 256:
            plan.insert(0, ("embedding/hidden norm pack", 4 * 2 * H))
        return plan
    I = cfg.intermediate
    gu, dn = 2 * aff(I, H), aff(H, I)
    if m == 1:
        plan = [("launch A: embedding pack + eh_proj + q/k/v", eh + qkv), ("attention", attn),
                ("launch B: split merge + o_proj + gate/up + down + lm_head", o + gu + dn + lm)]
        if H % 256:
            plan.insert(0, ("embedding/hidden norm pack", 4 * 2 * H))
        return plan
    return [("embedding/hidden norm pack", 4 * 2 * H * m), ("eh_proj", eh), ("q/k/v", qkv),
            ("attention", attn), ("o_proj", o), ("gate/up", gu), ("down", dn),
            ("lm_head + argmax", lm)]


def step_bytes(cfg, bf16_stacks=False):
    return sum(b for _, b in launch_plan(cfg, bf16_stacks)) * max(1, cfg.n_layers)


# --------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self):
        self.samples = []
        self._stop = threading.Event()
        self._proc = None

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self._proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self._proc.stdout:
            if self._stop.is_set():
                break
            self.samples.append([x.strip() for x in line.split(",")])

    def stop(self):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()

    def summary(self, dev_index=0):
        rows = [s for s in self.samples if s and s[0] == str(dev_index)] or self.samples
        sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for i, nm in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}




def measured_peaks():
    """(HBM GB/s, kind): the measured burst copy bandwidth of the GB300s
    (a kernel timed alone), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def gemv_source_hash():
    h = hashlib.sha256()
    for f in ("gemv.cuh", "gemv.cu", "common.cuh", "attn.cu"):
        with open(os.path.join(ROOT, "mtp_speculative_draft_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes per launch from profiles/traffic.json (ncu dram__bytes_read +
    write of one capture), or None when absent or taken on other sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            d = json.load(fh)
        e = d[key]
    except (OSError, KeyError, ValueError):
        return None
    if e.get("source_hash") != gemv_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


# --------------------------------------------------------------- CPU oracle
def _threads():
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return threads


def cpu_oracle_full_step(cfg, host):
    """One full draft step of the CPU oracle (float64), timed on this host."""
    from oracle import mtp_oracle as O
    w, shared, st, step = host
    e = shared["embed_rows"] if "embed_rows" in shared else shared["embed"][step["tokens"]]
    t0 = time.perf_counter()
    O.draft_layer(cfg, w, shared["lm_head"], st["k_cache"], st["v_cache"], step["hidden"], e)
    dt = time.perf_counter() - t0
    return {"value": 1.0 / dt, "unit": UNIT, "cores": _threads(), "kind": "oracle",
            "sample": f"one full draft step of {cfg.name} (all {cfg.vocab} vocabulary rows); "
                      f"measured {dt:.1f} s"}


def oracle_sampled_step(cfg, host, frac, rng):
    """Oracle time of one draft step estimated from a row sample.

    Every affine projection of the step runs through the oracle's qmatmul on
    ``frac`` of its output rows (time scaled by 1/frac); attention runs in
    full through the oracle's attention; norms are negligible and included.
    Returns seconds per step.
    """
    import numpy as np
    from oracle import mtp_oracle as O
    w, shared, st, step = host
    H, m = cfg.hidden, cfg.m
    mats = ["eh_proj", "wq", "wk", "wv", "wo"] + ([] if cfg.moe else ["ffn_gate", "ffn_up", "ffn_down"])
    total = 0.0
    for name in mats + ["lm_head"]:
        W = shared["lm_head"] if name == "lm_head" else w[name]
        n, k = W[0].shape[0], W[0].shape[1] * 8
        rows = np.arange(max(1, int(round(n * frac))))
        x = rng.standard_normal((1 if name == "lm_head" else m, k))
        t0 = time.perf_counter()
        O.qmatmul(x, W, rows=rows)
        total += (time.perf_counter() - t0) * n / len(rows)
    if cfg.moe:
        for name in ("exp_gate", "exp_up", "exp_down"):
            q, sc, b = w[name]
            for e in range(cfg.top_k):
                W = (q[e], sc[e], b[e])
                n, k = q.shape[1], q.shape[2] * 8
                rows = np.arange(max(1, int(round(n * frac))))
                t0 = time.perf_counter()
                O.qmatmul(rng.standard_normal((1, k)), W, rows=rows)
                total += (time.perf_counter() - t0) * n / len(rows)
    t0 = time.perf_counter()
    L = cfg.cache_len
    q = rng.standard_normal((m, cfg.n_heads, cfg.head_dim_qk))
    O.attention(q, st["k_cache"][:, :L + m], st["v_cache"][:, :L + m], [L + r for r in range(m)],
                cfg.window, w.get("sinks") if cfg.sinks else None)
    O.rmsnorm(step["hidden"], w["hnorm"], cfg.eps)
    total += time.perf_counter() - t0
    return total


# --------------------------------------------------------------- main arms
def barrier_max(world, value, device="cuda"):
    """The largest `value` over all ranks (an all-reduce; every rank returns it)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, steps, ms_total_max):
    """Whole-job draft tokens/s: the steps of every rank over the slowest rank's time."""
    return world * steps / (ms_total_max / 1000.0)


def run_reference(args):
    """CPU oracle arm: the oracle as it stands, on this host's cores.

    Each step is a bounded sample of the same draft step (every projection on
    a fraction of its rows, attention in full), sized so that the whole run
    takes a few minutes; its time is scaled to the full step.
    """
    import numpy as np
    from mtp_synth.configs import CONFIGS, make_layer_weights, make_shared, make_state, make_step
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    if args.config == "qmatmul_sweep":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the draft-layer "
                          "workloads; the sweep has no step of its own"}))
        return
    cfg = CONFIGS[args.config]
    step = make_step(cfg)
    host = (make_layer_weights(cfg), make_shared(cfg, embed_rows=step["tokens"]), make_state(cfg), step)
    rng = np.random.default_rng(0)
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    frac = 1.0 / 64
    t0 = time.perf_counter()
    oracle_sampled_step(cfg, host, frac, rng)
    took = time.perf_counter() - t0
    if took > budget:
        frac = max(1.0 / 4096, frac * budget / took)
    times = []
    for _ in range(max(1, args.warmup)):
        oracle_sampled_step(cfg, host, frac, rng)
    for _ in range(max(1, args.steps)):
        times.append(oracle_sampled_step(cfg, host, frac, rng))
    ms = 1000.0 * statistics.mean(times)
    val = 1000.0 / ms
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded SplitMix64)",
           "config": {"workload": cfg.name, "m": cfg.m, "hidden": cfg.hidden, "vocab": cfg.vocab,
                      "cache_len": cfg.cache_len},
           "cpu_baseline": {"value": val, "unit": UNIT, "cores": _threads(), "kind": "oracle",
                            "sample": (f"each step: every projection of one {cfg.name} draft step "
                                       f"on {frac:.5f} of its output rows (time scaled to all "
                                       f"rows), attention in full")},
           "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))



# --------------------------------------------------------------- device helpers
def _dev():
    import torch
    from mtp_speculative_draft_gb300 import build as B
    B.build()
    rank, world, local = dist_setup_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    return rank, world, local, dev


def dist_setup_env():
    import torch
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1 and not __import__("torch.distributed", fromlist=["x"]).is_initialized():
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


class L2Flush:
    """Writes a buffer of twice the L2 size (between timed steps, untimed)."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (128 << 20)
        self.buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.zero_()


def timed_launches(run_step, n_marks, steps, flush=None):
    """Each launch of ``run_step`` alone: a timing session per step records an
    event before every library launch and after the last; returns the mean
    duration of each launch (ms) over ``steps`` steps and the launch count."""
    import torch
    from mtp_speculative_draft_gb300.api import launch_timing
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_marks + 4)]
    for e in evs:            # create the events (torch makes them on first record)
        e.record()
    torch.cuda.synchronize()
    sums, n_launch = None, None
    for _ in range(steps):
        if flush:
            flush()
        with launch_timing(evs) as t:
            run_step()
        d = t.durations_ms()
        n_launch = len(d)
        sums = d if sums is None else [a + b for a, b in zip(sums, d)]
    return [v / steps for v in sums], n_launch


def roofline_of(plan, launch_ms, peak, peak_kind, traffic_key=None, traffic_scale=1):
    """Per-launch bandwidth and the dominant launch's roofline object."""
    rows = []
    for (name, nbytes), ms in zip(plan, launch_ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows.append({"launch": name, "ms": ms, "algorithmic_bytes": nbytes, "gbs": gbs,
                     "frac": gbs / peak})
    dom = max(range(len(plan)), key=lambda i: plan[i][1])
    traffic = profiled_traffic(traffic_key) if traffic_key else None
    r = rows[dom]
    roof = {"bound": "hbm", "kernel": r["launch"], "achieved": r["gbs"], "peak": peak,
            "unit": "GB/s", "frac": r["frac"], "traffic": traffic,
            "peak_kind": f"{peak_kind} burst copy bandwidth (kernel timed alone)",
            "algorithmic_bytes_per_launch": r["algorithmic_bytes"], "launch_ms": r["ms"]}
    return roof, rows


def graph_of(fn, stream):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
    stream.synchronize()
    return g


def time_replays(graph, stream, steps, warmup, world, flush=None):
    """Device time of ``steps`` graph replays (ms total, max over ranks), with a
    barrier and synchronize on both sides; with ``flush``, each replay is timed
    alone between its own events and the L2 is flushed between replays."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    stream.synchronize()
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        if flush is None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
            e1.synchronize()
            total = e0.elapsed_time(e1)
        else:
            pairs = []
            for _ in range(steps):
                flush()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graph.replay()
                b.record(stream)
                pairs.append((a, b))
            pairs[-1][1].synchronize()
            total = sum(a.elapsed_time(b) for a, b in pairs)
    torch.cuda.synchronize()
    clocks.stop()
    return barrier_max(world, total), clocks


# --------------------------------------------------------------- layer workloads
def run_layer_bench(args, cfg):
    import torch
    from mtp_speculative_draft_gb300 import api as A
    from mtp_speculative_draft_gb300.layer import DraftChain, DraftLayer, SharedHead
    from mtp_synth.configs import make_layer_weights, make_shared, make_state, make_step

    rank, world, local, dev = _dev()
    nl, m, H = max(1, cfg.n_layers), cfg.m, cfg.hidden
    step = make_step(cfg)
    shared = make_shared(cfg)
    sh = SharedHead(shared, dev)
    ws_l = [make_layer_weights(cfg, k) for k in range(nl)]
    sts = [make_state(cfg, k) for k in range(nl)]
    bfs = bool(args.bf16_stacks and cfg.moe)
    layers = [DraftLayer(cfg, ws_l[k], sh, sts[k], device=dev, bf16_stacks=bfs) for k in range(nl)]
    hidden = torch.from_numpy(step["hidden"]).to(dev)
    tokens = torch.from_numpy(step["tokens"]).to(dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(nl, dtype=torch.float32, device=dev)
    hid = torch.zeros((nl, H), dtype=torch.float32, device=dev)
    seq = torch.zeros(m + nl, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    if nl > 1:
        chain = DraftChain(layers)

        def fwd():
            seq[:m].copy_(tokens)   # the known tokens; the chain appends its drafts
            chain.forward(hidden, seq, [cfg.cache_len] * nl, val, hid, stream=stream)
    else:
        lyr = layers[0]

        def fwd():
            lyr.forward(hidden, cfg.cache_len, tokens=tokens, token=tok, value=val, hidden_out=hid,
                        stream=stream)

    flush = L2Flush(dev) if cfg.moe else None   # the MoE step reads less than it could cache
    graph = graph_of(fwd, stream)
    ms_total, clocks = time_replays(graph, stream, args.steps, args.warmup, world, flush)
    ms = ms_total / args.steps
    value = nl * job_value(world, args.steps, ms_total)   # draft tokens (one per layer step)

    # each launch alone (eager, same inputs)
    plan = launch_plan(cfg, bfs) * nl
    with torch.cuda.stream(stream):
        launch_ms, n_launch = timed_launches(fwd, len(plan) + 1, max(5, min(args.steps, 50)), flush)
    stream.synchronize()
    if n_launch != len(plan):
        raise RuntimeError(f"expected {len(plan)} launches per step, the library made {n_launch}")
    peak, peak_kind = measured_peaks()
    if nl > 1:  # average the chain's layers launch by launch
        per = len(plan) // nl
        launch_ms = [sum(launch_ms[i + k * per] for k in range(nl)) / nl for i in range(per)]
        plan = plan[:per]
    roof, rows = roofline_of(plan, launch_ms, peak, peak_kind, traffic_key=f"{cfg.name}.dominant")
    total_bytes = step_bytes(cfg, bfs)

    # end to end through the C ABI with pinned host buffers
    h_hidden = torch.from_numpy(step["hidden"]).pin_memory()
    h_tokens = torch.from_numpy(step["tokens"]).pin_memory()
    h_out_tok = torch.zeros(m + nl if nl > 1 else 1, dtype=torch.int32).pin_memory()
    h_out_val = torch.zeros(nl, dtype=torch.float32).pin_memory()
    e2e_steps = max(10, args.steps // 2)
    with torch.cuda.stream(stream):
        def e2e_step():
            hidden.copy_(h_hidden, non_blocking=True)
            tokens.copy_(h_tokens, non_blocking=True)
            fwd()
            h_out_tok.copy_(seq if nl > 1 else tok, non_blocking=True)
            h_out_val.copy_(val, non_blocking=True)
            stream.synchronize()
        for _ in range(3):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        t1 = time.perf_counter()
    e2e_s = barrier_max(world, t1 - t0)
    e2e_val = nl * job_value(world, e2e_steps, 1000.0 * e2e_s)
    h2d = h_hidden.numel() * 4 + h_tokens.numel() * 4
    d2h = h_out_tok.numel() * 4 + h_out_val.numel() * 4
    status = A.mtp_workspace_status(layers[0].ws)

    l2 = ("flushed between timed steps (a 2x L2 write, untimed)" if flush is not None else
          ("inputs larger than L2" if total_bytes > (256 << 20) else
           f"L2-resident ({total_bytes / 1e6:.1f} MB per step): latency-bound, roofline not meaningful"))
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded SplitMix64; value distributions of the workload)",
        "config": {"workload": cfg.name, "m": m, "layers": nl, "hidden": H, "n_heads": cfg.n_heads,
                   "n_kv_heads": cfg.n_kv_heads, "head_dim_qk": cfg.head_dim_qk,
                   "head_dim_v": cfg.head_dim_v, "intermediate": cfg.intermediate,
                   "vocab": cfg.vocab, "cache_len": cfg.cache_len, "window": cfg.window,
                   "gated_q": cfg.gated_q, "experts": cfg.n_experts, "top_k": cfg.top_k,
                   "expert_scales": ("bfloat16" if bfs else "float32") if cfg.moe else None,
                   "weights": "affine 4-bit g32", "l2": l2,
                   "timing": ("CUDA graph of one step, replayed; CUDA events on the launch "
                              "stream" + ("; each step between its own events" if flush else "")),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_draft_token": 1000.0 * ms / nl,
        "algorithmic_bytes_per_step": total_bytes,
        "hbm_gbs_step": total_bytes / (ms * 1e-3) / 1e9,
        "step_frac_of_peak": total_bytes / (ms * 1e-3) / 1e9 / peak,
        "roofline": roof,
        "launches": rows,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": len(plan) * nl * args.steps,
        "clocks": clocks.summary(local),
        "device_error_word": status,
    }
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and cfg.name == WORKLOAD):
        out["cpu_baseline"] = cpu_oracle_full_step(cfg, (ws_l[0], shared, sts[0], step))
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------- qmatmul sweep
def run_sweep(args, sc):
    import torch
    import mtp_synth
    from mtp_speculative_draft_gb300 import api as A
    from mtp_speculative_draft_gb300 import _lib as L
    from mtp_speculative_draft_gb300.layer import DeviceAffine

    rank, world, local, dev = _dev()
    peak, peak_kind = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (128 << 20)
    stream = torch.cuda.Stream(device=dev)
    results = []
    clock_all = []
    for (n, k) in sc.shapes:
        w = mtp_synth.affine4_weight(sc.seed, f"sweep.{n}x{k}", n, k)
        wbytes = aff(n, k)
        copies = max(1, -(-2 * l2 // wbytes))      # rotate copies so the L2 never serves weights
        devw = [DeviceAffine(w, dev)]
        for _ in range(copies - 1):
            d0 = devw[0]
            c = DeviceAffine.__new__(DeviceAffine)
            c.q, c.s, c.b = d0.q.clone(), d0.s.clone(), d0.b.clone()
            c.desc = A.affine4(c.q, c.s, c.b)
            devw.append(c)
        del w
        xall = torch.from_numpy(mtp_synth.normal_f32(sc.seed, f"sweep.x.{k}", (16, k))).to(dev)
        for m in sc.ms:
            x = xall[:m].contiguous()
            y = torch.zeros((m, n), dtype=torch.float32, device=dev)
            ws = A.workspace(L.load().qmatmul_affine4_workspace_bytes(m, k))

            def calls():
                for c in devw:
                    A.qmatmul_affine4(x, c.desc, y, m, ws, stream)
            g = graph_of(calls, stream)
            reps = max(3, args.steps // (4 * copies))
            total, clocks = time_replays(g, stream, reps, max(3, args.warmup // 4), world)
            clock_all.append(clocks.summary(local))
            call_ms = total / (reps * copies)
            with torch.cuda.stream(stream):
                lms, nl_ = timed_launches(calls, 2 * copies + 1, max(3, reps // 2))
            stream.synchronize()
            gemv = [lms[2 * i + 1] for i in range(copies)]   # launch 0 packs x, launch 1 is the GEMV
            gemv_ms = sum(gemv) / len(gemv)
            nbytes = wbytes + 4 * m * (k + n)
            gbs = nbytes / (gemv_ms * 1e-3) / 1e9
            results.append({"n": n, "k": k, "m": m, "call_ms": call_ms, "gemv_ms": gemv_ms,
                            "algorithmic_bytes": nbytes, "gbs": gbs, "frac": gbs / peak,
                            "weight_copies": copies})
        del devw
        torch.cuda.empty_cache()
    big = [r for r in results if r["n"] * r["k"] > 5120 * 5120]
    mean_gbs = statistics.mean(r["gbs"] for r in results)
    worst = min(results, key=lambda r: r["frac"])
    sms = [c["sm_mhz"] for c in clock_all if c["sm_mhz"]]
    out = {"metric": "qmatmul_affine4 HBM GB/s per (N x K, m)", "value": mean_gbs, "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic (seeded SplitMix64)",
           "config": {"workload": sc.name, "ms": list(sc.ms), "shapes": [list(s) for s in sc.shapes],
                      "l2": "weights rotated over copies totalling at least 2x L2",
                      "timing": "CUDA graph of the calls on every copy; the GEMV launch alone "
                                "from events between the library's launches"},
           "roofline": {"bound": "hbm", "kernel": "qmatmul_affine4 GEMV (worst case)",
                        "achieved": worst["gbs"], "peak": peak, "unit": "GB/s",
                        "frac": worst["frac"], "traffic": None, "peak_kind": peak_kind},
           "min_frac_large_shapes": min(r["frac"] for r in big) if big else None,
           "sweep": results,
           "clocks": {"sm_mhz": statistics.median(sms) if sms else None,
                      "sm_max_mhz": max((c["sm_max_mhz"] or 0) for c in clock_all) or None,
                      "reasons": sorted({x for c in clock_all for x in c["reasons"]})}}
    if rank == 0:
        print(json.dumps(out))


def run_ours(args):
    from mtp_synth.configs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.config == "qmatmul_sweep":
        run_sweep(args, cfg)
    else:
        run_layer_bench(args, cfg)


def run_profile_kernel(args):
    """Runs one entry point of the workload `--steps` times (for ncu captures)."""
    import numpy as np
    import torch
    import mtp_synth
    from mtp_speculative_draft_gb300 import build as B
    B.build()
    from mtp_speculative_draft_gb300 import api as A
    from mtp_speculative_draft_gb300.layer import DeviceAffine
    from mtp_synth.configs import CONFIGS
    cfg = CONFIGS[args.config]
    dev = torch.device("cuda", 0)
    H = cfg.hidden
    extra = {}
    if args.profile_kernel == "verify_head":
        # the pending token and three drafts through the final norm and the
        # lm_head in one pass, softcap 30, argmax per row
        rows = 4
        w = DeviceAffine(mtp_synth.affine4_weight(cfg.seed, cfg.name + ".lm_head", cfg.vocab, H), dev)
        h = torch.from_numpy(mtp_synth.normal_f32(cfg.seed, "profile.verify", (rows, H))).to(dev)
        nw = torch.ones(H, dtype=torch.float32, device=dev)
        tok = torch.zeros(rows, dtype=torch.int32, device=dev)
        val = torch.zeros(rows, dtype=torch.float32, device=dev)
        logits = torch.zeros((rows, cfg.vocab), dtype=torch.float32, device=dev)
        ws = A.verify_head_argmax(h, rows, nw, cfg.eps, w.desc, 1.0, 30.0, tok, val, logits)
        run = lambda: A.verify_head_argmax(h, rows, nw, cfg.eps, w.desc, 1.0, 30.0, tok, val,  # noqa: E731
                                           logits, ws)
        # weights once, the rows in, the logits out (read back once by the argmax pass)
        weight_bytes = cfg.vocab * H // 2 + 2 * cfg.vocab * (H // 32) * 4
        extra["rows"] = rows
        extra["algorithmic_bytes_per_call"] = weight_bytes + rows * H * 4 + 2 * rows * cfg.vocab * 4
    elif args.profile_kernel in ("lm_head", "ffn_down"):
        if args.profile_kernel == "lm_head":
            n, k, name = cfg.vocab, H, cfg.name + ".lm_head"
        else:
            n, k, name = H, cfg.intermediate, f"{cfg.name}.L0.ffn_down"
        w = DeviceAffine(mtp_synth.affine4_weight(cfg.seed, name, n, k), dev)
        x = torch.from_numpy(mtp_synth.normal_f32(cfg.seed, "profile.x", (1, k))).to(dev)
        extra["algorithmic_bytes_per_call"] = aff(n, k) + 4 * k
        if args.profile_kernel == "lm_head":
            tok = torch.zeros(1, dtype=torch.int32, device=dev)
            val = torch.zeros(1, dtype=torch.float32, device=dev)
            ws = A.workspace(__import__("mtp_speculative_draft_gb300._lib", fromlist=["x"]).load()
                             .lmhead_argmax_workspace_bytes(k, n))
            run = lambda: A.lmhead_argmax(x[0], None, cfg.eps, w.desc, tok, val, None, None, ws)  # noqa: E731
        else:
            y = torch.zeros((1, n), dtype=torch.float32, device=dev)
            ws = None
            run = lambda: A.qmatmul_affine4(x, w.desc, y, 1, ws)  # noqa: E731
            ws = A.qmatmul_affine4(x, w.desc, y, 1)
    elif args.profile_kernel == "catch_up":
        # KV catch-up of a target batch of --seq rows (tcgen05 projections)
        from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
        from mtp_synth.configs import make_layer_weights, make_shared, make_state
        seq = args.seq
        c2 = cfg.with_(cache_len=0, m=seq)
        shared = make_shared(c2, embed_rows=np.arange(seq) % cfg.vocab)
        lyr = DraftLayer(cfg, make_layer_weights(cfg), SharedHead(shared, dev), make_state(c2),
                         device=dev)
        rows = torch.from_numpy(shared["embed_rows"]).to(dev)
        target = torch.from_numpy(mtp_synth.normal_f32(cfg.seed, "profile.target", (seq, H))).to(dev)
        run = lambda: lyr.catch_up(target, seq, 0, embed_rows=rows, pending=target[0])  # noqa: E731
        nkv, dq, dv = cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v
        flop = 2 * seq * (H * 2 * H + H * nkv * (dq + dv))
        extra.update(seq=seq, algorithmic_flop_per_call=flop,
                     weight_bytes=aff(H, 2 * H) + aff(nkv * (dq + dv), H))
    elif args.profile_kernel == "step":
        # one whole draft step, embedding rows passed directly (no 3 GB table
        # on the device), for launch lists and captures of the step's launches
        from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
        from mtp_synth.configs import make_layer_weights, make_shared, make_state, make_step
        step = make_step(cfg)
        shared = make_shared(cfg, embed_rows=step["tokens"])
        lyr = DraftLayer(cfg, make_layer_weights(cfg), SharedHead(shared, dev), make_state(cfg),
                         device=dev)
        hidden = torch.from_numpy(step["hidden"]).to(dev)
        rows = torch.from_numpy(shared["embed_rows"]).to(dev)
        tok = torch.zeros(1, dtype=torch.int32, device=dev)
        val = torch.zeros(1, dtype=torch.float32, device=dev)
        run = lambda: lyr.forward(hidden, cfg.cache_len, embed_rows=rows, token=tok,  # noqa: E731
                                  value=val)
        extra["algorithmic_bytes_per_call"] = step_bytes(cfg)
    else:
        from mtp_synth.configs import make_state
        g = A.attn_geom(cfg.n_heads, cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v, cfg.rot_dim,
                        cfg.window, cfg.gated_q, cfg.eps)
        st = make_state(cfg)
        kc = torch.from_numpy(st["k_cache"]).to(dev)
        vc = torch.from_numpy(st["v_cache"]).to(dev)
        rng = np.random.default_rng(0)
        qp = torch.from_numpy(rng.standard_normal((cfg.m, cfg.q_rows)).astype(np.float32)).to(dev)
        kp = torch.from_numpy(rng.standard_normal((cfg.m, cfg.n_kv_heads * cfg.head_dim_qk)).astype(np.float32)).to(dev)
        vp = torch.from_numpy(rng.standard_normal((cfg.m, cfg.n_kv_heads * cfg.head_dim_v)).astype(np.float32)).to(dev)
        rope = torch.empty(kc.shape[1] * cfg.rot_dim, device=dev)
        A.mtp_rope_table(rope, kc.shape[1], cfg.rot_dim, cfg.rope_theta)
        out = torch.zeros((cfg.m, cfg.n_heads * cfg.head_dim_v), device=dev)
        ws = A.attn_decode_sink(g, qp, kp, vp, None, None, rope, None, kc, vc, cfg.cache_len,
                                kc.shape[1], cfg.m, out)
        run = lambda: A.attn_decode_sink(g, qp, kp, vp, None, None, rope, None, kc, vc,  # noqa: E731
                                         cfg.cache_len, kc.shape[1], cfg.m, out, ws)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    if args.profile_kernel == "catch_up":
        from mtp_speculative_draft_gb300.api import launch_timing
        lms, nl_ = timed_launches(run, 8, 10)
        extra["launch_ms"] = lms
        gemm_ms = lms[1] + lms[3]
        extra["gemm_tflops"] = extra["algorithmic_flop_per_call"] / (gemm_ms * 1e-3) / 1e12
        extra["call_tflops"] = extra["algorithmic_flop_per_call"] / (ms * 1e-3) / 1e12
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            pk = json.load(fh)
        # three bf16 products per K16 step (hi*hi, hi*lo, lo*hi): the tensor pipe
        # issues 3x the algorithmic flops
        extra["tensor_frac_of_bf16_peak"] = 3 * extra["gemm_tflops"] / float(pk["bf16_tflops"])
    if "algorithmic_bytes_per_call" in extra:
        peak, kind = measured_peaks()
        extra["gbs"] = extra["algorithmic_bytes_per_call"] / (ms * 1e-3) / 1e9
        extra["frac"] = extra["gbs"] / peak
        extra["peak_gbs"] = peak
        extra["peak_kind"] = kind
    print(json.dumps({"profile_kernel": args.profile_kernel, "workload": cfg.name,
                      "ms_per_call": ms, **extra}))


def main():
    args = parse()
    if args.profile_kernel:
        run_profile_kernel(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
