"""Benchmark of the MTP draft-layer forward on one GB300 (or N replicas).

Workload: the Qwen-style dense draft layer (hidden 5120, 40/8 heads, head 128,
sigmoid-gated q, per-head q/k norm, 4096-token cache, SwiGLU 17408, vocab
151936, affine 4-bit group-32 weights) at m = 1: one step = one full draft
forward (embedding gather through lm_head argmax).  Weights are 0.92 GB, far
above the 129 MB L2, so every step streams them from HBM.

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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-kernel", default=None, choices=["lm_head", "ffn_down", "attention", "verify_head"],
                    help="run only one entry point of the workload (small device footprint, for ncu)")
    return ap.parse_args()


# --------------------------------------------------------------- accounting
def layer_bytes(cfg):
    """Algorithmic HBM bytes of one draft step, by sub-step (weights at 0.75 B/element)."""
    H, m = cfg.hidden, cfg.m
    aff = lambda n, k: n * k * 3 // 4  # noqa: E731
    nh, nkv, dq, dv = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim_qk, cfg.head_dim_v
    keys = (min(cfg.cache_len, cfg.window - 1) if cfg.window > 0 else cfg.cache_len) + m
    b = {
        "eh_proj": aff(H, 2 * H) + 4 * (H + 2 * H * m),
        "qkv": aff(cfg.q_rows + nkv * (dq + dv), H) + 4 * H * m,
        "attention": 4 * keys * nkv * (dq + dv),
        "o_proj": aff(H, nh * dv),
    }
    if cfg.moe:
        E, I = cfg.n_experts, cfg.expert_intermediate
        b["ffn"] = 4 * E * H + (cfg.top_k + 1) * 3 * aff(I, H)
    else:
        b["ffn"] = 3 * aff(cfg.intermediate, H)
    b["lm_head"] = aff(cfg.vocab, H) + 4 * H
    return b


def launches_per_step(cfg):
    # m = 1 dense: one-row launch A (embedding pack + eh_proj + q/k/v), attention,
    # one-row launch B (split merge + o_proj + gate/up + down + lm_head).
    # m > 1 dense: norm/pack, eh_proj, q/k/v, attention, o_proj, gate/up, down, lm_head.
    # MoE (m = 1): launch A, attention, o_proj, router, expert gate/up, expert down,
    # final norm, lm_head.
    if cfg.moe:
        return 8
    return 3 if cfg.m == 1 else 8


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
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def gemv_source_hash():
    h = hashlib.sha256()
    for f in ("gemv.cuh", "gemv.cu", "common.cuh"):
        with open(os.path.join(ROOT, "mtp_speculative_draft_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    vals = {}
    for ln in lines:
        if ":" in ln and ln.strip().startswith("- "):
            k, v = ln.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != gemv_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


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
def dist_setup(args):
    import torch
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


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


def run_ours(args):
    import numpy as np
    import torch
    from mtp_speculative_draft_gb300 import build as B
    B.build()
    from mtp_speculative_draft_gb300 import _lib as L
    from mtp_speculative_draft_gb300.layer import DraftLayer, SharedHead
    from mtp_synth.configs import CONFIGS, make_layer_weights, make_shared, make_state, make_step

    rank, world, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = CONFIGS[args.config]
    step = make_step(cfg)
    w = make_layer_weights(cfg)
    shared = make_shared(cfg)
    st = make_state(cfg)
    lyr = DraftLayer(cfg, w, SharedHead(shared, dev), st, device=dev)
    H, m = cfg.hidden, cfg.m
    hidden = torch.from_numpy(step["hidden"]).to(dev)
    tokens = torch.from_numpy(step["tokens"]).to(dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    val = torch.zeros(1, dtype=torch.float32, device=dev)
    hid = torch.zeros(H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def fwd():
        lyr.forward(hidden, cfg.cache_len, tokens=tokens, token=tok, value=val, hidden_out=hid,
                    stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            fwd()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fwd()
    stream.synchronize()

    # ---------------- timed region: graph replays, inputs resident in HBM
    with torch.cuda.stream(stream):   # replay() launches on the current stream
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    clocks.stop()
    ms_total = barrier_max(world, ev0.elapsed_time(ev1))
    ms = ms_total / args.steps
    value = job_value(world, args.steps, ms_total)

    # ---------------- per-kernel breakdown (events between launches, same steps)
    # The dominant kernel is the lm_head GEMV; time it alone in the same stream
    # with the same inputs (normalised hidden already packed by the step).
    from mtp_speculative_draft_gb300 import api as A
    y_dev = hid.clone()
    logits = None
    lm_ws = A.workspace(L.load().lmhead_argmax_workspace_bytes(H, cfg.vocab))
    lm_desc = lyr.shared.lm_head.desc
    with torch.cuda.stream(stream):
        for _ in range(5):
            A.lmhead_argmax(y_dev, None, cfg.eps, lm_desc, tok, val, logits, None, lm_ws, stream)
        e_norm0 = torch.cuda.Event(enable_timing=True)
        e_norm1 = torch.cuda.Event(enable_timing=True)
        # norm-only cost (same launch with no weights streamed is not available):
        # time lm_head (norm + GEMV) and a norm-only rmsnorm of the same row.
        ta = torch.cuda.Event(enable_timing=True)
        tb = torch.cuda.Event(enable_timing=True)
        ta.record(stream)
        for _ in range(args.steps):
            A.lmhead_argmax(y_dev, None, cfg.eps, lm_desc, tok, val, logits, None, lm_ws, stream)
        tb.record(stream)
        e_norm0.record(stream)
        nw = torch.ones(H, device=dev)
        tmp = torch.empty(H, device=dev)
        for _ in range(args.steps):
            A.rmsnorm_residual(y_dev, None, nw, tmp, None, 1, H, cfg.eps, stream)
        e_norm1.record(stream)
    stream.synchronize()
    head_ms = (ta.elapsed_time(tb) - e_norm0.elapsed_time(e_norm1)) / args.steps
    bytes_map = layer_bytes(cfg)
    head_bytes = bytes_map["lm_head"]
    peak, peak_kind = measured_peaks()
    achieved = head_bytes / (head_ms * 1e-3) / 1e9
    traffic = profiled_traffic("gemv_lm_head_qwen_dense")
    total_bytes = sum(bytes_map.values())

    # ---------------- end to end through the C ABI with host buffers
    h_hidden = torch.from_numpy(step["hidden"]).pin_memory()
    h_tokens = torch.from_numpy(step["tokens"]).pin_memory()
    h_out_tok = torch.zeros(1, dtype=torch.int32).pin_memory()
    h_out_val = torch.zeros(1, dtype=torch.float32).pin_memory()
    e2e_steps = max(10, args.steps // 2)
    with torch.cuda.stream(stream):
        def e2e_step():
            hidden.copy_(h_hidden, non_blocking=True)
            tokens.copy_(h_tokens, non_blocking=True)
            fwd()
            h_out_tok.copy_(tok, non_blocking=True)
            h_out_val.copy_(val, non_blocking=True)
            stream.synchronize()
            return int(h_out_tok[0])
        for _ in range(3):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        t1 = time.perf_counter()
    e2e_s = barrier_max(world, t1 - t0)
    e2e_val = job_value(world, e2e_steps, 1000.0 * e2e_s)
    h2d = h_hidden.numel() * 4 + h_tokens.numel() * 4
    d2h = 8

    # ---------------- check the result once against itself (token = argmax)
    status = A.mtp_workspace_status(lyr.ws)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4-affine weights, f32 activations, bf16x2-split tensor-core products, f32 accumulate",
        "data": "synthetic (seeded SplitMix64; value distributions of the workload)",
        "config": {"workload": cfg.name, "m": m, "hidden": H, "n_heads": cfg.n_heads,
                   "n_kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim_qk,
                   "intermediate": cfg.intermediate, "vocab": cfg.vocab,
                   "cache_len": cfg.cache_len, "gated_q": cfg.gated_q,
                   "weights": "affine 4-bit g32", "l2": "inputs larger than L2 (0.92 GB of weights per step)",
                   "timing": "CUDA graph of one draft step, replayed; CUDA events on the launch stream",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "algorithmic_bytes_per_step": total_bytes,
        "hbm_gbs_step": total_bytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "gemv_row_kernel: lm_head projection + argmax, timed alone",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": head_bytes, "launch_ms": head_ms},
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step(cfg) * args.steps,
        "clocks": clocks.summary(local),
        "device_error_word": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_oracle_full_step(cfg, (w, shared, st, step))
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


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
