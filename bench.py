#!/usr/bin/env python
"""Benchmark of the per-step dynamic-vocabulary draft LM head on GB300.

One step = one decode step of the hot path on one sequence: verify Top-K,
draft-tree dedup, stream append, window counts and bitmap, ascending
compaction into I_t, gather of W_head[I_t, :] into the packed buffer,
projection of the draft hidden states and top-k remapped to global ids
(ns_step: one cooperative kernel that does all of it).  Workload: Llama-3-8B-shaped draft head (V=128256,
H=4096, W_max=3072, K_pre=K_ver=3, 60-node trees, top-10), seeded synthetic
inputs resident in HBM before the timed region; by default the first 20
decode steps after the prefill (|I_t| about 3k, the operating point of the
metric).  L2 (129 MB) is flushed
before every timed step by writing a 256 MiB buffer, and the time of the
flushes alone is subtracted: between two draft steps a real system runs the
target model, which evicts the sub-head rows.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft sub-LM-head steps/sec and us/step at V=128k,H=4096,|I_t|~3k; % HBM roofline"
DEFAULT_WORKLOAD = "llama3_8b_v128256_h4096"
FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-extra", action="store_true", help="skip the dense-head and pinned-point extras")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip extra.workloads (the Qwen-2.5-7B head, the Qwen3-8B W_max sweep with its dense heads, "
                        "the 16-sequence batch)")
    p.add_argument("--workload-steps", type=int, default=24,
                   help="decode steps per extra workload, from its prefill (0: the workload's full count)")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle sample")
    p.add_argument("--decode-steps", type=int, default=0,
                   help="generate inputs for only this many decode steps (0: the workload's count); "
                        "timed steps cycle through them")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            sel = [f"--id={self.index}"] if self.index is not None else []
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        load = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(load)}


def source_hash() -> str:
    """Hash of the sources the step kernel is compiled from (the one-launch
    step and the tcgen05 tile it runs)."""
    h = hashlib.sha256()
    for f in ("ns_step.cu", "ns_umma_tile.cuh", "ns_internal.cuh", "ns_ptx.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_draft_stream_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic_per_byte():
    """DRAM bytes per algorithmic byte of the step kernel, from the committed
    ncu summary, if it was taken on the current source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    return float(d["dram_bytes"]) / float(d["algorithmic_bytes"])


def step_bytes(m, n, H, V):
    """Algorithmic bytes of one whole step: rows read + packed written,
    logits written, hiddens read, one verify row read, bitmap and I_t."""
    return 2 * m * H * 2 + n * m * 4 + n * H * 2 + V * 4 + 2 * ((V + 7) // 8) + 4 * m


def proj_bytes(m, n, H):
    """Algorithmic bytes of the fused gather + projection + top-k kernel."""
    return 2 * m * H * 2 + n * m * 4 + n * H * 2 + 4 * m


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def time_oracle(cfg, wl, steps_wanted: int, budget_s: float, warmup: int = 0):
    import oracle

    W = wl.w_head()
    ost = oracle.OracleStream(cfg.V, cfg.W_max, cfg.K_pre, cfg.K_ver)
    ost.init(wl.prompt(0), wl.prefill_logits(0))
    trees = wl.trees(0)

    def one(t):
        u = t % cfg.steps
        ost.append(trees[u], wl.verify_logits(0, u), wl.verify_row(0, u))
        I = ost.active()
        oracle.sub_head_step(wl.hiddens(0, u), W, I, cfg.k)

    for t in range(warmup):
        one(t)
    done = 0
    t0 = time.perf_counter()
    while done < steps_wanted:
        one(warmup + done)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done, dt


def single_thread_oracle(workload: str, steps: int, timeout_s: float = 180.0):
    """The reference arm's oracle sample in a child process limited to one
    BLAS/OpenMP thread (the thread counts are read when numpy loads, so they
    are set in the child's environment).  None when the child fails."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
           "--steps", str(steps), "--warmup", "0"]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=timeout_s)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")][-1]
        d = json.loads(line)
        return {"value": d["value"], "unit": d["unit"], "cores": 1, "sample": d["cpu_baseline"]["sample"]}
    except (subprocess.SubprocessError, OSError, IndexError, ValueError, KeyError):
        return None


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synth import Workload, get_config

    cfg = get_config(args.workload)
    wl = Workload(cfg)
    done, dt = time_oracle(cfg, wl, args.steps, budget_s=150.0, warmup=args.warmup)
    v = done / dt
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / done, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "V": cfg.V, "H": cfg.H, "W_max": cfg.W_max, "K_pre": cfg.K_pre,
                   "K_ver": cfg.K_ver, "n_tree": cfg.n_tree, "k": cfg.k, "parallelism": "replicas x1"},
        "cpu_baseline": {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {done} decode steps of {cfg.name} after its prefill init"},
        "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our CUDA path
# ---------------------------------------------------------------------------
def graph_time_us(fn, flush, reps=32):
    """Device time of fn in us: (graph of reps x [flush + fn]) - (graph of reps x [flush])."""
    import torch

    def capture(with_op):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                flush.zero_()
                if with_op:
                    fn()
        return g

    fn()
    torch.cuda.synchronize()
    g_op, g_fl = capture(True), capture(False)
    out = []
    for g in (g_op, g_fl, g_op, g_fl):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return 1e3 * min(out[0] - out[1], out[2] - out[3]) / reps


def decode_inputs(cfg, dev, seq=0):
    """One sequence's inputs of a workload, on the device: W_head, prompt,
    prefill logits, trees, verify rows and hiddens of every decode step."""
    import torch
    from synth import Workload

    wl = Workload(cfg)
    T = cfg.steps
    return {"W": torch.from_numpy(wl.w_head().view(np.int16)).to(dev),
            "prompt": torch.from_numpy(wl.prompt(seq)).to(dev),
            "Z": torch.from_numpy(wl.prefill_logits(seq)).to(dev),
            "trees": torch.from_numpy(wl.trees(seq)).to(dev),
            "verify": torch.from_numpy(np.stack([wl.verify_logits(seq, t) for t in range(T)])).to(dev),
            "vrows": [wl.verify_row(seq, t) for t in range(T)],
            "hid": torch.from_numpy(np.stack([wl.hiddens(seq, t) for t in range(T)]).view(np.int16)).to(dev)}


def time_decode(ns, cfg, dev, flush, warmup, inp):
    """Per-step time of ns_step over every decode step of one workload (graph of
    steps minus graph of flushes, median of three replays from the prefill
    state) and the |I_t| of each step.  `inp` is decode_inputs(cfg, ...)."""
    import torch

    n, H, V, k, T = cfg.n_tree, cfg.H, cfg.V, cfg.k, cfg.steps
    W_d, prompt_d, Z_d, trees_d = inp["W"], inp["prompt"], inp["Z"], inp["trees"]
    verify_d, vrows, hid_d = inp["verify"], inp["vrows"], inp["hid"]
    logits = torch.empty((n, cfg.W_max), dtype=torch.float32, device=dev)
    ids = torch.empty((n, k), dtype=torch.int32, device=dev)
    vals = torch.empty((n, k), dtype=torch.float32, device=dev)
    h = ns.Handle(V, H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=n, max_k=k, max_prompt=prompt_d.numel())
    try:
        def init():
            h.stream_init(0, prompt_d, Z_d)
            h.build_active_vocab(0)

        def step(t):
            h.step(0, trees_d[t], verify_d[t], vrows[t], W_d, hid_d[t], k, logits=logits, ids=ids, vals=vals)

        init()
        for t in range(min(warmup, T)):
            step(t)
        torch.cuda.synchronize()
        graphs = []
        for with_steps in (True, False):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for t in range(T):
                    flush.zero_()
                    if with_steps:
                        step(t)
            graphs.append(g)
        diffs = []
        for _ in range(3):
            ms = []
            for g in graphs:
                init()
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(b))
            diffs.append(ms[0] - ms[1])
        del graphs
        init()
        _, cnt, _, _ = h.get_active(0)
        counts = torch.zeros(T, dtype=torch.int32, device=dev)
        for t in range(T):
            step(t)
            counts[t:t + 1].copy_(cnt)
        m = counts.cpu().numpy()
        if h.get_error() != 0:
            raise RuntimeError(f"device error flags set during the {cfg.name} steps")
        us = 1e3 * sorted(diffs)[1] / T
        pb = float(np.mean([proj_bytes(int(x), n, H) for x in m]))
        sb = float(np.mean([step_bytes(int(x), n, H, V) for x in m]))
        return {"us_per_step": us, "steps_per_s": 1e6 / us, "steps": T, "mean_active": float(m.mean()),
                "min_active": int(m.min()), "max_active": int(m.max()), "step_bytes_mean": sb,
                "step_hbm_frac": sb / (us * 1e-6) / 1e9 / load_peaks()[0], "proj_bytes_mean": pb}
    finally:
        h.close()


def run_workloads(ns, dev, flush, warmup, steps):
    """The other draft-head shapes: Qwen-2.5-7B (H = 3584) and the Qwen3-8B
    W_max sweep, each point over its first `steps` decode steps from prefill
    (0: all of them); the Qwen3 head also with the full-vocabulary dense head
    (cuBLAS and ours) and the static first-32768 sub-head on the same hiddens;
    the 16-sequence batch."""
    import torch
    from synth import get_config

    def short(cfg):
        return cfg.with_(steps=min(cfg.steps, steps)) if steps > 0 else cfg

    out = {}
    q25 = short(get_config("qwen25_7b_v152064_h3584"))
    out[q25.name] = time_decode(ns, q25, dev, flush, warmup, decode_inputs(q25, dev))
    torch.cuda.empty_cache()
    q3 = short(get_config("qwen3_8b_v151936_h4096"))
    inp = decode_inputs(q3, dev)  # the inputs do not depend on W_max
    pts = {}
    for W_max in q3.W_max_sweep:
        pts[str(W_max)] = time_decode(ns, q3.with_(W_max=W_max), dev, flush, warmup, inp)
    W_d, hid = inp["W"], inp["hid"][0]
    n, k, V = q3.n_tree, q3.k, q3.V
    h = ns.Handle(V, q3.H, q3.W_max, q3.K_pre, q3.K_ver, max_tree=n, max_k=k, max_prompt=16)
    try:
        ids = torch.empty((n, k), dtype=torch.int32, device=dev)
        vals = torch.empty((n, k), dtype=torch.float32, device=dev)
        dl = torch.empty((n, V), dtype=torch.float32, device=dev)
        dout = torch.empty((n, V), dtype=torch.bfloat16, device=dev)
        hb, Wb = hid.view(torch.bfloat16), W_d.view(torch.bfloat16)
        dense = {"cublas_matmul_us": graph_time_us(lambda: torch.matmul(hb, Wb.t(), out=dout), flush),
                 "ours_dense_topk_us": graph_time_us(lambda: h.dense_lm_head_topk(W_d, V, hid, k, logits=dl,
                                                                                  ids=ids, vals=vals), flush),
                 "ours_static32768_topk_us": graph_time_us(lambda: h.dense_lm_head_topk(W_d, 32768, hid, k,
                                                                                        logits=dl, ids=ids,
                                                                                        vals=vals), flush)}
    finally:
        h.close()
    out[q3.name] = {"W_max_sweep": pts, "dense_head": dense}
    del inp, W_d, hid
    torch.cuda.empty_cache()
    b16 = short(get_config("batched16_v128256_h4096"))
    out[b16.name] = time_batched(ns, b16, dev, flush, warmup)
    return out


def time_batched(ns, cfg, dev, flush, warmup):
    """The batched-serving workload: every decode step of all sequences by
    ns_step_batch (two launches), against the same steps issued as one ns_step
    per sequence; each timed from the prefill state (graph of steps minus
    graph of flushes, median of three replays)."""
    import torch
    from synth import Workload

    wl = Workload(cfg)
    B, n, H, V, k, T = cfg.batch, cfg.n_tree, cfg.H, cfg.V, cfg.k, cfg.steps
    W_d = torch.from_numpy(wl.w_head().view(np.int16)).to(dev)
    prompts = [torch.from_numpy(wl.prompt(b)).to(dev) for b in range(B)]
    Zs = [torch.from_numpy(wl.prefill_logits(b)).to(dev) for b in range(B)]
    trees_d = torch.from_numpy(np.ascontiguousarray(np.stack([wl.trees(b)[:T] for b in range(B)], axis=1))).to(dev)
    verify_d = torch.from_numpy(np.stack([np.stack([wl.verify_logits(b, t) for b in range(B)])
                                          for t in range(T)])).to(dev)  # [T, B, n_v, V]
    vrows = [[wl.verify_row(b, t) for b in range(B)] for t in range(T)]
    hid_d = torch.from_numpy(np.stack([np.stack([wl.hiddens(b, t) for b in range(B)])
                                       for t in range(T)]).view(np.int16)).to(dev)  # [T, B, n, H]
    logits = torch.empty((B, n, cfg.W_max), dtype=torch.float32, device=dev)
    ids = torch.empty((B, n, k), dtype=torch.int32, device=dev)
    vals = torch.empty((B, n, k), dtype=torch.float32, device=dev)
    h = ns.Handle(V, H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=n, max_k=k, batch=B,
                  max_prompt=max(p.numel() for p in prompts))
    try:
        def init():
            for b in range(B):
                h.stream_init(b, prompts[b], Zs[b])
                h.build_active_vocab(b)

        def batched(t):
            h.step_batch(trees_d[t], verify_d[t], vrows[t], W_d, hid_d[t], k, logits=logits, ids=ids, vals=vals)

        u_ids, u_cnt, _, _, cap = h.get_union()
        u_logits = torch.empty((B, n, cap), dtype=torch.float32, device=dev)

        def unioned(t):
            h.step_batch_union(trees_d[t], verify_d[t], vrows[t], W_d, hid_d[t], k, logits=u_logits, ids=ids,
                               vals=vals)

        def one_by_one(t):
            for b in range(B):
                h.step(b, trees_d[t, b], verify_d[t, b], vrows[t][b], W_d, hid_d[t, b], k, logits=logits[b],
                       ids=ids[b], vals=vals[b])

        def per_step_us(fn):
            init()
            for t in range(min(warmup, T)):
                fn(t)
            torch.cuda.synchronize()
            graphs = []
            for with_steps in (True, False):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for t in range(T):
                        flush.zero_()
                        if with_steps:
                            fn(t)
                graphs.append(g)
            diffs = []
            for _ in range(3):
                ms = []
                for g in graphs:
                    init()
                    torch.cuda.synchronize()
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    g.replay()
                    e.record()
                    torch.cuda.synchronize()
                    ms.append(a.elapsed_time(e))
                diffs.append(ms[0] - ms[1])
            return 1e3 * sorted(diffs)[1] / T

        us_b = per_step_us(batched)
        us_u = per_step_us(unioned)
        us_s = per_step_us(one_by_one)
        init()
        u_rows = torch.zeros(T, dtype=torch.int32, device=dev)
        sum_rows = torch.zeros(T, dtype=torch.int64, device=dev)
        for t in range(T):
            unioned(t)
            u_rows[t:t + 1].copy_(u_cnt)
            sum_rows[t] = sum(h.get_active(b)[1][0].to(torch.int64) for b in range(B))
        u_rows, sum_rows = u_rows.cpu().numpy(), sum_rows.cpu().numpy()
        init()
        _, cnt, _, _ = h.get_active(0)
        act = torch.zeros((T, B), dtype=torch.int32, device=dev)
        for t in range(T):
            batched(t)
            for b in range(B):
                act[t, b:b + 1].copy_(h.get_active(b)[1])
        act = act.cpu().numpy()
        if h.get_error() != 0:
            raise RuntimeError("device error flags set during the batched steps")
        return {"sequences": B, "steps": T, "batched_step_us": us_b, "sequence_steps_per_s": B * 1e6 / us_b,
                "one_call_per_sequence_step_us": us_s, "speedup_batched": us_s / us_b,
                "mean_active": float(act.mean()),
                "union_step_us": us_u, "union_sequence_steps_per_s": B * 1e6 / us_u,
                "union_rows_mean": float(u_rows.mean()), "rows_of_all_sequences_mean": float(sum_rows.mean()),
                "union_note": "ns_step_batch_union: one gather of W_head[U, :] for the union U of the sequences' "
                              "I_t; each sequence projects all of U and ranks its own columns"}
    finally:
        h.close()


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from speculative_decoding_draft_stream_gb300 import build as nsbuild

    nsbuild.build()
    import speculative_decoding_draft_stream_gb300 as ns
    from speculative_decoding_draft_stream_gb300 import replicas
    from synth import Workload, get_config

    cfg = get_config(args.workload)
    wl = Workload(cfg)
    (seq,) = replicas.rank_sequences(rank, world)  # replicas: every rank decodes its own sequence
    n, H, V, k = cfg.n_tree, cfg.H, cfg.V, cfg.k
    T = min(cfg.steps, args.decode_steps) if args.decode_steps > 0 else cfg.steps

    # ---- inputs, resident in HBM -------------------------------------------
    W = wl.w_head()
    W_d = torch.from_numpy(W.view(np.int16)).to(dev)
    prompt = wl.prompt(seq)
    prompt_d = torch.from_numpy(prompt).to(dev)
    Z_d = torch.from_numpy(wl.prefill_logits(seq)).to(dev)
    trees_h = wl.trees(seq)
    trees_d = torch.from_numpy(trees_h).to(dev)
    verify_h = np.stack([wl.verify_logits(seq, t) for t in range(T)])  # [T, n_v, V]
    vrows = [wl.verify_row(seq, t) for t in range(T)]
    hid_h = np.stack([wl.hiddens(seq, t) for t in range(T)]).view(np.int16)  # [T, n, H]
    verify_d = torch.from_numpy(verify_h).to(dev)
    hid_d = torch.from_numpy(hid_h).to(dev)
    logits = torch.empty((n, cfg.W_max), dtype=torch.float32, device=dev)
    ids = torch.empty((n, k), dtype=torch.int32, device=dev)
    vals = torch.empty((n, k), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    h = ns.Handle(V, H, cfg.W_max, cfg.K_pre, cfg.K_ver, max_tree=n, max_k=k, max_prompt=len(prompt))
    stream = torch.cuda.current_stream()

    def init():
        h.stream_init(0, prompt_d, Z_d)
        h.build_active_vocab(0)

    def step(t):
        u = t % T
        h.step(0, trees_d[u], verify_d[u], vrows[u], W_d, hid_d[u], k, logits=logits, ids=ids, vals=vals)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return replicas.max_over_ranks(x, dist, dev)

    clocks = ClockSampler(local if world > 1 else None)
    clocks.start()

    # ---- prefill init (per request, timed on its own) ------------------------
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    init()  # first call pays one-time costs
    torch.cuda.synchronize()
    flush.zero_()
    e0.record()
    init()
    e1.record()
    torch.cuda.synchronize()
    init_ms = e0.elapsed_time(e1)

    # ---- warm-up, then the timed decode steps -------------------------------
    # The K steps, each preceded by an L2 flush, are captured into one CUDA
    # graph (so the host never paces the GPU) and replayed from the same
    # prefill state; a second graph holds the K flushes alone.  Step time =
    # (steps graph - flush graph) / K, both timed with events on this stream.
    for t in range(args.warmup):
        step(t)
    K = args.steps
    torch.cuda.synchronize()

    def capture(with_steps, traced=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for t in range(K):
                flush.zero_()
                if with_steps:
                    if traced is not None:
                        h.trace_events(traced[t])
                    step(t)
                    if traced is not None:
                        counts[t:t + 1].copy_(cnt)
            if traced is not None:
                h.trace_events(None)
        return g

    def replay_ms(g, reset):
        if reset:
            init()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        barrier()
        return a.elapsed_time(b)

    act, cnt, _, _ = h.get_active(0)
    counts = torch.zeros(K, dtype=torch.int32, device=dev)
    g_steps, g_flush = capture(True), capture(False)
    rounds = [(replay_ms(g_steps, True), replay_ms(g_flush, False)) for _ in range(3)]
    if h.get_error() != 0:
        raise RuntimeError("device error flags set during the timed steps")
    diffs = sorted(x - y for x, y in rounds)
    total_ms = max_over_ranks(diffs[len(diffs) // 2])  # median of three
    steps_per_s = replicas.whole_job_rate(K, world, total_ms / 1e3)
    del g_steps, g_flush

    # ---- per-kernel breakdown: the same K steps with ns_step's trace events ---
    # ns_step records four events per step (external graph nodes): before the
    # state update, between the two kernels, after the fused kernel, after
    # its tail.  Tracing turns off the programmatic overlap of the two
    # kernels and each event node adds about a microsecond, so the breakdown
    # explains the step time but is not the step time.
    tev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for evs in tev:
        for e in evs:
            e.record()  # torch creates CUDA events lazily; create them before capture
    torch.cuda.synchronize()
    g_traced = capture(True, traced=tev)
    replay_ms(g_traced, True)
    if h.get_error() != 0:
        raise RuntimeError("device error flags set during the traced steps")
    ms_traced = [a[0].elapsed_time(a[3]) for a in tev]
    ms_state = [a[0].elapsed_time(a[1]) for a in tev]
    ms_proj = [a[1].elapsed_time(a[2]) for a in tev]
    ms_topk = [a[2].elapsed_time(a[3]) for a in tev]
    m_list = counts.cpu().tolist()
    del g_traced
    pb = sum(proj_bytes(m, n, H) for m in m_list)
    sb = sum(step_bytes(m, n, H, V) for m in m_list)
    step_gbs = sb / (total_ms * 1e-3) / 1e9
    peak, peak_kind = load_peaks()
    ratio = ncu_traffic_per_byte()
    launches = h.step_launches
    if launches == 1:  # the whole step is one kernel: its bytes are the step's
        kb, kname = sb, "step_kernel (one-launch decode step: state update, gather, tcgen05 projection, top-k)"
    else:
        kb, kname = pb, "umma_step_kernel (fused gather + tcgen05 projection + top-k)"
    kern_gbs = kb / (sum(ms_proj) * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": kern_gbs, "peak": peak, "unit": "GB/s",
                "frac": kern_gbs / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                "traffic": (ratio * kb / K) if ratio is not None else None, "algorithmic_bytes_per_launch": kb / K,
                "launch_us": 1e3 * float(np.mean(ms_proj)),
                "timing": "CUDA events around each launch in a traced replay of the same steps"}

    # ---- end to end through the C ABI with host buffers ------------------------
    # ns_step_host: one call per step takes the step's inputs (tree ids, the
    # verify row, the draft hiddens) from pinned host memory and returns the
    # top-k ids and values there, all on the stream (the hiddens by a copy,
    # the rest read and written by the step kernel in place); the host then
    # waits for the stream.  A second, traced pass splits the time.
    init()
    tree_p = [torch.from_numpy(np.ascontiguousarray(trees_h[u])).pin_memory() for u in range(T)]
    ver_p = [torch.from_numpy(np.ascontiguousarray(verify_h[u][vrows[u]])).pin_memory() for u in range(T)]
    hid_p = [torch.from_numpy(np.ascontiguousarray(hid_h[u]).view(np.int16)).pin_memory() for u in range(T)]
    ids_p = torch.empty((n, k), dtype=torch.int32).pin_memory()
    vals_p = torch.empty((n, k), dtype=torch.float32).pin_memory()
    h2d = n * 4 + V * 4 + n * H * 2
    d2h = 2 * n * k * 4

    def host_step(t):
        u = t % T
        h.step_host(0, tree_p[u], ver_p[u], W_d, hid_p[u], k, ids_p, vals_p, stream=stream)

    for t in range(args.warmup):
        host_step(t)
    torch.cuda.synchronize()
    init()
    barrier()
    e2e_s = 0.0
    for t in range(K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        host_step(t)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    barrier()
    # where the time goes: the call's trace events around the input copies,
    # the step and the output copies, and the host time of the call
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    init()
    h.trace_events(evs)
    split = {"h2d_us": 0.0, "step_us": 0.0, "d2h_us": 0.0, "dispatch_us": 0.0}
    for t in range(K):
        flush.zero_()
        torch.cuda.synchronize()
        td = time.perf_counter()
        host_step(t)
        split["dispatch_us"] += 1e6 * (time.perf_counter() - td)
        stream.synchronize()
        split["h2d_us"] += 1e3 * evs[0].elapsed_time(evs[1])
        split["step_us"] += 1e3 * evs[1].elapsed_time(evs[2])
        split["d2h_us"] += 1e3 * evs[2].elapsed_time(evs[3])
    h.trace_events(None)
    if h.get_error() != 0:
        raise RuntimeError("device error flags set during the end-to-end steps")
    e2e_split = {key: v / K for key, v in split.items()}
    e2e_split["wall_us"] = 1e6 * e2e_s / K
    e2e_split["timing"] = ("wall time per step from the ns_step_host call to the stream's completion; the split "
                           "comes from a second pass with the call's trace events (each adds about a microsecond)")
    e2e_s = max_over_ranks(e2e_s)
    e2e = replicas.whole_job_rate(K, world, e2e_s)

    # ---- extras: the |I_t|~3k point and the dense heads ----------------------
    # Each is timed as (graph of R x [flush + op]) - (graph of R x [flush]).
    extra = {}
    if not args.no_extra:
        def graph_us(fn, reps=32):
            return graph_time_us(fn, flush, reps)

        # the slot-stable buffer: K steps of ns_step_slots (state update, slot
        # update + copy of the newly placed rows, projection over the slots;
        # one launch, as the slot table matches the window from slot_init on),
        # timed like the headline steps
        def slot_step(t):
            u = t % T
            h.step_slots(0, trees_d[u], verify_d[u], vrows[u], W_d, hid_d[u], k, logits=logits, ids=ids, vals=vals)

        def slot_graph(with_steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for t in range(K):
                    flush.zero_()
                    if with_steps:
                        slot_step(t)
            return g

        def slot_init():
            init()
            h.gather_new_head_rows(0, W_d)

        slot_init()
        for t in range(args.warmup):
            slot_step(t)
        torch.cuda.synchronize()
        gs, gf = slot_graph(True), slot_graph(False)
        sr = []
        for _ in range(3):
            slot_init()
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gs.replay()
            b.record()
            barrier()
            sr.append(a.elapsed_time(b) - replay_ms(gf, False))
        del gs, gf
        slot_init()
        _, smeta, _, _, _ = h.get_slots(0)
        copied = torch.zeros(K, dtype=torch.int32, device=dev)
        for t in range(K):
            slot_step(t)
            copied[t:t + 1].copy_(smeta[1:2])
        copied = copied.cpu().numpy()
        if h.get_error() != 0:
            raise RuntimeError("device error flags set during the slot-buffer steps")
        us_slot = 1e3 * sorted(sr)[1] / K
        extra["slot_step"] = {"us_per_step": us_slot, "one_launch": bool(h.step_slots_fused(0)),
                              "rows_copied_mean": float(copied.mean()),
                              "rows_copied_max": int(copied.max()), "mean_active": float(np.mean(m_list)),
                              "vs_full_repack_step": (1e3 * total_ms / K) / us_slot}

        init()
        torch.cuda.synchronize()
        m0 = int(cnt.item())
        # the sub-head step on the post-prefill window (|I_t| ~ W_max): build,
        # gather + projection + top-k; nothing is appended, so it repeats
        us0 = graph_us(lambda: (h.build_active_vocab(0),
                                h.gather_sub_lm_head_topk(0, W_d, hid_d[0], k, logits=logits, ids=ids, vals=vals)))
        b0 = step_bytes(m0, n, H, V) - V * 4  # no verify row in this sub-head step
        extra["pinned_point"] = {"active": m0, "us": us0, "frac_of_peak": b0 / (us0 * 1e-6) / 1e9 / peak}

        hid_bf = hid_d[0].view(torch.bfloat16)
        W_bf = W_d.view(torch.bfloat16)

        # the PyTorch way on the same |I_t|: index_select of the rows (a
        # packed copy), a cuBLAS GEMM and torch.topk (the ids stay indices
        # into I_t; the remap would be one more gather)
        idx_m = act[:m0].long()
        sel = torch.empty((m0, H), dtype=torch.bfloat16, device=dev)
        sub = torch.empty((n, m0), dtype=torch.bfloat16, device=dev)
        us_torch = graph_us(lambda: (torch.index_select(W_bf, 0, idx_m, out=sel),
                                     torch.matmul(hid_bf, sel.t(), out=sub), torch.topk(sub.float(), k, dim=1)))
        extra["pinned_point"]["torch_index_select_matmul_topk_us"] = us_torch
        # the indexed product (W_head rows through I_t, nothing packed: the
        # naive indexed GEMM of NanoSpec's ablation) on the same state
        init()
        extra["pinned_point"]["indexed_no_pack_us"] = graph_us(
            lambda: (h.build_active_vocab(0),
                     h.sub_lm_head_indexed_topk(0, W_d, hid_d[0], k, logits=logits, ids=ids, vals=vals)))

        # the vocabulary policies of NanoSpec's ablation, as decode steps
        # (timed like the headline: T2 steps from the initial state, graph
        # of steps minus graph of flushes): Ctx-only appends nothing after
        # the prefill, Ext-only starts from an empty stream
        def policy_us(init_fn, step_fn, T2=64):
            init_fn()
            for t in range(3):
                step_fn(t)
            torch.cuda.synchronize()
            gs = []
            for with_steps in (True, False):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for t in range(T2):
                        flush.zero_()
                        if with_steps:
                            step_fn(t)
                gs.append(g)
            ms = []
            for g in gs:
                init_fn()
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(b))
            return 1e3 * (ms[0] - ms[1]) / T2

        hc = ns.Handle(V, H, cfg.W_max, cfg.K_pre, 0, max_tree=n, max_k=k, max_prompt=len(prompt))
        try:
            def ctx_init():
                hc.stream_init(0, prompt_d, Z_d)
                hc.build_active_vocab(0)

            us_ctx = policy_us(ctx_init, lambda t: hc.step(0, None, None, 0, W_d, hid_d[t % T], k, logits=logits,
                                                           ids=ids, vals=vals))
        finally:
            hc.close()

        def ext_init():
            h.stream_init(0, None, None)
            h.build_active_vocab(0)

        us_ext = policy_us(ext_init, step)
        extra["policies"] = {"ctx_only_step_us": us_ctx, "ext_only_step_us": us_ext,
                             "ctx_plus_ext_step_us": 1e3 * total_ms / K,
                             "note": f"64 steps from the initial state each; the headline is the first {K} steps"}

        # an EAGLE-style draft phase on one step's I_t: D = 6 tree levels, each
        # a projection of its own hidden rows over the same I_t.  Four ways to
        # serve it, each a decode step (state update included) timed like the
        # policies: the slot buffer (copy the rows new to I_t, then D
        # projections over the slots); one full repack then D projections; D
        # fused repack + projection calls; D indexed products (nothing packed).
        depth = 6

        def level_hid(t, d):
            return hid_d[(t * depth + d) % T]

        def upd(t):
            u = t % T
            h.state_update(0, trees_d[u], verify_d[u], vrows[u])

        def dp_slots(t):
            upd(t)
            h.gather_new_head_rows(0, W_d)
            for d in range(depth):
                h.slot_lm_head_logits_topk(0, level_hid(t, d), k, logits=logits, ids=ids, vals=vals)

        def dp_slots_fused(t):
            # one ns_step_slots (a single launch while the table matches the
            # window: state and slot update, the new rows' copy, level 0's
            # projection), then the other levels over the slots
            u = t % T
            h.step_slots(0, trees_d[u], verify_d[u], vrows[u], W_d, level_hid(t, 0), k, logits=logits, ids=ids,
                         vals=vals)
            for d in range(1, depth):
                h.slot_lm_head_logits_topk(0, level_hid(t, d), k, logits=logits, ids=ids, vals=vals)

        def dp_one_repack(t):
            upd(t)
            h.gather_head_rows(0, W_d)
            for d in range(depth):
                h.sub_lm_head_logits_topk(0, level_hid(t, d), k, logits=logits, ids=ids, vals=vals)

        def dp_fused_each(t):
            upd(t)
            for d in range(depth):
                h.gather_sub_lm_head_topk(0, W_d, level_hid(t, d), k, logits=logits, ids=ids, vals=vals)

        def dp_indexed_each(t):
            upd(t)
            for d in range(depth):
                h.sub_lm_head_indexed_topk(0, W_d, level_hid(t, d), k, logits=logits, ids=ids, vals=vals)

        T3 = min(T, 32)
        extra["draft_phase"] = {
            "depth": depth,
            "slots_us": policy_us(slot_init, dp_slots, T3),
            "slots_one_launch_step_us": policy_us(slot_init, dp_slots_fused, T3),
            "one_repack_us": policy_us(init, dp_one_repack, T3),
            "fused_repack_each_us": policy_us(init, dp_fused_each, T3),
            "indexed_each_us": policy_us(init, dp_indexed_each, T3),
            "note": f"per decode step: state update + {depth} projections of n={n} rows with top-{k}, "
                    f"{T3} steps from the prefill state",
        }
        if h.get_error() != 0:
            raise RuntimeError("device error flags set during the draft-phase steps")

        # two-stream pipeline (MicroSpec §3.3): the gather of W_head[I_t, :] on
        # a copy stream while the draft backbone runs on the compute stream,
        # which waits for the gather only before the first projection.  The
        # backbone stands in for an EAGLE draft phase: `depth` levels, each one
        # Llama-3-8B-sized decoder layer whose weights (4 x H^2 + 3 x H x 14336
        # bf16, 436 MB) are read once by the n tree rows, then that level's
        # projection.  NanoSpec's 1.4 ms backbone is this on a GPU with about
        # a third of GB300's HBM bandwidth.  A second stand-in is
        # tensor-bound: four 2048^3 bf16 GEMMs before the first projection.
        copy_s = torch.cuda.Stream()
        n_layer = 4 * H + 3 * 14336
        W_layer = torch.empty((n_layer, H), dtype=torch.bfloat16, device=dev).normal_(0.0, 0.02)
        y_layer = torch.empty((n, n_layer), dtype=torch.bfloat16, device=dev)
        xs = torch.empty((2048, 2048), dtype=torch.bfloat16, device=dev).normal_()
        ys = torch.empty((2048, 2048), dtype=torch.bfloat16, device=dev)

        def layer():
            torch.matmul(hid_bf, W_layer.t(), out=y_layer)

        def square():
            for _ in range(4):
                torch.matmul(xs, xs, out=ys)

        def gather():
            h.gather_head_rows(0, W_d, copy_stream=torch.cuda.current_stream())

        def project(d=0):
            h.sub_lm_head_logits_topk(0, hid_d[d % T], k, logits=logits, ids=ids, vals=vals)

        def eagle_serial():
            gather()
            for d in range(depth):
                layer()
                project(d)

        def eagle_overlapped():
            cur = torch.cuda.current_stream()
            copy_s.wait_stream(cur)
            h.gather_head_rows(0, W_d, copy_stream=copy_s)
            for d in range(depth):
                layer()
                if d == 0:
                    cur.wait_stream(copy_s)
                project(d)

        def square_serial():
            square()
            gather()
            project()

        def square_overlapped():
            cur = torch.cuda.current_stream()
            copy_s.wait_stream(cur)
            h.gather_head_rows(0, W_d, copy_stream=copy_s)
            square()
            cur.wait_stream(copy_s)
            project()

        init()
        h.build_active_vocab(0)
        us_project = graph_us(project)
        us_layer = graph_us(layer)
        us_sq = graph_us(square)
        ov = {"active": m0, "project_us": us_project, "layer_us": us_layer, "depth": depth,
              "eagle_backbone_us": depth * us_layer, "square_gemms_us": us_sq, "by_copy_ctas": {}}
        for ctas in (0, 152, 38, 16):
            h.set_copy_ctas(ctas)
            us_gather = graph_us(gather)
            e_ser, e_ov = graph_us(eagle_serial), graph_us(eagle_overlapped)
            s_ser, s_ov = graph_us(square_serial), graph_us(square_overlapped)
            ov["by_copy_ctas"][str(ctas) if ctas else "default"] = {
                "gather_us": us_gather,
                "eagle_serial_us": e_ser, "eagle_overlapped_us": e_ov,
                "eagle_gather_hidden_frac": (e_ser - e_ov) / us_gather,
                "square_serial_us": s_ser, "square_overlapped_us": s_ov,
                "square_gather_hidden_frac": (s_ser - s_ov) / us_gather}
        h.set_copy_ctas(0)
        extra["copy_stream_overlap"] = ov
        del W_layer, y_layer, xs, ys
        dense_out = torch.empty((n, V), dtype=torch.bfloat16, device=dev)
        dense_logits = torch.empty((n, V), dtype=torch.float32, device=dev)
        us_cublas = graph_us(lambda: torch.matmul(hid_bf, W_bf.t(), out=dense_out))
        us_dense = graph_us(lambda: h.dense_lm_head_topk(W_d, V, hid_d[0], k, logits=dense_logits, ids=ids,
                                                         vals=vals))
        us_static = graph_us(lambda: h.dense_lm_head_topk(W_d, 32768, hid_d[0], k, logits=dense_logits, ids=ids,
                                                          vals=vals))
        extra["dense_head"] = {"cublas_matmul_us": us_cublas, "ours_dense_topk_us": us_dense,
                               "ours_static32768_topk_us": us_static,
                               "speedup_step_vs_cublas_dense": us_cublas / (1e3 * total_ms / K),
                               "speedup_pinned_point_vs_cublas_dense": us_cublas / us0}
    if not args.no_extra and not args.no_workloads:
        torch.cuda.empty_cache()
        extra["workloads"] = run_workloads(ns, dev, flush, args.warmup, args.workload_steps)
    clock = clocks.stop()

    # ---- the CPU oracle on a bounded sample (rank 0, one GPU) ----------------
    cpu = None
    if rank == 0 and world == 1:
        done, dt = time_oracle(cfg, wl, T, budget_s=args.cpu_seconds)
        cpu = {"value": done / dt, "unit": "steps/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"first {done} decode steps of {cfg.name} after its prefill init (prefill not timed)",
               "single_thread": single_thread_oracle(cfg.name, steps=16)}

    if rank == 0:
        mean_m = float(np.mean(m_list))
        line = {
            "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_ms / K, "us_per_step": 1e3 * total_ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "V": V, "H": H, "W_max": cfg.W_max, "K_pre": cfg.K_pre,
                       "K_ver": cfg.K_ver, "n_tree": n, "k": k, "decode_steps_per_pass": T,
                       "l2": "flushed before every timed step (256 MiB write); the flush-only graph's time "
                             "is subtracted",
                       "timing": "graph of K x (flush + step) minus graph of K x flush, median of 3",
                       "mean_active": mean_m, "min_active": int(min(m_list)), "max_active": int(max(m_list)),
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline,
            "step_roofline": {"achieved": step_gbs, "frac": step_gbs / peak,
                              "bytes_per_step": sb / K},
            "kernel_us": ({"step_kernel": 1e3 * float(np.mean(ms_proj)),
                           "traced_step": 1e3 * float(np.mean(ms_traced)),
                           "timing": "traced replay: events around the one step kernel"} if launches == 1 else
                          {"state_update": 1e3 * float(np.mean(ms_state)),
                           "gather_project_topk": 1e3 * float(np.mean(ms_proj)),
                           "trace_gap": 1e3 * float(np.mean(ms_topk)),
                           "traced_step": 1e3 * float(np.mean(ms_traced)),
                           "timing": "traced replay: events around each kernel, no programmatic overlap"}),
            "step_launches": launches,
            "init_ms": init_ms,
            "e2e": {"value": e2e, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "split_us_per_step": e2e_split},
            "gpu_launches": launches * K,
            "clocks": clock,
            "cpu_baseline": cpu,
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
