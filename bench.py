"""Benchmark of one MLA decode step on the DeepSeek-V2-shaped layer (batch 64, context 8192).

A step is one pass of the whole decode path over one batch: append the new
token's latent row, project and absorb its query, attend over the paged latent
cache (with the split-KV merge), and apply the value and output projections.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line.  `value` is cached tokens attended per second over the
whole job (sum over sequences of the attended length, times ranks, divided by
the device time of a step).  Several GPUs run independent replicas (each rank
its own batch; no collective on the data path).  `--impl reference` times the
float64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import mla_inputs as I  # noqa: E402

METRIC = "MLA decode cached-tokens/s and achieved HBM GB/s (% roofline), b64 ctx8192"
UNIT = "cached tokens/s"
DEFAULT_WORKLOAD = "dsv2_b64_ctx8192"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")
DECODE_SOURCES = ["mla_latent_kv_81_b300/csrc/mla_decode_tc.cu", "mla_latent_kv_81_b300/csrc/mla_sm100.cuh"]


# ------------------------------------------------------------------ algorithmic work
def decode_algorithmic(p: I.Problem) -> dict:
    """Bytes and FLOPs mla_decode_attention must move / perform for one step.

    Per attended (token, query): the cached row once per sequence ((d_c + d_rope)
    * elem bytes, read once for all heads and both queries), and
    2 * H * (d_c + d_rope + d_c) FLOPs (scores over the full row, weighted sum
    over the latent).  Per query row: q read and o_lat written.  Block table:
    4 B per 64-token block.  A reduced-precision cache row is d_c + 2 d_rope + 4
    bytes (codes, bf16 key divided by the scale, fp32 scale)."""
    d = p.dims
    eb = 2 if p.w.dtype == "bf16" else 4
    kv = p.kv_len.astype(np.int64)
    n_q = p.w.n_q
    rows = int(kv.sum())
    vis = int(sum(max(0, int(k) - (n_q - 1 - j)) for k in kv for j in range(n_q)))
    row_bytes = d.d_c + 2 * d.d_rope + 4 if getattr(p.w, "cache_fp8", False) else d.row * eb
    latent_bytes = rows * row_bytes
    q_bytes = p.w.batch * n_q * d.n_heads * d.row * eb
    o_bytes = p.w.batch * n_q * d.n_heads * d.d_c * eb
    table_bytes = int(sum((int(k) + d.block_size - 1) // d.block_size for k in kv)) * 4
    flops = 2 * d.n_heads * (d.row + d.d_c) * vis
    return dict(bytes=latent_bytes + q_bytes + o_bytes + table_bytes, latent_bytes=latent_bytes, flops=flops,
                cached_tokens=rows)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        path = os.path.join(ROOT, rel)
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, or None when the
    decode sources changed since those counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("source_sha") != decode_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample_absorbed(p: I.Problem, budget_s: float):
    """Time the float64 oracle's absorbed form (query folded through W_UK, attention in latent space,
    all heads of one sequence per step) until `budget_s`.  Returns (cached tokens per second, steps)."""
    from oracle import mla_oracle as O
    d, W = p.dims, p.weights
    n_q, H = p.w.n_q, d.n_heads
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    done_tok, elapsed, steps, b = 0.0, 0.0, 0, 0
    while elapsed < budget_s:
        rows = I.draw_latent_rows(p.w, b, int(p.kv_len[b])).astype(np.float64)
        sl = slice(b * n_q, (b + 1) * n_q)
        t0 = time.perf_counter()
        q_nope, q_rope = O.project_query(p.x_q[sl], W["W_Q"], W["W_QR"], p.q_pos[sl], H, d.rope_base)
        q_abs = O.absorb_query(q_nope, W["W_UK"])
        O.attend_latent(q_abs, q_rope, rows[:, :d.d_c], rows[:, d.d_c:], int(p.kv_len[b]), scale)
        elapsed += time.perf_counter() - t0
        done_tok += float(p.kv_len[b])
        steps += 1
        b = (b + 1) % p.w.batch
    return done_tok / elapsed, steps


def oracle_sample(p: I.Problem, budget_s: float, heads_per_step: int | None = None, max_steps: int | None = None):
    """Time the float64 oracle (explicit form, as it stands) on whole heads of whole
    sequences of the workload until `budget_s` or `max_steps` is reached.
    Returns (cached-token equivalents per second, description, threads, step times)."""
    from oracle import mla_oracle as O
    d, W = p.dims, p.weights
    n_q = p.w.n_q
    H = d.n_heads
    hps = heads_per_step or H
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    done_tok, elapsed, steps, times = 0.0, 0.0, 0, []
    b, h0 = 0, 0
    rows_cache = {}
    while True:
        if b not in rows_cache:
            rows_cache.clear()
            rows = I.draw_latent_rows(p.w, b, int(p.kv_len[b])).astype(np.float64)
            rows_cache[b] = rows
        rows = rows_cache[b]
        sl = slice(b * n_q, (b + 1) * n_q)
        hs = slice(h0, min(H, h0 + hps))
        nh = hs.stop - hs.start
        t0 = time.perf_counter()
        q_nope, q_rope = O.project_query(p.x_q[sl], W["W_Q"].reshape(H, d.qk_nope, -1)[hs].reshape(nh * d.qk_nope, -1),
                                         W["W_QR"].reshape(H, d.d_rope, -1)[hs].reshape(nh * d.d_rope, -1),
                                         p.q_pos[sl], nh, d.rope_base)
        O.attend_explicit(q_nope, q_rope, rows[:, :d.d_c], rows[:, d.d_c:], W["W_UK"][hs], W["W_UV"][hs],
                          int(p.kv_len[b]), scale)
        dt = time.perf_counter() - t0
        times.append(dt)
        elapsed += dt
        done_tok += float(p.kv_len[b]) * nh / H
        steps += 1
        h0 += nh
        if h0 >= H:
            h0, b = 0, (b + 1) % p.w.batch
        if (max_steps is not None and steps >= max_steps) or (max_steps is None and elapsed >= budget_s):
            break
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or str(len(os.sched_getaffinity(0)))
    desc = (f"explicit-form oracle (float64, K/V rebuilt per head) over {steps} sample(s) of {hps} head(s) "
            f"of one sequence each; {done_tok:.0f} cached-token equivalents")
    return done_tok / elapsed, desc, threads, times


# ------------------------------------------------------------------ multi-rank arithmetic
def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(tokens_per_rank: float, world: int, ms_per_step: float) -> float:
    """Cached tokens attended per second by all ranks together (replicas: every rank does the same work)."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ main paths
def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    w = I.WORKLOADS[args.workload]
    p = I.make_problem(w)
    heads = 8
    oracle_sample(p, 0.0, heads_per_step=heads, max_steps=args.warmup)
    rate, desc, threads, times = oracle_sample(p, 0.0, heads_per_step=heads, max_steps=args.steps)
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(w, p), parallelism=parallelism(world)),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + f"; BLAS threads {threads}"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parallelism(world: int) -> str:
    return f"replicas x{world}" if world > 1 else "single GPU"


def workload_config(w: I.Workload, p: I.Problem) -> dict:
    d = w.dims
    return {"workload": w.name, "batch": w.batch, "ctx": int(p.kv_len.max()), "ctx_min": int(p.kv_len.min()),
            "n_q": w.n_q, "n_heads": d.n_heads, "d_c": d.d_c, "d_rope": d.d_rope, "d_model": d.d_model,
            "qk_nope": d.qk_nope, "v_head": d.v_head, "block_size": d.block_size, "paged": "shuffled block table",
            "l2": "inputs larger than L2 (latent cache and weights each exceed 126 MB; no flush)",
            "step": "append new token + absorb query + decode attention (+split-KV merge) + output projection",
            "timing": "step replayed as three CUDA graphs; e2e uses the plain API with host buffers"}


def run_ours(args, rank: int, world: int):
    import torch
    import mla_harness as Hn
    import mla_latent_kv_81_b300 as M

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    w = I.WORKLOADS[args.workload]
    p = I.make_problem(w)
    L = Hn.DeviceLayer(p)
    L.fill()
    # the step rewrites the appended rows in place, so every step sees the same cache
    stream = torch.cuda.current_stream()
    alg = decode_algorithmic(p)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        L.step(with_lse=False)
    code, flags = L.status()
    if code != 0:
        raise RuntimeError(f"device status after warm-up: {M.mla_status_string(code)} ({flags})")

    # ---- the step as three CUDA graphs (projections before attention, attention, output projection),
    #      replayed back to back; the attention graph is bracketed by events for its own duration
    def pre():
        n = L.x_q.shape[0]
        if p.w.n_append:
            M.mla_compress_append(L.cfg, L.x_q, L.W["W_DKV"], L.W["W_KR"], L.app_seq, L.app_pos, L.rope, L.cache,
                                  ws=L._ws("c", M.mla_compress_workspace_bytes(L.cfg, n)))
        M.mla_absorb_query(L.cfg, L.x_q, L.W["W_Q"], L.W["W_QR"], L.W["W_UK"], L.q_pos, L.rope, L.q,
                           ws=L._ws("a", M.mla_absorb_workspace_bytes(L.cfg, n)))

    def post():
        M.mla_output_project(L.cfg, L.o_lat, L.W["W_UV"], L.W["W_O"], L.out,
                             ws=L._ws("o", M.mla_output_workspace_bytes(L.cfg, L.x_q.shape[0])))

    graphs = []
    launches_per_step = 0
    for fn in (pre, lambda: L.attend(with_lse=False), post):
        g = torch.cuda.CUDAGraph()
        l0 = M.mla_kernel_launches()
        with torch.cuda.graph(g):
            fn()
        launches_per_step += M.mla_kernel_launches() - l0
        graphs.append(g)
    g_pre, g_dec, g_post = graphs
    for _ in range(3):
        g_pre.replay(); g_dec.replay(); g_post.replay()
    torch.cuda.synchronize()

    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.2)
    t_start.record(stream)
    for i in range(args.steps):
        g_pre.replay()
        ev_dec[i][0].record(stream)
        g_dec.replay()
        ev_dec[i][1].record(stream)
        g_post.replay()
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    launches = launches_per_step * args.steps
    ms_total = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) for a, b in ev_dec]
    ms_total, dec_mean = max_over_ranks([ms_total, statistics.mean(dec_ms)], dist, "cuda")
    ms_step = ms_total / args.steps
    tokens = alg["cached_tokens"] * world
    value = whole_job_rate(alg["cached_tokens"], world, ms_step)

    # ---- end to end through the public API from pinned host buffers
    x_host = L.x_q.cpu().pin_memory()
    out_host = torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory()
    x_dev = torch.empty_like(L.x_q)
    h2d = x_host.numel() * x_host.element_size()
    d2h = out_host.numel() * out_host.element_size()
    e2e_steps = max(100, min(args.steps, 500))

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        L.step(x_q=x_dev, with_lse=False)
        out_host.copy_(L.out, non_blocking=True)

    def drain():
        # wait for the queued steps by polling an event: a blocking synchronize leaves the host idle
        ev = torch.cuda.Event()
        ev.record(stream)
        while not ev.query():
            pass

    # Warm-up: at least 3 steps and 0.3 s of continuous host work.  An idle host CPU clocks down and
    # needs some 0.1-0.2 s of load to come back; until then each step's Python and library calls take
    # ~430 us instead of ~160 us and the loop is host-bound.  A serving loop keeps the host busy.
    n_warm, t_warm = 0, time.perf_counter()
    while n_warm < 3 or time.perf_counter() - t_warm < 0.3:
        e2e_step()
        n_warm += 1
    drain()
    if dist is not None:
        dist.barrier()
        drain()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    host_us = (time.perf_counter() - h0) / e2e_steps * 1e6
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], dist, "cuda")[0]
    code, flags = L.status()
    if code != 0:
        raise RuntimeError(f"device status after timing: {M.mla_status_string(code)} ({flags})")

    hbm_peak, tf_peak, peak_kind = load_peaks()
    achieved = alg["bytes"] / (dec_mean * 1e-3) / 1e9
    flops_time = alg["flops"] / (tf_peak * 1e12)
    bytes_time = alg["bytes"] / (hbm_peak * 1e9)
    bound = "hbm" if bytes_time >= flops_time else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak}
    else:
        ach_tf = alg["flops"] / (dec_mean * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach_tf, "peak": tf_peak, "unit": "TFLOP/s", "frac": ach_tf / tf_peak}
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    roof["traffic"] = recorded_traffic(w.name)
    roof["kernel"] = ("mla_decode_attention (attention and split-KV merge launches, replayed as one CUDA "
                      "graph), CUDA events on its stream")
    roof["ms_per_launch"] = dec_mean
    roof["algorithmic_bytes_per_launch"] = alg["bytes"]
    roof["algorithmic_flops_per_launch"] = alg["flops"]

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": p.w.dtype, "data": "synthetic (seeded Gaussian activations, weights, latents)",
        "config": dict(workload_config(w, p), parallelism=parallelism(world)),
        "roofline": roof, "clocks": clk,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "host_enqueue_us_per_step": host_us, "warmup_steps": n_warm,
                "path": "plain API calls (no graph), pinned host input copied in and output copied out every step"},
        "gpu_launches": int(launches),
    }
    if not args.no_cpu_baseline:
        rate, desc, threads, _ = oracle_sample(p, args.cpu_budget, heads_per_step=8)
        abs_rate, abs_steps = oracle_sample_absorbed(p, max(1.0, args.cpu_budget / 3))
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": desc + f"; BLAS threads {threads}",
                                "absorbed": {"value": abs_rate, "unit": UNIT,
                                             "sample": f"absorbed-form oracle (float64, all heads) over {abs_steps} "
                                                       f"whole sequence(s)"}}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_sweep(args):
    """One JSON line per workload: the decode call (attention + merge) as the median of
    `--sweep-reps` runs with L2 flushed before each (a 256 MB write outside the timed region), its
    cached tokens/s, algorithmic GB/s and roofline fraction, and the projection calls timed the same way."""
    import torch
    import mla_harness as Hn
    import mla_latent_kv_81_b300 as M

    hbm_peak, tf_peak, peak_kind = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timed(fn, reps):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    for name, w in I.WORKLOADS.items():
        p = I.make_problem(w)
        L = Hn.DeviceLayer(p)
        L.fill()
        L.step(with_lse=False)
        n = L.x_q.shape[0]
        alg = decode_algorithmic(p)
        t_dec = timed(lambda: L.attend(with_lse=False), args.sweep_reps)
        proj = {}
        if p.w.n_append:
            wsc = L._ws("c", M.mla_compress_workspace_bytes(L.cfg, n))
            proj["compress_append"] = timed(lambda: M.mla_compress_append(
                L.cfg, L.x_q, L.W["W_DKV"], L.W["W_KR"], L.app_seq, L.app_pos, L.rope, L.cache, ws=wsc), args.sweep_reps)
        wsa = L._ws("a", M.mla_absorb_workspace_bytes(L.cfg, n))
        proj["absorb_query"] = timed(lambda: M.mla_absorb_query(
            L.cfg, L.x_q, L.W["W_Q"], L.W["W_QR"], L.W["W_UK"], L.q_pos, L.rope, L.q, ws=wsa), args.sweep_reps)
        wso = L._ws("o", M.mla_output_workspace_bytes(L.cfg, n))
        proj["output_project"] = timed(lambda: M.mla_output_project(
            L.cfg, L.o_lat, L.W["W_UV"], L.W["W_O"], L.out, ws=wso), args.sweep_reps)
        code, flags = L.status()
        if code != 0:
            raise RuntimeError(f"{name}: device status {M.mla_status_string(code)} ({flags})")
        t_roof = max(alg["bytes"] / (hbm_peak * 1e9), alg["flops"] / (tf_peak * 1e12))
        bound = "hbm" if alg["bytes"] / (hbm_peak * 1e9) >= alg["flops"] / (tf_peak * 1e12) else "tensor"
        print(json.dumps({
            "sweep": name, "dtype": w.dtype, "config": workload_config(w, p), "decode_ms": t_dec,
            "cached_tokens_per_s": alg["cached_tokens"] / (t_dec * 1e-3),
            "achieved_gbs": alg["bytes"] / (t_dec * 1e-3) / 1e9,
            "achieved_tflops": alg["flops"] / (t_dec * 1e-3) / 1e12,
            "roofline": {"bound": bound, "t_roof_ms": t_roof * 1e3, "frac": t_roof / (t_dec * 1e-3),
                         "peaks": f"{peak_kind}: {hbm_peak} GB/s, {tf_peak} TFLOP/s bf16"},
            "projections_ms": proj, "timing": f"median of {args.sweep_reps}, L2 flushed (256 MB write) before each"}),
            flush=True)
        del L
        torch.cuda.empty_cache()


def prefill_algorithmic(c: I.PrefillCase) -> dict:
    """Work of one mla_prefill_attention call in the explicit form: the per-head keys and values rebuilt
    for every cached token (2 d_c (qk_nope + v_head) FLOP per token and head), and for every (query,
    visible key, head) 2 (qk_nope + d_rope) FLOP of score and 2 v_head of P V.  Bytes: the latent rows,
    the up-projections, the queries and the outputs."""
    d = c.dims
    H, L, T = d.n_heads, c.prompt, c.queries
    pairs = sum(L - T + j + 1 for j in range(T))
    flops = 2.0 * L * d.d_c * H * (d.qk_nope + d.v_head) + 2.0 * pairs * H * (d.qk_nope + d.d_rope + d.v_head)
    row = d.d_c + (H if c.rope_per_head else 1) * d.d_rope
    nbytes = 2.0 * (L * row + H * (d.qk_nope + d.v_head) * d.d_c + T * H * (d.qk_nope + d.d_rope) + T * H * d.v_head)
    return {"flops": flops, "bytes": nbytes, "pairs": pairs}


def run_prefill(args):
    """One JSON line per prefill case: the explicit-form attention call (latent gather, K/V GEMM,
    attention kernel) as the median of `--sweep-reps` runs with L2 flushed before each, its TFLOP/s and
    the fraction of the tensor roofline."""
    import torch
    import mla_harness as Hn

    hbm_peak, tf_peak, peak_kind = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for name in args.prefill_cases.split(","):
        c = I.PREFILL_CASES[name]
        p = I.make_prefill(c)
        L = Hn.PrefillLayer(p)
        L.fill()
        for _ in range(3):
            L.attend(with_lse=False)
        ts = []
        for _ in range(args.sweep_reps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            L.attend(with_lse=False)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        code, flags = L.status()
        if code != 0:
            raise RuntimeError(f"{name}: device status {code} ({flags})")
        t = statistics.median(ts)
        alg = prefill_algorithmic(c)
        t_tc, t_hbm = alg["flops"] / (tf_peak * 1e12), alg["bytes"] / (hbm_peak * 1e9)
        print(json.dumps({
            "prefill": name, "dtype": c.dtype, "prompt": c.prompt, "queries": c.queries, "call_ms": t,
            "achieved_tflops": alg["flops"] / (t * 1e-3) / 1e12,
            "roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "t_roof_ms": max(t_tc, t_hbm) * 1e3,
                         "frac": max(t_tc, t_hbm) / (t * 1e-3),
                         "peaks": f"{peak_kind}: {hbm_peak} GB/s, {tf_peak} TFLOP/s bf16"},
            "algorithmic_flops": alg["flops"], "algorithmic_bytes": alg["bytes"],
            "timing": f"median of {args.sweep_reps}, L2 flushed (256 MB write) before each"}), flush=True)
        del L
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the step benchmark, one JSON line per workload (decode call and projections)")
    ap.add_argument("--sweep-reps", type=int, default=50)
    ap.add_argument("--prefill", action="store_true",
                    help="instead of the step benchmark, one JSON line per prefill case (explicit-form attention)")
    ap.add_argument("--prefill-cases", default="prefill_dsv2_L4096_T4096,prefill_dsv2_L8192_T8192,prefill_dsv2_L4096_T4096_rh")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.sweep:
        if rank == 0:
            run_sweep(args)
    elif args.prefill:
        if rank == 0:
            run_prefill(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
