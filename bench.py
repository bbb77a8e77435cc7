#!/usr/bin/env python3
"""Decode throughput of the quantized MoE OCR decoder on one GB300.

Headline workload (one "step" = one decode step of every row through the
whole path: embedding, 12 layers of RMSNorm/QKV/RoPE/KV append/attention/
O-proj and the dense MLP or router + experts + combine, final norm, LM head,
argmax): the throughput stress configuration, i.e. the 12-layer
DeepSeek-V2-style decoder (hidden 1280, 10x128 heads, layer 0 dense MLP 3584,
layers 1-11 with 64 routed top-6 experts + 2 shared of 896, fp16 LM head over
102400 tokens) at 64 rows with 2048 cached prefix tokens per row plus the
128-slot ring, all experts Q4_0, greedy decoding.  Weights, cache and first
ids are seeded synthetic data (seed 4).

The same line carries the full decoder at 8 rows and at 1 row (256 image
embeddings + 32 prompt ids per row, built by uocr_prefill), the per-kernel
table with the dominant kernel's roofline, the end-to-end host-buffer figure
and the float64 oracle timed on the host cores (all threads, and 6 threads).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-side-configs] [--no-cpu-baseline] [--sweep]

Prints one JSON line on rank 0.
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

_CORES = os.cpu_count() or 1
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_moe_decode_gb300 import synth  # noqa: E402

METRIC = "decode tokens/s (rows x steps/s) and achieved HBM GB/s vs GB300 peak, 1 GPU"
WORKLOAD = "stress_b64"
HEADLINE_CONFIG = {
    "workload": "throughput stress: full 12-layer MoE decoder (hidden 1280, 10x128 heads, layer 0 dense MLP 3584, "
                "layers 1-11 64 routed top-6 + 2 shared experts of 896, vocab 102400 fp16 LM head), 64 rows, "
                "2048 cached prefix tokens + 128-slot ring, all experts Q4_0, Q8_0 attention/dense, greedy",
    "rows": 64, "prefix": 2048, "ring": 128, "seed": 4}
BPW = {synth.F16: 2.0, synth.Q8_0: 34 / 32, synth.Q4_0: 18 / 32, synth.I8ASYM: 36 / 32, synth.Q8_0_G64: 66 / 64,
       synth.Q4_0_G64: 34 / 64}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ algorithmic bytes
def class_bytes(cfg, rows, positions, distinct):
    """Bytes the method must move per launch of each kernel class in one step.

    Weights touched (canonical block bytes: Q8_0 34/32, Q4_0 18/32 B per
    weight, fp16 2 B), KV read/written, and the activation vectors each class
    reads or writes.  distinct[l] = experts that received a token at layer l.
    """
    H, S, V, L = cfg.hidden, cfg.n_heads * cfg.head_dim, cfg.vocab, cfg.n_layers
    P, R = cfg.prefix_len, cfg.ring_len
    act = rows * H * 4
    out = {}
    out["embed"] = [rows * H * 2 + act]
    # bytes of one cache slot of one row and layer (keys and values): fp16, or
    # INT8 codes plus one fp32 scale per head
    slot = 2 * (S + 4 * cfg.n_heads) if getattr(cfg, "kv_int8", 0) else 2 * S * 2
    if getattr(cfg, "kv_int8", 0):
        out["qkv"] = [3 * S * H * BPW[cfg.fmt_attn] + act + rows * S * (4 + 2 * 4)] * L
        out["kv_quant"] = [rows * (2 * S * 4 + slot)] * L
    else:
        out["qkv"] = [3 * S * H * BPW[cfg.fmt_attn] + act + rows * S * (4 + 2 * 2)] * L
    kv = 0
    for p in positions:
        n_valid = p + 1 if p < P else P + min(p - P + 1, R)
        kv += n_valid * slot
    out["attention"] = [kv + rows * S * (4 + 2)] * L
    out["o_proj"] = [H * S * BPW[cfg.fmt_attn] + rows * S * 2 + 2 * act] * L
    Ie, Ish = cfg.expert_inter, cfg.n_shared * cfg.expert_inter
    for l in range(L):
        if cfg.is_dense(l):
            I = cfg.dense_inter
            out.setdefault("mlp_gate_up", []).append(2 * I * H * BPW[cfg.fmt_dense] + act + rows * I * 2)
            out.setdefault("mlp_down", []).append(H * I * BPW[cfg.fmt_dense] + rows * I * 2 + 2 * act)
        else:
            U = distinct[l]
            out.setdefault("router", []).append(cfg.n_experts * H * 2 + act + rows * H * 2)
            out.setdefault("expert_gate_up", []).append(
                U * 2 * Ie * H * BPW[cfg.fmt_routed] + 2 * Ish * H * BPW[cfg.fmt_shared]
                + rows * H * 2 + rows * (cfg.top_k * Ie + Ish) * 2)
            out.setdefault("expert_down", []).append(
                U * H * Ie * BPW[cfg.fmt_routed] + H * Ish * BPW[cfg.fmt_shared]
                + rows * (cfg.top_k * Ie + Ish) * 2 + rows * (cfg.top_k + 1) * H * 4)
            # residual + k weighted partials + the shared partial in, the layer output out
            out.setdefault("expert_combine", []).append(rows * (cfg.top_k + 2) * H * 4 + rows * cfg.top_k * 4
                                                        + act)
    if V:
        out["lm_head_argmax"] = [V * H * 2 + act + rows * 8]
    return out


def sources_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_moe_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_class):
    """DRAM bytes per launch of a kernel class from the committed ncu summary,
    valid only while the kernel sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = sources_sha()
    for line in open(p):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("class") == kernel_class and f.get("sources_sha") == sha:
            return float(f["dram_bytes_per_launch"])
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU / reference arm
ORACLE_ROWS = 2  # rows of the headline workload the oracle steps through in its timed sample


def time_oracle(wl, rows, min_s, max_steps, warm=2):
    """Oracle decode steps of the workload's first `rows` rows, from its own
    starting state (cached prefix, or the prefix embeddings' positions), LM
    head included; returns (steps, seconds).  Weight dequantisation is cached
    on the warm-up steps."""
    import oracle

    kv = None if wl.kv_prefix is None else wl.kv_prefix.subset(list(range(rows)))
    m = oracle.OracleModel(wl.cfg, wl.tensors, rows, kv_prefix=kv, sinks=wl.sinks, cache="float64")
    if wl.prefill_embeds is not None:  # positions of the prefix, embedding inputs
        step = lambda p: m.step(np.full(rows, p, np.int32), x=wl.prefill_embeds[:rows, p])
        p0 = 0
    else:  # greedy decoding from the cached prefix
        ids = [wl.first_ids[:rows].copy()]

        def step(p):
            r = m.step(np.full(rows, p, np.int32), ids=ids[0])
            ids[0] = r.next_ids.astype(np.int32)
        p0 = wl.start_pos
    for p in range(warm):
        step(p0 + p)
    t0 = time.perf_counter()
    n = 0
    while n < max_steps and (time.perf_counter() - t0) < min_s:
        step(p0 + warm + n)
        n += 1
    return n, time.perf_counter() - t0


def cpu_sample_desc(rows, n, warm, cores):
    return (f"{rows} rows x {n} greedy decode steps of the 64-row stress workload from its 2048-token cached "
            f"prefix (float64 NumPy oracle on {cores} host threads, weight dequantisation cached on {warm} "
            f"warm-up steps)")


def cpu_baseline_threads(threads, min_s=15.0, max_steps=20):
    """The oracle sample in a child process whose BLAS / OpenMP pools have `threads` threads."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(min_s), str(max_steps)],
                       env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": ORACLE_ROWS * d["steps"] / d["seconds"], "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "sample": cpu_sample_desc(ORACLE_ROWS, d["steps"], 2, threads)}


def run_cpu_sample(min_s, max_steps):
    wl = synth.workload(WORKLOAD, steps=0)
    n, dt = time_oracle(wl, ORACLE_ROWS, min_s=min_s, max_steps=max_steps)
    print(json.dumps({"steps": n, "seconds": dt}), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = synth.workload(WORKLOAD, steps=0)
    K, W = args.steps, args.warmup
    n, dt = time_oracle(wl, ORACLE_ROWS, min_s=90.0, max_steps=min(K, 40), warm=max(min(W, 3), 2))
    v = ORACLE_ROWS * n / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": n, "steps_requested": K, "warmup": W, "ms_per_step": 1e3 * dt / max(n, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(HEADLINE_CONFIG, oracle_rows=ORACLE_ROWS),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
                             "sample": cpu_sample_desc(ORACLE_ROWS, n, max(min(W, 3), 2), _CORES) +
                             ", capped at 90 s"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ replicas
# With N GPUs the path runs as N independent replicas (rows need no exchange):
# every rank times its own steps, the job's time is the slowest rank's, and
# the job processed world x rows x steps tokens in it.
def max_over_ranks(x, dist, device):
    """The maximum of a per-rank float over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, rows, steps, seconds):
    """Whole-job tokens/s of `world` replicas of `rows` rows over `steps` steps."""
    return world * rows * steps / seconds


# ------------------------------------------------------------------ our arm
def open_workload(name, dev, stream, cfg_overrides=None, **kw):
    """Context with the workload loaded and its prefix in the cache (cached
    prefixes written, image + prompt prefixes built by uocr_prefill).  Returns
    (ctx, wl, first ids on the device, prefill seconds or None)."""
    import torch

    from quantized_moe_decode_gb300 import binding

    wl = synth.workload(name, steps=0, **kw)
    if cfg_overrides:
        wl.cfg = wl.cfg.replace(**cfg_overrides)
    cfg, rows = wl.cfg, wl.rows
    ctx = binding.Context(cfg, max_rows=rows, stream=stream.cuda_stream, device=dev.index or 0)
    binding.load_workload(ctx, wl)
    ids = torch.zeros(rows, dtype=torch.int32, device=dev)
    if not cfg.vocab:  # hidden-vector inputs: nothing to prefill, no ids
        return ctx, wl, ids, None
    t_pre = None
    if wl.prefill_embeds is not None:
        ne = wl.prefill_embeds.shape[1]
        emb = torch.from_numpy(np.ascontiguousarray(wl.prefill_embeds).view(np.int16)).to(dev)
        pids = torch.from_numpy(np.ascontiguousarray(wl.prefill_ids)).to(dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for r in range(rows):
            ctx.uocr_prefill(r, ne, 0, x_ptr=emb[r].data_ptr())
            ctx.uocr_prefill(r, cfg.prefix_len - ne, ne, ids_ptr=pids[r].data_ptr(), next_ptr=ids[r:].data_ptr())
        ctx.uocr_sync()
        t_pre = time.perf_counter() - t0
    else:
        ids.copy_(torch.from_numpy(wl.first_ids))
    return ctx, wl, ids, t_pre


def time_greedy(ctx, wl, ids, dev, stream, K, W, dist=None):
    """W untimed then K timed greedy steps chained on the device (one graph
    replay per step), CUDA events on the caller's stream.  Returns (ms, first
    timed position, last ids).  Workloads without a vocabulary take a resident
    hidden vector per step instead (uocr_decode_step_embeds)."""
    import torch

    rows, start = wl.rows, wl.start_pos
    if not wl.cfg.vocab:
        n = W + K
        xs = np.resize(np.ascontiguousarray(wl.step_x), (n, rows, wl.cfg.hidden)).astype(np.float16)
        x_all = torch.from_numpy(xs.view(np.int16)).to(dev)
        pos_all = torch.tensor([[start + s] * rows for s in range(n)], dtype=torch.int32, device=dev)
        for s_ in range(W):
            ctx.uocr_decode_step_embeds(rows, x_all[s_].data_ptr(), pos_all[s_].data_ptr())
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e0.record(stream)
        for s_ in range(W, n):
            ctx.uocr_decode_step_embeds(rows, x_all[s_].data_ptr(), pos_all[s_].data_ptr())
        e1.record(stream)
        torch.cuda.synchronize()
        ctx.uocr_sync()
        return e0.elapsed_time(e1), start + W, x_all[n - 1].clone()
    out = torch.zeros((max(K, W, 1), rows), dtype=torch.int32, device=dev)
    pos = torch.full((rows,), start, dtype=torch.int32, device=dev)
    if W:
        ctx.uocr_generate(rows, ids.data_ptr(), pos.data_ptr(), W, out.data_ptr())
        ctx.uocr_sync()
        ids = out[W - 1].clone()
    pos.fill_(start + W)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    ctx.uocr_generate(rows, ids.data_ptr(), pos.data_ptr(), K, out.data_ptr())
    e1.record(stream)
    torch.cuda.synchronize()
    ctx.uocr_sync()
    return e0.elapsed_time(e1), start + W, out[K - 1].clone()


def kernel_table(ctx, wl, ids, dev, position):
    """Per kernel class: its launches of one step replayed alone in a graph
    (uocr_profile, CUDA events on the library stream), algorithmic bytes, GB/s."""
    import torch

    cfg, rows = wl.cfg, wl.rows
    pos = torch.full((rows,), position, dtype=torch.int32, device=dev)
    prof = {}
    n_prof = 3
    for _ in range(n_prof):
        if cfg.vocab:
            t = ctx.uocr_profile(rows, 0, ids.data_ptr(), 0, pos.data_ptr())
        else:  # `ids` holds the last hidden vectors
            t = ctx.uocr_profile(rows, 1, 0, ids.data_ptr(), pos.data_ptr())
        for k_, v_ in t.items():
            prof[k_] = prof.get(k_, 0.0) + v_ / n_prof
    distinct = {l: int(np.count_nonzero(ctx.uocr_debug_router(l, rows)["count"]))
                for l in range(cfg.n_layers) if not cfg.is_dense(l)}
    cb = class_bytes(cfg, rows, [position] * rows, distinct)
    kernels = {}
    for name, t_ms in prof.items():
        b = sum(cb.get(name, [0]))
        n_l = len(cb.get(name, [1]))
        kernels[name] = {"ms_per_step": t_ms, "launches_per_step": n_l, "ms_per_launch": t_ms / n_l,
                         "bytes_per_launch": b / n_l, "gbs": b / (t_ms * 1e-3) / 1e9 if t_ms > 0 else None}
    return kernels, distinct


def step_bytes_over(cfg, rows, positions, distinct):
    """Mean algorithmic bytes per step over the timed steps' positions."""
    tot = 0.0
    for p in positions:
        tot += sum(sum(v) for v in class_bytes(cfg, rows, [p] * rows, distinct).values())
    return tot / len(positions)


def wl_label(wl):
    """Workload name plus the cache / activation options that change the kernels."""
    return wl.name + (" INT8 KV" if wl.cfg.kv_int8 else "") + (" int8 act" if getattr(wl.cfg, "act_int8", 0) else "")


def side_config(name, dev, stream, K, W, hbm_peak, cfg_overrides=None, **kw):
    """One extra configuration of the same line: time K greedy steps, report
    tokens/s, bytes and the HBM fraction, and the uocr_prefill time."""
    ctx, wl, ids, t_pre = open_workload(name, dev, stream, cfg_overrides, **kw)
    cfg, rows = wl.cfg, wl.rows
    ms, p0, last = time_greedy(ctx, wl, ids, dev, stream, K, W)
    kernels, distinct = kernel_table(ctx, wl, last, dev, p0 + K)
    sb = step_bytes_over(cfg, rows, range(p0, p0 + K), distinct)
    ms_step = ms / K
    d = {"workload": wl_label(wl), "rows": rows, "prefix": cfg.prefix_len,
         "steps": K, "warmup": W,
         "positions": [p0, p0 + K - 1], "ms_per_step": ms_step, "tokens_per_s": rows / (ms_step * 1e-3),
         "bytes_per_step": sb, "hbm_gbs": sb / (ms_step * 1e-3) / 1e9,
         "hbm_frac": sb / (ms_step * 1e-3) / 1e9 / hbm_peak,
         "kernels": {k_: {"ms_per_launch": round(v_["ms_per_launch"], 5), "gbs": round(v_["gbs"] or 0, 1)}
                     for k_, v_ in kernels.items()}}
    if t_pre is not None:
        d["prefill"] = {"tokens": rows * cfg.prefix_len, "seconds": t_pre,
                        "tokens_per_s": rows * cfg.prefix_len / t_pre,
                        "how": "uocr_prefill per row: 256 image embeddings (4 chunks of 64) + 32 prompt ids, "
                               "host wall clock around the calls and one uocr_sync"}
    ctx.close()
    return d


def time_projector(dev, stream, hbm_peak, n=256, reps=20):
    """uocr_project of n visual feature vectors of 2048 into the 1280-wide hidden
    space (Q8_0 weights): CUDA events over `reps` back-to-back calls."""
    import torch

    from quantized_moe_decode_gb300 import binding

    cfg = synth.ModelConfig(hidden=1280, n_heads=10, head_dim=128, n_layers=1, n_dense_layers=1, dense_inter=256,
                            prefix_len=4, ring_len=8, max_rows=1, proj_in=2048, fmt_proj=synth.Q8_0)
    wl = synth.make_workload("projector", cfg, 1, 1, 7)
    ctx = binding.Context(cfg, max_rows=1, stream=stream.cuda_stream, device=dev.index or 0)
    binding.load_workload(ctx, wl)
    x = torch.randn((n, 2048), device=dev).half()
    out = torch.empty((n, 1280), dtype=torch.float16, device=dev)
    for _ in range(3):
        ctx.uocr_project(n, x.data_ptr(), out.data_ptr())
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        ctx.uocr_project(n, x.data_ptr(), out.data_ptr())
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    ctx.close()
    wbytes = 1280 * 2048 * BPW[synth.Q8_0] + 1280 * 2
    b = wbytes + n * 2048 * 2 + n * 1280 * 2
    flops = 2.0 * n * 2048 * 1280
    return {"features": n, "shape": "2048 -> 1280, Q8_0 + fp16 bias", "ms_per_call": ms,
            "tokens_per_s": n / (ms * 1e-3), "bytes_per_call": b, "gbs": b / (ms * 1e-3) / 1e9,
            "tflops": flops / (ms * 1e-3) / 1e12,
            "how": "uocr_project, %d back-to-back calls, CUDA events on the caller's stream (weights L2-resident "
                   "after the first call: a latency figure, not an HBM one)" % reps}


def run_ours(args, rank, world):
    import torch

    from quantized_moe_decode_gb300 import build

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    if rank == 0:
        build.build()
    if dist:
        dist.barrier()
    t_setup = time.perf_counter()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    kw = {"rows": args.rows} if args.rows else {}
    over = dict(({"kv_int8": 1} if args.kv_int8 else {}), **({"act_int8": 1} if args.act_int8 else {}))
    ctx, wl, ids, _ = open_workload(args.workload, dev, stream, over or None, **kw)
    cfg, rows = wl.cfg, wl.rows
    K, W = args.steps, args.warmup
    log(f"[bench] setup {time.perf_counter() - t_setup:.1f}s")

    # ---- timed region: K greedy steps chained on the device
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    torch.cuda.profiler.start()  # a profiler run with --profile-from-start off sees the timed steps only
    ms, p0, last = time_greedy(ctx, wl, ids, dev, stream, K, W, dist)
    torch.cuda.profiler.stop()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = max_over_ranks(ms, dist, dev)

    # ---- per-kernel-class durations and the roofline of the dominant class
    kernels, distinct = kernel_table(ctx, wl, last, dev, p0 + K)
    hbm_peak, peak_kind = peaks()
    dom = max(kernels, key=lambda k_: kernels[k_]["ms_per_step"])
    dk = kernels[dom]
    step_bytes = step_bytes_over(cfg, rows, range(p0, p0 + K), distinct)
    launches_per_step = sum(len(v) for v in class_bytes(cfg, rows, [p0] * rows, distinct).values())
    ms_per_step = ms / K
    value = replica_throughput(world, rows, K, ms * 1e-3)

    # ---- end to end through the host-buffer entry point (pinned host buffers)
    K_e2e = min(K, 100) if cfg.vocab else 0
    h_ids = torch.empty(rows, dtype=torch.int32, pin_memory=True)
    h_pos = torch.empty(rows, dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(rows, dtype=torch.int32, pin_memory=True)
    if cfg.vocab:
        h_ids.copy_(last.cpu())
    lib = ctx.lib
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(K_e2e):
        h_pos.fill_(p0 + K + 1 + s)
        st_ = lib.uocr_decode_step_host(ctx.h, rows, h_ids.data_ptr(), h_pos.data_ptr(), h_out.data_ptr())
        if st_ != 0:
            raise RuntimeError(lib.uocr_last_error(ctx.h).decode())
        h_ids.copy_(h_out)
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e = {"value": replica_throughput(world, rows, K_e2e, e2e_s) if K_e2e else None, "unit": "tokens/s",
           "h2d_bytes_per_step": rows * 4 * 2, "d2h_bytes_per_step": rows * 4, "steps": K_e2e,
           "how": "uocr_decode_step_host (host ids/positions in, host ids out, synchronous) per step"}
    ctx.close()
    del ctx
    torch.cuda.empty_cache()

    if rank != 0:
        return
    # ---- the other configurations of the statement, as fields of the same line
    others = {}
    if not args.no_side_configs:
        K2 = min(K, 200)
        others["full_b8"] = side_config("full_b8", dev, stream, K2, W, hbm_peak)
        others["full_b1"] = side_config("full_b8", dev, stream, K2, W, hbm_peak, rows=1)
        others["stress_b64_int8_kv"] = side_config(WORKLOAD, dev, stream, K2, W, hbm_peak, {"kv_int8": 1})
        others["full_b8_g64"] = side_config("full_b8_g64", dev, stream, K2, W, hbm_peak)
        # the Falcon-OCR card's serving setting: INT8-asym weights, INT8 KV cache, int8 activations
        others["sink_b24_T350_int8"] = side_config("sink", dev, stream, K2, W, hbm_peak,
                                                   {"kv_int8": 1, "act_int8": 1}, rows=24, T=350)
        others["projector"] = time_projector(dev, stream, hbm_peak)
    cpu = cpu6 = None
    if not args.no_cpu_baseline:
        n_c, dt_c = time_oracle(wl, ORACLE_ROWS, min_s=15.0, max_steps=20)
        cpu = {"value": ORACLE_ROWS * n_c / dt_c, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
               "sample": cpu_sample_desc(ORACLE_ROWS, n_c, 2, _CORES)}
        cpu6 = cpu_baseline_threads(6)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 activations x Q8_0/Q4_0 weights, f32 accumulate", "data": "synthetic",
        "config": dict(HEADLINE_CONFIG if (args.workload == WORKLOAD and not args.rows and not over)
                       else {"workload": wl_label(wl), "rows": rows,
                             "prefix": cfg.prefix_len, "ring": cfg.ring_len},
                       global_batch=rows * world, positions=[p0, p0 + K - 1],
                       parallelism="replicas" if world > 1 else "single",
                       l2="inputs larger than L2: %.2f GB touched per step" % (step_bytes / 1e9)),
        "hbm_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "hbm_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
        "bytes_per_step": step_bytes,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dk["gbs"], "peak": hbm_peak, "unit": "GB/s",
                     "frac": dk["gbs"] / hbm_peak if dk["gbs"] else None, "traffic": ncu_traffic(dom),
                     "algorithmic_bytes_per_launch": dk["bytes_per_launch"],
                     "ms_per_launch": dk["ms_per_launch"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "timing": "the class's launches of one step replayed alone in a CUDA graph (every layer, "
                               "programmatic dependent launch between them), CUDA events on the launching "
                               "stream, 5 replays x 3"},
        "kernels": kernels,
        "other_configs": others,
        "cpu_baseline": cpu,
        "cpu_baseline_6_threads": cpu6,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ other workloads
def run_sweep(args):
    """One extra JSON line per workload (not the benchmark line): the sink decoder at
    1 and 64 rows with 350 and 3000 cached tokens, and at the Falcon-OCR card's
    1 / 6 / 12 / 24 rows with 350 cached tokens in its own serving setting (INT8 KV
    cache, dynamic int8 activations).  Each times `--steps` decode steps (capped at
    24) after 4 warm-up steps with CUDA events on the caller's stream; inputs are
    resident on the device."""
    import torch

    from quantized_moe_decode_gb300 import binding, build

    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_peak, _ = peaks()
    K, W = min(args.steps, 24), 4
    falcon = {"kv_int8": 1, "act_int8": 1}
    cases = [("sink", dict(rows=1, T=350), None), ("sink", dict(rows=64, T=350), None),
             ("sink", dict(rows=1, T=3000), None), ("sink", dict(rows=64, T=3000), None)]
    cases += [("sink", dict(rows=r, T=350), falcon) for r in (1, 6, 12, 24, 64)]
    for name, kw, over in cases:
        t0 = time.perf_counter()
        wl = synth.workload(name, steps=K + W, **kw)
        if over:
            wl.cfg = wl.cfg.replace(**over)
        cfg, rows = wl.cfg, wl.rows
        ctx = binding.Context(cfg, max_rows=rows, stream=stream.cuda_stream, device=0)
        binding.load_workload(ctx, wl)
        start = cfg.prefix_len
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if wl.step_x is not None:  # hidden-vector inputs each step, no LM head
            x_all = torch.from_numpy(np.ascontiguousarray(wl.step_x).view(np.int16)).to(dev)
            pos_all = torch.tensor([[start + s] * rows for s in range(K + W)], dtype=torch.int32, device=dev)
            for s in range(W):
                ctx.uocr_decode_step_embeds(rows, x_all[s].data_ptr(), pos_all[s].data_ptr())
            torch.cuda.synchronize()
            e0.record(stream)
            for s in range(W, W + K):
                ctx.uocr_decode_step_embeds(rows, x_all[s].data_ptr(), pos_all[s].data_ptr())
            e1.record(stream)
        else:  # token ids, greedy steps chained on the device
            ids = torch.zeros(rows, dtype=torch.int32, device=dev)
            pos = torch.zeros(rows, dtype=torch.int32, device=dev)
            if wl.prefill_embeds is not None:  # prefix built by decode steps
                nxt = torch.zeros(rows, dtype=torch.int32, device=dev)
                x = torch.zeros((rows, cfg.hidden), dtype=torch.int16, device=dev)
                ne = wl.prefill_embeds.shape[1]
                emb_all = torch.from_numpy(wl.prefill_embeds.view(np.int16)).to(dev)
                ids_all = torch.from_numpy(wl.prefill_ids).to(dev)
                for p in range(start):
                    pos.fill_(p)
                    if p < ne:
                        x.copy_(emb_all[:, p])
                        ctx.uocr_decode_step_embeds(rows, x.data_ptr(), pos.data_ptr())
                    else:
                        ids.copy_(ids_all[:, p - ne])
                        ctx.uocr_decode_step(rows, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr())
                ids.copy_(nxt)
            else:
                ids.copy_(torch.from_numpy(wl.first_ids))
            out = torch.zeros((K + W, rows), dtype=torch.int32, device=dev)
            pos.fill_(start)
            ctx.uocr_generate(rows, ids.data_ptr(), pos.data_ptr(), W, out.data_ptr())
            ids.copy_(out[W - 1])
            pos.fill_(start + W)
            torch.cuda.synchronize()
            e0.record(stream)
            ctx.uocr_generate(rows, ids.data_ptr(), pos.data_ptr(), K, out.data_ptr())
            e1.record(stream)
        torch.cuda.synchronize()
        ctx.uocr_sync()
        ms = e0.elapsed_time(e1) / K
        last = start + W + K - 1
        distinct = {l: int(np.count_nonzero(ctx.uocr_debug_router(l, rows)["count"]))
                    for l in range(cfg.n_layers) if not cfg.is_dense(l)}
        step_bytes = sum(sum(v) for v in class_bytes(cfg, rows, [last] * rows, distinct).values())
        gbs = step_bytes / (ms * 1e-3) / 1e9
        print(json.dumps({"sweep": wl_label(wl), "rows": rows, "cached_prefix": cfg.prefix_len, "steps": K,
                          "positions": [start + W, last], "ms_per_step": ms, "tokens_per_s": rows / (ms * 1e-3),
                          "bytes_per_step": step_bytes, "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak,
                          "setup_s": round(time.perf_counter() - t0, 1)}), flush=True)
        ctx.close()
        del ctx
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-configs", action="store_true", help="only the headline configuration")
    ap.add_argument("--workload", default=WORKLOAD, help="measure another named workload instead (profiling runs)")
    ap.add_argument("--rows", type=int, default=0, help="rows of that workload (0: its own)")
    ap.add_argument("--kv-int8", action="store_true", help="with an INT8 KV cache")
    ap.add_argument("--act-int8", action="store_true", help="with dynamic int8 activations")
    ap.add_argument("--cpu-sample", nargs=2, type=float, help=argparse.SUPPRESS)
    ap.add_argument("--sweep", action="store_true", help="time the other workloads (extra JSON lines) instead")
    args = ap.parse_args()
    if args.cpu_sample:
        run_cpu_sample(args.cpu_sample[0], int(args.cpu_sample[1]))
        return
    if args.sweep:
        run_sweep(args)
        return
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
