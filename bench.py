#!/usr/bin/env python3
"""Prompt-prefill benchmark of the KV-shared library on GB300.

Workload: the E2B-shaped synthetic model (24 layers, layers 16-23 KV-shared,
d_model 1536, 8/1 heads of 256, GeGLU 6144, vocab 32768, per-layer embedding
256, Q4_0 weights drawn from seed 0) prefilling one sequence of 512 random
tokens (seed 1) in one ubatch, with the KV-shared row pruning on.  A "step" is
one whole prefill pass of that prompt (every layer, the pruning, the head)
from tokens resident in device memory to the last row's logits.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
same workload instead.  Multi-GPU runs are independent replicas (one
sequence per GPU, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s (1 seq) at 512/2048/8192 prompt, pruning on vs off, % roofline"
UNIT = "tokens/s"
WORKLOAD = "e2b-512"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep-steps", type=int, default=5)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hbm", action="store_true", help="skip the single-row attention / KV restore timings")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="reference arm: time passes over the first N prompt tokens (0: sized to ~2 minutes)")
    ap.add_argument("--hbm-only", action="store_true",
                    help="run only the single-row attention / KV restore timings and print them (for ncu)")
    ap.add_argument("--profile-passes", type=int, default=0,
                    help="run this many untimed prefill passes of the workload and exit (for ncu)")
    ap.add_argument("--profile-prompt", type=int, default=512,
                    help="prompt length of the --profile-passes passes (ubatches of 512)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: barrier + max of the timings only)


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if os.environ.get("PREFILL_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def source_sha(paths):
    import hashlib
    m = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            m.update(f.read())
    return m.hexdigest()[:16]


def gemm_traffic():
    """DRAM bytes per GEMM launch from the committed one-kernel ncu capture
    (profiles/gemm_tc_e2b512_dram.json: the six projections of one writing
    layer), or None when it is absent or the kernel source has changed since
    those counters were taken."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_e2b512_dram.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if source_sha(d["source_files"]) != d["source_sha"]:
            return None
        return d["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)


def oracle_rate(cfg, weights, tokens, budget_s: float, min_steps: int = 1, warm: bool = True):
    """Tokens/s of the oracle's pruned prefill of `tokens`, timed on the host
    cores for at least min_steps passes and about budget_s seconds."""
    import numpy as np
    from oracle.prefill import OracleContext
    ctx = OracleContext(cfg, weights, len(tokens))
    if warm:  # decodes and caches the weights
        ctx.prefill(tokens, 512, prune=True)
        ctx.reset()
    n, t0 = 0, time.perf_counter()
    while True:
        ctx.reset()
        out = ctx.prefill(tokens, 512, prune=True)
        n += 1
        el = time.perf_counter() - t0
        if n >= min_steps and el >= budget_s:
            break
    assert np.isfinite(out).all()
    return n * len(tokens) / el, el / n, n


def cpu_threads() -> int:
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count() or 1


def run_reference(args, dist: Dist):
    """The oracle on the host cores.  A step is one pruned prefill pass over a
    prompt sample: the whole 512-token prompt when K such passes fit in about
    two minutes, else its first S tokens with S sized to fit."""
    if dist.rank != 0:
        return
    from oracle.prefill import OracleContext
    from prefill_kv_shared_gb300 import synth
    cfg = synth.config("e2b")
    w = synth.make_weights(cfg)
    tok = synth.make_tokens(cfg, 512)
    ctx = OracleContext(cfg, w, 512)
    if args.ref_tokens > 0:
        S = min(512, args.ref_tokens)
        t512 = None
        ctx.prefill(tok[:S], 512, prune=True)  # decodes and caches the weights
    else:
        ctx.prefill(tok, 512, prune=True)  # decodes and caches the weights
        ctx.reset()
        t0 = time.perf_counter()
        ctx.prefill(tok, 512, prune=True)
        t512 = time.perf_counter() - t0
        budget = 120.0
        S = 512 if args.steps * t512 <= budget else max(16, int(512 * budget / (args.steps * t512)))
    sample = tok[:S]
    for _ in range(args.warmup):
        ctx.reset()
        ctx.prefill(sample, 512, prune=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ctx.reset()
        ctx.prefill(sample, 512, prune=True)
    el = time.perf_counter() - t0
    value = args.steps * S / el
    cores = cpu_threads()
    desc = (f"{args.steps} pruned prefill passes over the first {S} tokens of the 512-token prompt"
            + ("" if S == 512 or t512 is None else f" (a full 512-token pass takes {t512:.2f} s)"))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "prompt": 512, "prompt_sample": S, "ubatch": 512, "pruning": True,
                   "program": "numpy fp32 oracle (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# HBM-bound kernels on their own: the single-row KV-shared attention and the
# KV image restore, each cold (L2 scrubbed before every timed launch) and warm


def hbm_kernels(dev, stream, peaks, iters: int = 20):
    import ctypes as C

    import torch

    from prefill_kv_shared_gb300 import binding
    lib = binding.load()
    bw = peaks["hbm_gbs"]
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # 512 MB > L2 (129 MB)
    sp = C.c_void_p(scrub.data_ptr())
    us = C.c_float(0.0)
    sh = C.c_void_p(stream.cuda_stream)
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    out = {"shared_attention": {}, "kv_restore": {}}
    # (model, Hq, Hkv, hd, keys): the single-row attention of a KV-shared layer
    for name, hq, hkv, hd, n in (("e2b", 8, 1, 256, 8192), ("e2b", 8, 1, 256, 32768),
                                 ("e4b", 8, 2, 256, 8192), ("e4b", 8, 2, 256, 32768)):
        q = torch.randn(hq * hd, generator=g, device=dev).half()
        k = torch.randn(n, hkv * hd, generator=g, device=dev).half()
        v = torch.randn(n, hkv * hd, generator=g, device=dev).half()
        o = torch.empty(hq * hd, dtype=torch.bfloat16, device=dev)
        algo = 2.0 * n * hkv * hd * 2  # K and V read once
        row = {"keys": n, "bytes": algo}
        for tag, sc in (("cold", sp), ("warm", None)):
            rc = lib.pfop_attention_bench(1, q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, hq, hkv, hd, n - 1, n,
                                          o.data_ptr(), sc, scrub.numel() if sc else 0, 3, iters, C.byref(us), sh)
            binding.check_op(rc)
            gbs = algo / (us.value * 1e-6) / 1e9
            row[tag] = {"us": us.value, "gbs": gbs, "frac": gbs / bw}
        out["shared_attention"][f"{name}_{n}"] = row
        del q, k, v, o
    # (workload, writing layers, kv_dim, positions): kv_load of a KV image
    for name, lw, kv, n in (("tinyllama_500", 22, 256, 500), ("e2b_8192", 16, 256, 8192),
                            ("e4b_8192", 24, 512, 8192), ("e4b_32768", 24, 512, 32768)):
        seg = n * kv * 2
        image = torch.empty(16 + 2 * lw * seg, dtype=torch.uint8, device=dev)
        cache = torch.empty(2 * lw * n * kv, dtype=torch.float16, device=dev)
        algo = 2.0 * (2 * lw * seg)  # read the image body, write the cache
        row = {"image_bytes": image.numel(), "bytes": algo}
        for tag, sc in (("cold", sp), ("warm", None)):
            rc = lib.pfop_kv_copy_bench(1, cache.data_ptr(), n * kv, image.data_ptr(), seg, 2 * lw, seg, sc,
                                        scrub.numel() if sc else 0, 3, iters, C.byref(us), sh)
            binding.check_op(rc)
            gbs = algo / (us.value * 1e-6) / 1e9
            row[tag] = {"us": us.value, "gbs": gbs, "frac": gbs / bw}
        out["kv_restore"][name] = row
        del image, cache
    del scrub
    torch.cuda.empty_cache()
    out["peak_gbs"] = bw
    out["note"] = ("bytes = algorithmic traffic (K and V read once; image read + cache written); "
                   "cold: 512 MB written before every timed launch; mean of %d launches" % iters)
    return out


# Reuse of a fixed prompt prefix through its KV image (PicoLM KV cache
# article, "usage" and "measured": a system prompt is prefilled once and its
# FP16 KV image restored for every later request).  TinyLlama shape: a
# 500-token prefix, requests that each append a 32-token suffix.  full = the
# whole prompt prefilled in ubatches of `ub`; reuse = restore the prefix's
# positions from the image (device or host memory), then prefill the suffix.


def prefix_reuse(ctx, prefix, suffixes, ub, logits, images, timer):
    """ctx: a PrefillContext (or a stand-in with its methods); images:
    {name: (image, nbytes)}; timer(fn) -> ms that one call of fn took on the
    context's stream.  Returns ms per request for each way."""
    import numpy as np
    n0 = len(prefix)
    prompts = [np.concatenate([prefix, s]) for s in suffixes]

    def full():
        for p in prompts:
            ctx.reset()
            for i in range(0, len(p), ub):
                ctx.ubatch(p[i:i + ub], i, i + ub >= len(p), logits)

    def reuse(img, nbytes):
        for s in suffixes:
            ctx.reset()
            ctx.kv_load(img, nbytes, n0)
            ctx.ubatch(s, n0, True, logits)

    out = {"requests": len(suffixes), "prefix": n0, "suffix": len(suffixes[0]),
           "full_ms": timer(full) / len(suffixes)}
    for name, (img, nbytes) in images.items():
        ms = timer(lambda: reuse(img, nbytes)) / len(suffixes)
        out[f"reuse_{name}_ms"] = ms
        out[f"speedup_{name}"] = out["full_ms"] / ms
    return out


def run_prefix_reuse(dev, stream):
    """prefix_reuse on the GPU: the 500-token prefix of the TinyLlama-shaped
    model (no KV-shared layers, so no pruning) cached once as a device image
    and as a host (pageable) copy, 64 requests of 32 tokens (seeds 2..65)."""
    import numpy as np
    import torch

    from prefill_kv_shared_gb300 import binding, synth
    tl = synth.make_weights(synth.config("tinyllama"))
    cfg = tl.cfg
    ctx = binding.PrefillContext(tl, max_ctx=532, ubatch_max=512, stream=stream)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)
    prefix = synth.make_tokens(cfg, 500, seed=1)
    suffixes = [synth.make_tokens(cfg, 32, seed=2 + i) for i in range(64)]
    ctx.ubatch(prefix, 0, False)
    nbytes = ctx.kv_image_bytes(500)
    img = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ctx.kv_save(img, nbytes)
    host_img = np.empty(nbytes, dtype=np.uint8)
    ctx.kv_save(host_img, nbytes)
    ctx.sync()

    def timer(fn):
        fn()  # warm-up
        ctx.sync()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    out = prefix_reuse(ctx, prefix, suffixes, 512, logits, {"device": (img, nbytes), "host": (host_img, nbytes)},
                       timer)
    # the restored pass computes what the full pass computes (first request)
    ctx.reset()
    p = np.concatenate([prefix, suffixes[0]])
    ctx.ubatch(p[:512], 0, False)
    ctx.ubatch(p[512:], 512, True, logits)
    ctx.sync()
    want = logits.cpu().numpy().copy()
    ctx.reset()
    ctx.kv_load(img, nbytes, 500)
    ctx.ubatch(suffixes[0], 500, True, logits)
    ctx.sync()
    got = logits.cpu().numpy()
    out["max_rel_diff"] = float(np.abs(got - want).max() / np.abs(want).max())
    out["image_bytes"] = nbytes
    out["note"] = "CUDA events on the library's stream per request, tokens from host memory"
    ctx.close()
    del tl, img, logits
    torch.cuda.empty_cache()
    return out


def run_multi_seq(w, dev, stream, steps: int = 10):
    """Four E2B sequences of 128 tokens in one ubatch of 512 over a unified
    KV cache (the server setting of the Gemma 4 prefill news, section 5):
    the per-sequence gather (pruning on), the unpruned pass, and the same
    four prompts as four one-sequence prefills; ms per batch of four."""
    import numpy as np
    import torch

    from prefill_kv_shared_gb300 import binding, synth
    cfg = w.cfg
    toks = [synth.make_tokens(cfg, 128, seed=40 + q) for q in range(4)]
    flat = torch.from_numpy(np.concatenate(toks)).to(dev)
    runs = [(q, 128, True) for q in range(4)]
    lg = torch.empty((4, cfg["vocab"]), dtype=torch.float32, device=dev)
    out = {"sequences": 4, "tokens_per_sequence": 128}

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    ctx = binding.PrefillContext(w, max_ctx=128, ubatch_max=512, n_seq_max=4, stream=stream)

    def batch():
        ctx.reset()
        ctx.ubatch_seqs(flat, runs, lg)
    res = {}
    for name, mode in (("gathered", True), ("unpruned", False)):
        ctx.set_prune(mode)
        out[f"{name}_ms"] = timed(batch)
        res[name] = lg.cpu().numpy().copy()
    ctx.close()
    one = binding.PrefillContext(w, max_ctx=128, ubatch_max=128, stream=stream)
    d_toks = [torch.from_numpy(t).to(dev) for t in toks]

    def separate():
        for q in range(4):
            one.reset()
            one.ubatch(d_toks[q], 0, True, lg[q])
    out["four_single_sequence_ms"] = timed(separate)
    one.close()
    out["gathered_tokens_per_s"] = 512 / (out["gathered_ms"] * 1e-3)
    out["gathered_vs_unpruned"] = out["unpruned_ms"] / out["gathered_ms"]
    out["gathered_vs_single_sequence"] = out["four_single_sequence_ms"] / out["gathered_ms"]
    out["gathered_equals_unpruned"] = bool(np.array_equal(res["gathered"], res["unpruned"]))
    return out


def run_cache_cli():
    """The command-line cache-file flow (PicoLM KV cache article, "usage" and
    "measured": a 25-token TinyLlama prompt, first run without the file,
    then a run that restores it), 16 generated tokens each; wall-clock
    seconds of each run after the weights are built (host work included)."""
    import io
    import tempfile

    from prefill_kv_shared_gb300 import cli, synth
    w = synth.make_weights(synth.config("tinyllama"))
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "prompt.kvcp")
        args = cli.parse_args(["--prompt-tokens", "25", "--cache", path, "--gen", "16"])
        cli.run(args, weights=w, out=io.StringIO())  # warm-up (writes the file)
        os.remove(path)
        full = cli.run(args, weights=w, out=io.StringIO())
        cached = cli.run(args, weights=w, out=io.StringIO())
    return {"prompt_tokens": 25, "generated": 16, "file_bytes": full.get("cache_bytes"),
            "full_run_s": full["run_s"], "cached_run_s": cached["run_s"], "restored": cached["restored"],
            "same_tokens": full["generated"] == cached["generated"],
            "note": "wall clock of cli.run after the weights exist: create, restore or prefill, save, generation"}


# ---------------------------------------------------------------------------
# per-class roofline fractions from a run with CUDA events around every launch

CLASS_BOUNDS = {"gemm": "tensor", "attention": "tensor", "norm": "hbm", "other": "hbm", "gemm_row": "hbm",
                "attention_row": "hbm"}


def class_fractions(stats, steps, peaks):
    """Per launch class: launches and device ms per step, achieved rate and
    its fraction of the measured peak (tensor classes: algorithmic FLOPs
    against the burst bf16 peak, since every launch is timed on its own;
    HBM classes: algorithmic bytes against the measured copy bandwidth)."""
    peak_t = peaks["bf16_tflops"]
    out = {}
    for k, v in stats.items():
        d = {"bound": CLASS_BOUNDS.get(k, "hbm"), "launches_per_step": v["launches"] / steps,
             "ms_per_step": v["ms"] / steps,
             "tflops": (v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["ms"] > 0 and v["flops"] > 0 else None,
             "gbs": (v["bytes"] / (v["ms"] * 1e-3) / 1e9) if v["ms"] > 0 else None}
        if d["bound"] == "tensor":
            d["frac"] = d["tflops"] / peak_t if d["tflops"] else None
        else:
            d["frac"] = d["gbs"] / peaks["hbm_gbs"] if d["gbs"] else None
        out[k] = d
    return out


def pass_fraction(stats, steps, peaks, pass_ms):
    """Whole-pass roofline fraction: the sum over launch classes of
    max(FLOPs / bf16 peak, bytes / HBM bandwidth), over the measured pass."""
    ideal_ms = sum(max(v["flops"] / (peaks["bf16_tflops"] * 1e12), v["bytes"] / (peaks["hbm_gbs"] * 1e9))
                   for v in stats.values()) * 1e3 / steps
    return ideal_ms / pass_ms


def timed_classes(ctx, step, steps):
    """Run `steps` steps with per-launch event timing; the context's stats."""
    ctx.reset_stats()
    ctx.set_timing(True)
    for _ in range(steps):
        step()
    st = ctx.stats()
    ctx.set_timing(False)
    ctx.reset_stats()
    return st


# ---------------------------------------------------------------------------
# our arm


def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    from prefill_kv_shared_gb300 import binding, synth

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    binding.load()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    if args.hbm_only:
        if dist.rank == 0:
            print(json.dumps(hbm_kernels(dev, stream, load_peaks()[0])), flush=True)
        return
    cfg = synth.config("e2b")
    w = synth.make_weights(cfg)
    N, UB = 512, 512
    tok_host = synth.make_tokens(cfg, N)
    tok = torch.from_numpy(tok_host).to(dev)
    ctx = binding.PrefillContext(w, max_ctx=N, ubatch_max=UB, prune=True, stream=stream)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device=dev)

    def step():
        ctx.reset()
        ctx.ubatch(tok, 0, True, logits)

    if args.profile_passes:
        n = args.profile_prompt
        pctx, ptok = ctx, tok
        if n != N:
            pctx = binding.PrefillContext(w, max_ctx=n, ubatch_max=UB, prune=True, stream=stream)
            ptok = torch.from_numpy(synth.make_tokens(cfg, n)).to(dev)
        for _ in range(args.profile_passes):
            pctx.reset()
            for i in range(0, n, UB):
                pctx.ubatch(ptok[i:i + UB], i, i + UB >= n, logits)
            pctx.sync()
        print("ok", float(logits.abs().max()), flush=True)
        if pctx is not ctx:
            pctx.close()
        ctx.close()
        return

    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    ctx.sync()
    torch.cuda.synchronize(dev)
    dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ctx.sync()
    dist.barrier()
    ms_stream = dist.max(e0.elapsed_time(e1) / args.steps)

    # the same pass recorded once as a CUDA graph and replayed (the tokens
    # stay in the recorded device buffer): one graph launch per step
    ms_graph, graph_err = None, None
    try:
        ctx.reset()
        ctx.graph_capture(tok, 0, True, logits)

        def gstep():
            ctx.reset()
            ctx.graph_launch()
        for _ in range(args.warmup):
            gstep()
        ctx.sync()
        torch.cuda.synchronize(dev)
        dist.barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            gstep()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ctx.sync()
        dist.barrier()
        ms_graph = dist.max(e0.elapsed_time(e1) / args.steps)
    except binding.PrefillError as e:  # recorded in the line; the stream figure stands
        graph_err = str(e)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    ms = ms_graph if ms_graph is not None else ms_stream
    value = dist.world * N / (ms * 1e-3)
    clk = clocks.summary(t_wall0 - 0.3, t_wall1 + 0.3)

    # the same steps again with CUDA events around every launch: per-class
    # device time and algorithmic work
    st = timed_classes(ctx, step, args.steps)
    launches_per_step = sum(v["launches"] for v in st.values()) / args.steps

    peaks, peak_src = load_peaks()
    g = st["gemm"]
    gemm_ms_avg = g["ms"] / max(g["timed"], 1)
    gemm_flops_avg = g["flops"] / max(g["launches"], 1)
    achieved = gemm_flops_avg / (gemm_ms_avg * 1e-3) / 1e12 if gemm_ms_avg > 0 else None
    peak = peaks["bf16_tflops"]
    traffic = gemm_traffic()
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "kernel": "gemm_tc_kernel, projections of the 512-row ubatch (launches of more than 16 rows)",
                "peak_source": f"{peak_src} bf16 burst (each launch timed on its own)",
                "classes": class_fractions(st, args.steps, peaks),
                "class_note": ("per-launch CUDA events around every launch (PDL overlap removed); gemm_row = the "
                               "one-row projections (the output row of the KV-shared layers and the LM head), "
                               "bound by their weight bytes; attention_row = the single-row attention of the "
                               "KV-shared layers")}
    roofline["pass_frac"] = pass_fraction(st, args.steps, peaks, ms)

    # end to end through the C ABI with host buffers: tokens from pinned host
    # memory each step, logits read back to pinned host memory each step
    tok_pinned = torch.from_numpy(tok_host.copy()).pin_memory()
    out_pinned = torch.empty(cfg["vocab"], dtype=torch.float32).pin_memory()
    tok_np = tok_pinned.numpy()

    def e2e_stream_step():
        ctx.reset()
        ctx.ubatch(tok_np, 0, True, logits)
        out_pinned.copy_(logits, non_blocking=True)
        torch.cuda.synchronize(dev)

    def e2e_graph_step():
        tok.copy_(tok_pinned, non_blocking=True)  # into the recorded buffer, on the library's stream
        ctx.reset()
        ctx.graph_launch()
        out_pinned.copy_(logits, non_blocking=True)
        torch.cuda.synchronize(dev)

    def e2e_time(fn):
        for _ in range(3):
            fn()
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            fn()
        return dist.max((time.perf_counter() - t0) / args.steps)
    e2e_stream_s = e2e_time(e2e_stream_step)
    e2e_s = e2e_time(e2e_graph_step) if ms_graph is not None else e2e_stream_s
    e2e = {"value": dist.world * N / e2e_s, "unit": UNIT, "h2d_bytes_per_step": N * 4,
           "d2h_bytes_per_step": cfg["vocab"] * 4,
           "path": "graph replay" if ms_graph is not None else "stream launches",
           "stream_launches_value": dist.world * N / e2e_stream_s}
    assert np.isfinite(out_pinned.numpy()).all()
    ctx.close()

    # pruning on/off: E2B at 512/2048/8192/32768 (ubatches of 512) and E4B at
    # 8192 and 32768 (ubatches of 1024), rank 0's GPU only; each entry with
    # its class fractions from one more pass with every launch timed.  "off"
    # keeps the output row of the KV-shared layers on the single-row kernels
    # (logits bit-identical to "on"); "off_plain" runs every row through the
    # prefill kernels (the fastest unpruned pass).
    sweep = None
    if not args.no_sweep and dist.rank == 0:
        sweep = {}
        models = {"e2b": w}
        peaks = load_peaks()[0]
        for mname, n, ub in (("e2b", 512, 512), ("e2b", 2048, 512), ("e2b", 8192, 512), ("e2b", 32768, 512),
                             ("e4b", 8192, 1024), ("e4b", 32768, 1024)):
            if mname not in models:
                models.clear()  # one model's weights resident at a time
                models[mname] = synth.make_weights(synth.config(mname))
            wm = models[mname]
            big = binding.PrefillContext(wm, max_ctx=n, ubatch_max=ub, prune=True, stream=stream)
            lg = torch.empty(wm.cfg["vocab"], dtype=torch.float32, device=dev)
            t = torch.from_numpy(synth.make_tokens(wm.cfg, n)).to(dev)
            key = f"{n}" if mname == "e2b" else f"{mname}_{n}"
            steps_n = args.sweep_steps if n <= 8192 else max(2, args.sweep_steps // 2)
            for prune in (True, False, binding.PF_PRUNE_OFF_PLAIN):
                big.set_prune(prune)
                tag = "off_plain" if prune is binding.PF_PRUNE_OFF_PLAIN else ("on" if prune else "off")

                def sweep_step():
                    big.reset()
                    for i in range(0, n, ub):
                        big.ubatch(t[i:i + ub], i, i + ub >= n, lg)
                sweep_step()
                big.sync()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(steps_n):
                    sweep_step()
                b.record(stream)
                torch.cuda.synchronize(dev)
                sms = a.elapsed_time(b) / steps_n
                st_n = timed_classes(big, sweep_step, 1)
                cl = class_fractions(st_n, 1, peaks)
                sweep[f"{key}_{tag}"] = {
                    "ms": sms, "tokens_per_s": n / (sms * 1e-3), "ubatch": ub,
                    "pass_frac": pass_fraction(st_n, 1, peaks, sms),
                    "frac": {k: cl[k]["frac"] for k in ("gemm", "attention", "gemm_row", "attention_row", "norm")},
                    "class_ms": {k: cl[k]["ms_per_step"] for k in cl}}
            sweep[f"{key}_speedup"] = sweep[f"{key}_off"]["ms"] / sweep[f"{key}_on"]["ms"]
            sweep[f"{key}_speedup_vs_plain"] = sweep[f"{key}_off_plain"]["ms"] / sweep[f"{key}_on"]["ms"]
            big.close()
            del t, lg
        models.clear()
        # generation after the prompt (llama-bench tg128): 128 one-token
        # ubatches after a 512-token prefill, pruning on and off
        dec = binding.PrefillContext(w, max_ctx=512 + 128, ubatch_max=UB, prune=True, stream=stream)
        tg = torch.from_numpy(synth.make_tokens(cfg, 512 + 128)).to(dev)
        for prune in (True, False):
            dec.set_prune(prune)

            def prefill_prompt():
                dec.reset()
                dec.ubatch(tg[:512], 0, True, logits)

            def gen128():
                for i in range(512, 512 + 128):
                    dec.ubatch(tg[i:i + 1], i, True, logits)
            prefill_prompt()
            gen128()
            dec.sync()
            tot = 0.0
            for _ in range(2):
                prefill_prompt()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                gen128()
                b.record(stream)
                torch.cuda.synchronize(dev)
                tot += a.elapsed_time(b)
            gms = tot / 2
            sweep[f"tg128_{'on' if prune else 'off'}"] = {"ms": gms, "tokens_per_s": 128 / (gms * 1e-3)}
        dec.close()

    hbm = None
    if not args.no_hbm and dist.rank == 0:
        hbm = hbm_kernels(dev, stream, load_peaks()[0])

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        rate, per, n = oracle_rate(cfg, w, tok_host, budget_s=10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{n} pruned prefill passes of the same 512-token prompt ({per:.2f} s each), weights decoded once before timing"}

    if sweep is not None:
        try:
            sweep["prefix_reuse_tinyllama"] = run_prefix_reuse(dev, stream)
        except Exception as e:  # recorded, never fatal to the line
            sweep["prefix_reuse_tinyllama"] = {"error": f"{type(e).__name__}: {e}"}
        try:
            sweep["multi_sequence_e2b_4x128"] = run_multi_seq(w, dev, stream)
        except Exception as e:  # recorded, never fatal to the line
            sweep["multi_sequence_e2b_4x128"] = {"error": f"{type(e).__name__}: {e}"}
        try:
            sweep["cache_file_cli_tinyllama_25"] = run_cache_cli()
        except Exception as e:  # recorded, never fatal to the line
            sweep["cache_file_cli_tinyllama_25"] = {"error": f"{type(e).__name__}: {e}"}

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "model": "E2B-shaped synthetic, Q4_0 weights", "prompt": N,
                       "ubatch": UB, "pruning": True, "global_batch": dist.world, "seq_len": N,
                       "parallelism": f"replicas x{dist.world}",
                       "l2": "inputs larger than L2 (488 MB of Q4_0 weights streamed every step)"},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "launch_path": ("one CUDA graph replay per step (prefill_graph_launch)" if ms_graph is not None
                            else "stream launches (prefill_ubatch)"),
            "stream_launches": {"ms_per_step": ms_stream, "value": dist.world * N / (ms_stream * 1e-3)},
            "graph_error": graph_err,
            "e2e": e2e, "roofline": roofline, "clocks": clk, "cpu_baseline": cpu, "sweep": sweep,
            "hbm_kernels": hbm,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
