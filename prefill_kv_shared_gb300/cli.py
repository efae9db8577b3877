"""Command-line prompt prefill with a reusable KV cache file.

    python -m prefill_kv_shared_gb300.cli --model tinyllama --prompt-tokens 25 \
        --cache prefix.kvcp [--gen 16]

The flow of the PicoLM KV cache article ("PicoLM KV Cache persistence",
xxqk.cn news 668802, "usage", "file" and "rules" paragraphs), on the GPU
library: when the cache file holds a valid FP16 KV image for this model, the
prompt positions it covers are restored instead of recomputed and only the
remaining prompt tokens are prefilled (at least the last one, whose logits
start generation); when the file is missing or refused (wrong magic, layer
count, KV width or range), the whole prompt is prefilled and its cache is
written to the file.  Generated tokens are never written to the file.

The model is one of the synthetic configurations of `synth` (random weights;
no checkpoints exist here) and the prompt is seeded random token ids: the
image stores no tokens, so reusing a file with another prompt is the
caller's mistake, exactly as with the article's cache.  Every step runs in
the CUDA library; this module only orders the calls and prints what
happened, ending with one JSON line of timings.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--model", default="tinyllama", help="synthetic configuration name (synth.CONFIGS)")
    ap.add_argument("--prompt-tokens", type=int, default=25, help="prompt length")
    ap.add_argument("--seed", type=int, default=1, help="seed of the prompt's token ids")
    ap.add_argument("--cache", default=None, help="KV cache file to restore from, or to write")
    ap.add_argument("--gen", type=int, default=0, help="tokens to generate greedily after the prompt")
    ap.add_argument("--ubatch", type=int, default=512)
    ap.add_argument("--max-ctx", type=int, default=0, help="context length (0: prompt + generated tokens)")
    return ap.parse_args(argv)


def run(args, weights=None, out=sys.stdout) -> dict:
    """Run the flow; returns the summary printed as the last line."""
    import numpy as np
    import torch

    from . import binding, synth

    t_start = time.perf_counter()
    w = weights if weights is not None else synth.make_weights(synth.config(args.model))
    cfg = w.cfg
    n = args.prompt_tokens
    if n < 1:
        raise ValueError("the prompt needs at least one token")
    tokens = synth.make_tokens(cfg, n, seed=args.seed)
    max_ctx = args.max_ctx or n + args.gen
    ctx = binding.PrefillContext(w, max_ctx=max_ctx, ubatch_max=min(args.ubatch, max_ctx))
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    summary = {"model": cfg["name"], "prompt_tokens": n, "cache": args.cache, "restored": 0}
    t0 = time.perf_counter()
    start = 0
    if args.cache and os.path.exists(args.cache):
        rc, n_file = binding.kv_file_check(args.cache, ctx.n_layers_written, ctx.kv_dim, max_ctx)
        if rc == binding.PF_OK:
            take = min(n_file, n - 1)  # the last prompt token is always run: its logits start generation
            if take > 0 and ctx.kv_load_file(args.cache, take) == binding.PF_OK:
                start = take
                print(f"restored {take} prompt positions from {args.cache} ({n_file} in the file); "
                      f"prefilling the remaining {n - take} tokens", file=out)
        else:
            print(f"cache file {args.cache} refused (status {rc}); prefilling the whole prompt", file=out)
    for i in range(start, n, args.ubatch):
        ctx.ubatch(tokens[i:i + args.ubatch], i, i + args.ubatch >= n, logits)
    ctx.sync()
    t1 = time.perf_counter()
    summary["restored"] = start
    summary["prefill_s"] = t1 - t0
    if args.cache and start == 0:
        ctx.kv_save_file(args.cache)
        size = os.path.getsize(args.cache)
        summary["cache_bytes"] = size
        print(f"wrote the cache of {n} prompt positions to {args.cache} ({size} bytes)", file=out)
    first = logits.cpu().numpy().copy()
    summary["first_token"] = int(np.argmax(first))
    generated = []
    tok = summary["first_token"]
    for i in range(args.gen):
        generated.append(tok)
        if n + i >= max_ctx:
            break
        ctx.ubatch(np.array([tok], dtype=np.int32), n + i, True, logits)
        ctx.sync()
        tok = int(torch.argmax(logits).item())
    summary["generated"] = generated
    summary["total_s"] = time.perf_counter() - t_start
    summary["run_s"] = time.perf_counter() - t0
    ctx.close()
    print(json.dumps(summary), file=out, flush=True)
    summary["logits"] = first
    return summary


def main(argv=None):
    args = parse_args(argv)
    run(args)


if __name__ == "__main__":
    main()
