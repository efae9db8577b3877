"""bench.py's host-side logic on a machine without a GPU: the prefix-reuse
measurement drives the context in the order the cached-prefix flow needs
(PicoLM KV cache article, "usage": restore the prefix, then prefill only the
new tokens), checked with a stand-in context that records the calls."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class RecordingCtx:
    def __init__(self):
        self.calls = []
        self.n_pos = 0

    def reset(self):
        self.calls.append(("reset",))
        self.n_pos = 0

    def kv_load(self, img, nbytes, n_pos):
        self.calls.append(("kv_load", img, nbytes, n_pos))
        self.n_pos = n_pos

    def ubatch(self, tokens, pos0, is_last, logits=None):
        assert pos0 == self.n_pos, "ubatch must continue at the cached position count"
        self.calls.append(("ubatch", len(tokens), pos0, bool(is_last), tuple(int(t) for t in tokens[:2])))
        self.n_pos += len(tokens)


def test_prefix_reuse_call_order():
    prefix = np.arange(500, dtype=np.int32)
    suffixes = [np.full(32, 1000 + i, dtype=np.int32) for i in range(3)]
    ctx = RecordingCtx()
    runs = []

    def timer(fn):
        before = len(ctx.calls)
        fn()
        runs.append(ctx.calls[before:])
        return 6.0

    out = bench.prefix_reuse(ctx, prefix, suffixes, 512, "LOGITS", {"device": ("IMG", 123)}, timer)
    full, reuse = runs
    # full: every request prefills its whole 532-token prompt in ubatches of
    # 512 and 20 rows; only the second is the last ubatch
    assert full == [c for i in range(3) for c in (
        ("reset",), ("ubatch", 512, 0, False, (0, 1)), ("ubatch", 20, 512, True, (1000 + i, 1000 + i)))]
    # reuse: restore the 500 cached positions, then only the 32 new tokens
    assert reuse == [c for i in range(3) for c in (
        ("reset",), ("kv_load", "IMG", 123, 500), ("ubatch", 32, 500, True, (1000 + i, 1000 + i)))]
    assert out["full_ms"] == 2.0 and out["reuse_device_ms"] == 2.0 and out["speedup_device"] == 1.0
    assert out["requests"] == 3 and out["prefix"] == 500 and out["suffix"] == 32
