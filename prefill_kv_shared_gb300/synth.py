"""Seeded synthetic inputs: model shapes, weights and prompt tokens.

This module only draws random numbers and lays them out in the storage
formats the library accepts.  It holds none of the prefill arithmetic: no
dequantisation, no norm, no attention.  Both the CPU oracle (through the
tests) and the CUDA path consume what it produces.

Shapes follow the synthetic workloads of the prefill-pruning write-up for
Gemma 4 E2B/E4B (devotd.net llama.cpp Gemma 4 prefill news, section 1) and the
TinyLlama-shaped KV-cache-persistence workload (xxqk.cn PicoLM KV cache
article, "file" paragraph: 22 layers, kv_dim 256, FP16 keys and values).

Q4_0 storage (per 32-element block, 18 bytes): a little-endian fp16 scale d,
then 16 bytes; byte j carries element j in its low nibble and element j+16 in
its high nibble.  A weight value is d * (nibble - 8).  Scales are drawn as
fp16(|N(0, 0.002)|) for the whole tensor first, then nibbles uniform on 0..15.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

import numpy as np

WEIGHT_SEED = 0
TOKEN_SEED = 1


def _kv_src_by_parity(n_layer: int, n_kv_start: int) -> list[int]:
    """Writing layers map to -1.  A shared layer reads the last writing layer
    of its own parity (even -> second to last, odd -> last)."""
    last_even = n_kv_start - 2 if (n_kv_start - 2) % 2 == 0 else n_kv_start - 1
    last_odd = n_kv_start - 1 if (n_kv_start - 1) % 2 == 1 else n_kv_start - 2
    src = []
    for il in range(n_layer):
        if il < n_kv_start:
            src.append(-1)
        else:
            src.append(last_even if il % 2 == 0 else last_odd)
    return src


CONFIGS: dict[str, dict] = {
    # 4 layers, layers 0-1 write KV, layers 2-3 read layer 1.
    "tiny": dict(
        n_layer=4, n_layer_kv_from_start=2, d_model=256, n_head=4, n_head_kv=1,
        head_dim=64, ffn_dim=1024, ffn="geglu", vocab=1024, ple_dim=64,
        rms_eps=1e-6, rope_base=10000.0, kv_src=[-1, -1, 1, 1], wtype="f32",
    ),
    # E2B-shaped: 24 layers, 0-15 write, 16-23 shared (even -> 14, odd -> 15).
    "e2b": dict(
        n_layer=24, n_layer_kv_from_start=16, d_model=1536, n_head=8, n_head_kv=1,
        head_dim=256, ffn_dim=6144, ffn="geglu", vocab=32768, ple_dim=256,
        rms_eps=1e-6, rope_base=10000.0, kv_src=_kv_src_by_parity(24, 16),
        wtype="q4_0",
    ),
    # E4B-shaped: 36 layers, 0-23 write, 24-35 shared (even -> 22, odd -> 23).
    "e4b": dict(
        n_layer=36, n_layer_kv_from_start=24, d_model=2560, n_head=8, n_head_kv=2,
        head_dim=256, ffn_dim=10240, ffn="geglu", vocab=32768, ple_dim=256,
        rms_eps=1e-6, rope_base=10000.0, kv_src=_kv_src_by_parity(36, 24),
        wtype="q4_0",
    ),
    # TinyLlama-shaped dense model: every layer writes KV, no PLE, SwiGLU.
    "tinyllama": dict(
        n_layer=22, n_layer_kv_from_start=22, d_model=2048, n_head=32, n_head_kv=4,
        head_dim=64, ffn_dim=5632, ffn="swiglu", vocab=32000, ple_dim=0,
        rms_eps=1e-6, rope_base=10000.0, kv_src=[-1] * 22, wtype="q4_0",
    ),
}

# Prompt workloads: (config, prompt length, ubatch size).
WORKLOADS: dict[str, tuple[str, int, int]] = {
    "tiny-64": ("tiny", 64, 64),
    "e2b-512": ("e2b", 512, 512),
    "e2b-2048": ("e2b", 2048, 512),
    "e2b-8192": ("e2b", 8192, 512),
    "e2b-32768": ("e2b", 32768, 512),
    "e4b-8192": ("e4b", 8192, 1024),
    "e4b-32768": ("e4b", 32768, 1024),
}


def config(name: str, **overrides) -> dict:
    cfg = copy.deepcopy(CONFIGS[name])
    cfg["name"] = name
    cfg.update(overrides)
    return cfg


def _kv_src_last(n_layer: int, n_kv_start: int) -> list[int]:
    """Every shared layer reads the last writing layer (the tiny model's rule)."""
    return [-1 if il < n_kv_start else n_kv_start - 1 for il in range(n_layer)]


def scaled_config(name: str, **dims) -> dict:
    """A smaller model with the same structure as `name` (for fast tests).
    kv_src is recomputed with the base model's rule unless given."""
    cfg = config(name)
    cfg.update(dims)
    if "kv_src" not in dims:
        L, S = cfg["n_layer"], cfg["n_layer_kv_from_start"]
        if S >= L:
            cfg["kv_src"] = [-1] * L
        elif name == "tiny":
            cfg["kv_src"] = _kv_src_last(L, S)
        else:
            cfg["kv_src"] = _kv_src_by_parity(L, S)
    cfg["name"] = name + "-scaled"
    return cfg


# ---------------------------------------------------------------------------
# weight drawing

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
              "w_down", "ple_gate", "ple_proj")


def layer_shapes(cfg: dict, il: int) -> dict[str, tuple[int, ...] | None]:
    """Shapes of one layer's tensors ([out, in] for matrices); None = absent."""
    D, q, kv = cfg["d_model"], cfg["n_head"] * cfg["head_dim"], cfg["n_head_kv"] * cfg["head_dim"]
    F, P = cfg["ffn_dim"], cfg["ple_dim"]
    writes = il < cfg["n_layer_kv_from_start"]
    return {
        "attn_norm": (D,),
        "wq": (q, D),
        "wk": (kv, D) if writes else None,
        "wv": (kv, D) if writes else None,
        "wo": (D, q),
        "ffn_norm": (D,),
        "w_gate": (F, D),
        "w_up": (F, D),
        "w_down": (D, F),
        "ple_gate": (P, D) if P > 0 else None,
        "ple_proj": (D, P) if P > 0 else None,
    }


def draw_q4_0(rng: np.random.Generator, n_rows: int, n_cols: int) -> np.ndarray:
    """Q4_0 blocks for an [n_rows, n_cols] matrix: uint8 [n_rows, n_cols/32, 18]."""
    assert n_cols % 32 == 0
    nb = n_rows * (n_cols // 32)
    d = np.abs(rng.normal(0.0, 0.002, nb)).astype(np.float16)
    nib = rng.integers(0, 16, size=(nb, 32), dtype=np.uint8)
    out = np.empty((nb, 18), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    out[:, 2:18] = nib[:, :16] | (nib[:, 16:] << 4)
    return out.reshape(n_rows, n_cols // 32, 18)


def draw_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.normal(0.0, 0.02, shape).astype(np.float32)


@dataclass
class Weights:
    cfg: dict
    tok_embd: np.ndarray            # q4_0 [V, D/32, 18] or f32 [V, D]
    ple_embd: np.ndarray | None     # q4_0 [V, L*P/32, 18] or f32 [V, L*P]
    out_norm: np.ndarray            # f32 [D]
    layers: list[dict] = field(default_factory=list)


def make_weights(cfg: dict, seed: int = WEIGHT_SEED) -> Weights:
    """Draw every tensor in a fixed order: tok_embd, ple_embd, out_norm, then
    per layer in LAYER_KEYS order, skipping absent tensors.  Norm gains are
    always fp32 N(0, 0.02); matrices follow cfg['wtype']."""
    rng = np.random.default_rng(seed)
    D, V, L, P = cfg["d_model"], cfg["vocab"], cfg["n_layer"], cfg["ple_dim"]
    q4 = cfg["wtype"] == "q4_0"

    def mat(n, k):
        return draw_q4_0(rng, n, k) if q4 else draw_f32(rng, (n, k))

    tok = mat(V, D)
    ple = mat(V, L * P) if P > 0 else None
    out_norm = draw_f32(rng, (D,))
    layers = []
    for il in range(L):
        lw = {}
        for key, shp in layer_shapes(cfg, il).items():
            if shp is None:
                lw[key] = None
            elif len(shp) == 1:
                lw[key] = draw_f32(rng, shp)
            else:
                lw[key] = mat(*shp)
        layers.append(lw)
    return Weights(cfg=cfg, tok_embd=tok, ple_embd=ple, out_norm=out_norm, layers=layers)


def make_tokens(cfg: dict, n: int, seed: int = TOKEN_SEED) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, cfg["vocab"], size=n).astype(np.int32)


def split_ubatches(tokens: np.ndarray, ubatch: int) -> list[np.ndarray]:
    return [tokens[i:i + ubatch] for i in range(0, len(tokens), ubatch)]
