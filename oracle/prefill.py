"""Plain fp32 prefill of a decoder whose last layers are KV-shared.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module.

Every step is written out with numpy in the order the method states it.  The
matrix products use numpy's matmul as a library primitive; there is no
blocking, fusion or reordering beyond that.  Activations stay fp32; the KV
cache is FP16 (round to nearest even), as the PicoLM KV-cache article's "file"
paragraph states the cache stores half-precision keys and values.
"""
from __future__ import annotations

import math
import struct

import numpy as np

F32 = np.float32

# ---------------------------------------------------------------------------
# weight formats


def q4_0_decode(blocks: np.ndarray) -> np.ndarray:
    """Q4_0 blocks uint8 [..., nb, 18] -> fp32 [..., nb*32].

    One block: fp16 scale d (little endian), then 16 bytes; byte j holds
    element j in its low nibble and element j+16 in its high nibble; the value
    is d * (nibble - 8).  The product of an fp16 and a 4-bit integer is exact
    in fp32, so this decode is exact.
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(F32)
    qs = blocks[..., 2:18]
    q = np.empty(blocks.shape[:-1] + (32,), dtype=F32)
    q[..., :16] = qs & 0x0F          # element j: low nibble of byte j
    q[..., 16:] = qs >> 4            # element j+16: high nibble of byte j
    q -= F32(8.0)
    q *= d[..., None]
    return q.reshape(*blocks.shape[:-2], blocks.shape[-2] * 32)


def as_f32_matrix(w: np.ndarray) -> np.ndarray:
    """A weight matrix in either storage format as fp32 [rows, cols]."""
    if w.dtype == np.uint8:
        return q4_0_decode(w)
    return np.asarray(w, dtype=F32)


def rows_f32(table: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Selected rows of an embedding table, decoded to fp32."""
    return as_f32_matrix(table[rows])


# ---------------------------------------------------------------------------
# per-row operations


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * (1 + g), per row (gain read as 1+g)."""
    x = np.asarray(x, dtype=F32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=F32)
    return (x / np.sqrt(ms + F32(eps))) * (F32(1.0) + g.astype(F32))


def rope_tables(pos: np.ndarray, head_dim: int, base: float):
    """cos/sin of pos * base^(-2i/hd) for i < hd/2; angle in fp64, result fp32."""
    half = head_dim // 2
    inv = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def rope_neox(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate x [M, H, hd] by its row position, pairing element i with i+hd/2."""
    M, H, hd = x.shape
    half = hd // 2
    cos, sin = rope_tables(pos, hd, base)
    c = cos[:, None, :]
    s = sin[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1).astype(F32)


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh approximation: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, dtype=F32)
    k = F32(math.sqrt(2.0 / math.pi))
    return F32(0.5) * x * (F32(1.0) + np.tanh(k * (x + F32(0.044715) * x * x * x)))


def silu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=F32)
    return x / (F32(1.0) + np.exp(-x))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention.

    q [M, Hq, hd] fp32; k, v [n_keys, Hkv, hd] (any float type, read as fp32);
    pos [M] absolute positions.  Query head h uses KV head h // (Hq/Hkv); row m
    sees keys j <= pos[m]; scores are q.k / sqrt(hd); softmax takes the max
    first, then the exponentials and their sum.
    """
    M, Hq, hd = q.shape
    n_keys, Hkv, _ = k.shape
    group = Hq // Hkv
    kf = k.astype(F32)
    vf = v.astype(F32)
    hidden = np.arange(n_keys)[None, :] > np.asarray(pos)[:, None]
    scale = F32(1.0 / math.sqrt(hd))
    out = np.empty((M, Hq, hd), dtype=F32)
    for h in range(Hq):
        g = h // group
        s = (q[:, h, :] @ kf[:, g, :].T) * scale
        s[hidden] = -np.inf
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True, dtype=F32)
        out[:, h, :] = (p @ vf[:, g, :]) / l
    return out


# ---------------------------------------------------------------------------
# the pruning predicate and the KV image


def prune_shared(n_layer: int, n_layer_kv_from_start: int, *, n_seq_max: int = 1,
                 embeddings: bool = False, embeddings_layer_inp=None,
                 crop_before_nextn: bool = True) -> bool:
    """The condition under which non-output rows are pruned before the first
    KV-shared layer (Gemma 4 prefill news, section 1 listing): a NextN crop is
    allowed, 0 < n_layer_kv_from_start < n_layer, no embeddings output, a
    single sequence, and no per-layer embedding input requested for any layer
    from n_layer_kv_from_start up to and including n_layer."""
    ok = (crop_before_nextn and 0 < n_layer_kv_from_start < n_layer
          and not embeddings and n_seq_max == 1)
    if ok and embeddings_layer_inp is not None:
        for il in range(n_layer_kv_from_start, n_layer + 1):
            if embeddings_layer_inp[il]:
                ok = False
                break
    return ok


KV_MAGIC = b"KVCP"
KV_HEADER_BYTES = 16


def kv_image_bytes(n_layers_written: int, n_pos: int, kv_dim: int) -> int:
    """Header plus FP16 keys then values: 16 + 2 * L * N * kv_dim * 2 bytes."""
    return KV_HEADER_BYTES + 2 * n_layers_written * n_pos * kv_dim * 2


class KVImageError(ValueError):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


# ---------------------------------------------------------------------------
# the model


class OracleContext:
    """One sequence's prefill state: the FP16 cache of the writing layers and
    the number of positions already in it."""

    def __init__(self, cfg: dict, weights, max_ctx: int, cache_weights: bool = True):
        self.cfg = cfg
        self.w = weights
        self.max_ctx = max_ctx
        self.L = cfg["n_layer"]
        self.S = cfg["n_layer_kv_from_start"]
        self.L_w = min(self.S, self.L)
        self.Hq, self.Hkv, self.hd = cfg["n_head"], cfg["n_head_kv"], cfg["head_dim"]
        self.kv_dim = self.Hkv * self.hd
        self.K = np.zeros((self.L_w, max_ctx, self.Hkv, self.hd), dtype=np.float16)
        self.V = np.zeros((self.L_w, max_ctx, self.Hkv, self.hd), dtype=np.float16)
        self.n_pos = 0
        self._wcache = {} if cache_weights else None

    # -- weights ------------------------------------------------------------
    def mat(self, il: int, key: str) -> np.ndarray:
        if self._wcache is not None and (il, key) in self._wcache:
            return self._wcache[(il, key)]
        m = as_f32_matrix(self.w.layers[il][key])
        if self._wcache is not None:
            self._wcache[(il, key)] = m
        return m

    def head_matrix(self) -> np.ndarray:
        key = (-1, "tok_embd")
        if self._wcache is not None and key in self._wcache:
            return self._wcache[key]
        m = as_f32_matrix(self.w.tok_embd)
        if self._wcache is not None:
            self._wcache[key] = m
        return m

    # -- one layer ------------------------------------------------------------
    def _layer(self, il: int, x: np.ndarray, ple: np.ndarray | None, pos: np.ndarray,
               kv_len: int) -> np.ndarray:
        cfg, lw = self.cfg, self.w.layers[il]
        M = x.shape[0]
        eps, base = cfg["rms_eps"], cfg["rope_base"]
        y = rmsnorm(x, lw["attn_norm"], eps)
        q = (y @ self.mat(il, "wq").T).reshape(M, self.Hq, self.hd)
        q = rope_neox(q, pos, base)
        if il < self.S:
            k = (y @ self.mat(il, "wk").T).reshape(M, self.Hkv, self.hd)
            k = rope_neox(k, pos, base)
            v = (y @ self.mat(il, "wv").T).reshape(M, self.Hkv, self.hd)
            self.K[il, pos] = k.astype(np.float16)
            self.V[il, pos] = v.astype(np.float16)
            src = il
        else:
            src = cfg["kv_src"][il]
        o = attention(q, self.K[src, :kv_len], self.V[src, :kv_len], pos)
        x = x + o.reshape(M, self.Hq * self.hd) @ self.mat(il, "wo").T
        y = rmsnorm(x, lw["ffn_norm"], eps)
        g = y @ self.mat(il, "w_gate").T
        u = y @ self.mat(il, "w_up").T
        act = gelu_tanh(g) if cfg["ffn"] == "geglu" else silu(g)
        x = x + (act * u) @ self.mat(il, "w_down").T
        if cfg["ple_dim"] > 0:
            gate = gelu_tanh(x @ self.mat(il, "ple_gate").T) * ple[:, il, :]
            x = x + gate @ self.mat(il, "ple_proj").T
        return x.astype(F32)

    # -- one ubatch ----------------------------------------------------------
    def ubatch(self, tokens: np.ndarray, is_last: bool, prune: bool = False, embeddings: bool = False,
               embd_layer_inp=None, capture: dict | None = None):
        """Run one ubatch at positions n_pos .. n_pos+T-1.

        prune=False is the plain definition: every row passes every layer.
        prune=True is the pruned ordering: before layer n_layer_kv_from_start
        only the output row (the last row of the last ubatch) is kept, and an
        intermediate ubatch stops there -- when the pruning condition holds,
        which embeddings (an embeddings output of every row) and
        embd_layer_inp (n_layer + 1 flags: the hidden state entering layer il
        of every row, il == n_layer the final one) can make false.  With
        `capture` a dict, the requested outputs are stored in it: capture[il]
        the rows entering layer il (fp32 [T, d_model]), capture["embd"] the
        embeddings output rmsnorm(final hidden state) * (1 + g_out).  Returns
        fp32 logits [vocab] of the last row when is_last, else None.
        """
        cfg = self.cfg
        tokens = np.asarray(tokens, dtype=np.int64)
        T = len(tokens)
        if T <= 0 or self.n_pos + T > self.max_ctx:
            raise ValueError("ubatch does not fit the context")
        if tokens.min() < 0 or tokens.max() >= cfg["vocab"]:
            raise ValueError("token id out of range")
        pos0 = self.n_pos
        pos = pos0 + np.arange(T)
        kv_len = pos0 + T
        x = rows_f32(self.w.tok_embd, tokens)
        ple = None
        P = cfg["ple_dim"]
        if P > 0:
            ple = rows_f32(self.w.ple_embd, tokens).reshape(T, self.L, P) * F32(1.0 / math.sqrt(P))
        pruning = prune and prune_shared(self.L, self.S, embeddings=embeddings,
                                         embeddings_layer_inp=embd_layer_inp)
        want = embd_layer_inp if embd_layer_inp is not None else [False] * (self.L + 1)
        stopped = False
        for il in range(self.L):
            if pruning and il == self.S:
                if not is_last:
                    stopped = True
                    break
                keep = [T - 1]
                x, pos = x[keep], pos[keep]
                ple = ple[keep] if ple is not None else None
            if capture is not None and want[il]:
                capture[il] = x.copy()
            x = self._layer(il, x, ple, pos, kv_len)
        self.n_pos = kv_len
        if capture is not None and not stopped:
            if want[self.L]:
                capture[self.L] = x.copy()
            if embeddings:
                capture["embd"] = rmsnorm(x, self.w.out_norm, cfg["rms_eps"])
        if not is_last:
            return None
        y = rmsnorm(x[-1:], self.w.out_norm, cfg["rms_eps"])
        return (y @ self.head_matrix().T)[0].astype(F32)

    def prefill(self, tokens: np.ndarray, ubatch: int, prune: bool = False) -> np.ndarray:
        chunks = [tokens[i:i + ubatch] for i in range(0, len(tokens), ubatch)]
        out = None
        for i, c in enumerate(chunks):
            out = self.ubatch(c, is_last=(i == len(chunks) - 1), prune=prune)
        return out

    def reset(self):
        self.n_pos = 0

    # -- KV image ------------------------------------------------------------
    def kv_save(self) -> bytes:
        """Header (magic, n_pos, writing layers, kv_dim as int32 LE), then the
        FP16 keys [L_w][n_pos][kv_dim], then the FP16 values."""
        n = self.n_pos
        hdr = KV_MAGIC + struct.pack("<iii", n, self.L_w, self.kv_dim)
        k = self.K[:, :n].reshape(self.L_w, n, self.kv_dim)
        v = self.V[:, :n].reshape(self.L_w, n, self.kv_dim)
        return hdr + k.tobytes() + v.tobytes()

    def kv_load(self, img: bytes, n_pos: int):
        """Restore the first n_pos positions from an image.  A wrong magic,
        a layer or KV-dim mismatch, or n_pos beyond the image or the context
        is refused and leaves the state unchanged."""
        if len(img) < KV_HEADER_BYTES or img[:4] != KV_MAGIC:
            raise KVImageError("magic", "not a KV image")
        n_img, l_img, kv_img = struct.unpack("<iii", img[4:16])
        if l_img != self.L_w or kv_img != self.kv_dim:
            raise KVImageError("shape", "layers or kv_dim do not match the model")
        if n_pos < 0 or n_pos > n_img or n_pos > self.max_ctx or n_img < 0:
            raise KVImageError("range", "position count out of range")
        if len(img) < kv_image_bytes(self.L_w, n_img, self.kv_dim):
            raise KVImageError("range", "image shorter than its header says")
        seg = n_img * self.kv_dim
        body = np.frombuffer(img, dtype=np.float16, offset=KV_HEADER_BYTES,
                             count=2 * self.L_w * seg).reshape(2, self.L_w, n_img, self.Hkv, self.hd)
        self.K[:, :n_pos] = body[0, :, :n_pos]
        self.V[:, :n_pos] = body[1, :, :n_pos]
        self.n_pos = n_pos
