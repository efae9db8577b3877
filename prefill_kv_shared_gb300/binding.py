"""ctypes binding of the C ABI (include/prefill.h, include/prefill_ops.h).

Argument marshalling only: every step of the prefill pass runs in the CUDA
library.  There is no fallback: if the library is missing or a call fails,
the binding raises.  PyTorch is used by callers for device memory and
streams; this module passes raw pointers and sizes.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libprefill_kv_shared.so")

PF_OK = 0
PF_E_ARG = -1
PF_E_KV_MAGIC = -2
PF_E_KV_SHAPE = -3
PF_E_KV_RANGE = -4
PF_E_CUDA = -5
PF_E_DEVICE_TIMEOUT = -6
PF_E_DEVICE_TOKEN = -7
PF_E_NOMEM = -8
PF_E_IO = -9

PF_OUT_EMBD = -1

PF_PRUNE_OFF = 0
PF_PRUNE_ON = 1
PF_PRUNE_OFF_PLAIN = 2

PF_W_F32 = 0
PF_W_Q4_0 = 2
PF_FFN_GEGLU = 0
PF_FFN_SWIGLU = 1

# every symbol the headers declare
EXPORTS = (
    "prefill_create", "prefill_ubatch", "prefill_sync", "prefill_n_pos", "prefill_reset",
    "prefill_set_prune", "prefill_prune_active", "prefill_kv_image_bytes", "kv_save", "kv_load",
    "prefill_destroy", "prefill_last_error", "prefill_prune_predicate", "prefill_kv_header_check",
    "prefill_kv_image_bytes_for", "prefill_set_timing", "prefill_get_stats", "prefill_reset_stats",
    "pfop_linear_f32", "pfop_linear_resid", "pfop_linear_glu", "pfop_linear_ple", "pfop_linear_qkv",
    "pfop_attention", "pfop_rmsnorm", "pfop_embed", "pfop_kv_copy", "pfop_last_error", "pfop_linear_bench",
    "pfop_attention_split_noalloc", "pfop_attention_bench", "pfop_kv_copy_bench",
    "kv_save_file", "kv_load_file", "prefill_kv_file_check", "pfop_linear_row", "prefill_set_output",
    "pfop_linear_wait_test", "prefill_ubatch_seqs", "prefill_seq_n_pos", "prefill_seq_reset",
    "prefill_graph_capture", "prefill_graph_launch", "pfop_set_gemm_pairs", "pfop_qkv_row_order",
    "pfop_repack_q4",
)


class PrefillError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"status {code}: {msg}")
        self.code = code


class ModelDesc(C.Structure):
    _fields_ = [
        ("n_layer", C.c_int32), ("n_layer_kv_from_start", C.c_int32), ("d_model", C.c_int32),
        ("n_head", C.c_int32), ("n_head_kv", C.c_int32), ("head_dim", C.c_int32),
        ("ffn_dim", C.c_int32), ("vocab", C.c_int32), ("ple_dim", C.c_int32),
        ("ffn_kind", C.c_int32), ("wtype", C.c_int32), ("rms_eps", C.c_float),
        ("rope_base", C.c_float), ("kv_src", C.POINTER(C.c_int32)), ("max_ctx", C.c_int32),
        ("ubatch_max", C.c_int32), ("prune_shared_enable", C.c_int32), ("n_seq_max", C.c_int32),
        ("embeddings", C.c_int32), ("embd_layer_inp", C.POINTER(C.c_int32)),
    ]


KC_GEMM, KC_ATTN, KC_NORM, KC_OTHER, KC_GEMM_ROW, KC_ATTN_ROW = 0, 1, 2, 3, 4, 5
KC_NAMES = ("gemm", "attention", "norm", "other", "gemm_row", "attention_row")
KC_COUNT = len(KC_NAMES)


class Stats(C.Structure):
    _fields_ = [("launches", C.c_int64 * KC_COUNT), ("flops", C.c_double * KC_COUNT),
                ("bytes", C.c_double * KC_COUNT), ("timed", C.c_int64 * KC_COUNT), ("ms", C.c_double * KC_COUNT)]


class LayerWeights(C.Structure):
    _fields_ = [(k, C.c_void_p) for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate",
                                          "w_up", "w_down", "ple_gate", "ple_proj")]


class SeqRun(C.Structure):
    _fields_ = [("seq_id", C.c_int32), ("n_tokens", C.c_int32), ("is_last", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [("tok_embd", C.c_void_p), ("ple_embd", C.c_void_p), ("out_norm", C.c_void_p),
                ("layers", C.POINTER(LayerWeights))]


_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load the library (building it first if the sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path) or os.environ.get("PREFILL_REBUILD"):
        from . import build as _b
        _b.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not found: {path}")
    lib = C.CDLL(path)
    vp, i32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t
    sig = {
        "prefill_create": (C.c_int, [C.POINTER(ModelDesc), C.POINTER(Weights), vp, C.POINTER(vp)]),
        "prefill_ubatch": (C.c_int, [vp, vp, i32, i64, i32, vp]),
        "prefill_sync": (C.c_int, [vp]),
        "prefill_set_output": (C.c_int, [vp, i32, vp]),
        "prefill_ubatch_seqs": (C.c_int, [vp, vp, C.POINTER(SeqRun), i32, vp]),
        "prefill_seq_n_pos": (i64, [vp, i32]),
        "prefill_seq_reset": (C.c_int, [vp, i32]),
        "prefill_graph_capture": (C.c_int, [vp, vp, i32, i64, i32, vp]),
        "prefill_graph_launch": (C.c_int, [vp]),
        "prefill_n_pos": (i64, [vp]),
        "prefill_reset": (C.c_int, [vp]),
        "prefill_set_prune": (C.c_int, [vp, i32]),
        "prefill_prune_active": (C.c_int, [vp]),
        "prefill_kv_image_bytes": (i64, [vp, i64]),
        "kv_save": (C.c_int, [vp, vp, sz]),
        "kv_load": (C.c_int, [vp, vp, sz, i64]),
        "kv_save_file": (C.c_int, [vp, C.c_char_p]),
        "kv_load_file": (C.c_int, [vp, C.c_char_p, i64]),
        "prefill_kv_file_check": (C.c_int, [C.c_char_p, i32, i32, i64, C.POINTER(C.c_int64)]),
        "prefill_destroy": (None, [vp]),
        "prefill_last_error": (C.c_char_p, [vp]),
        "prefill_prune_predicate": (C.c_int, [C.POINTER(ModelDesc)]),
        "prefill_kv_header_check": (C.c_int, [vp, i32, i32, i64, i64, sz]),
        "prefill_kv_image_bytes_for": (i64, [i32, i64, i32]),
        "prefill_set_timing": (C.c_int, [vp, i32]),
        "prefill_get_stats": (C.c_int, [vp, C.POINTER(Stats)]),
        "prefill_reset_stats": (C.c_int, [vp]),
        "pfop_linear_f32": (C.c_int, [i32, vp, i32, i32, i32, vp, i32, i32, vp, vp]),
        "pfop_linear_resid": (C.c_int, [i32, vp, i32, i32, vp, i32, i32, vp, vp, vp]),
        "pfop_linear_glu": (C.c_int, [i32, vp, vp, i32, i32, i32, vp, i32, i32, vp, vp]),
        "pfop_linear_ple": (C.c_int, [i32, vp, i32, i32, vp, i32, i32, vp, i32, vp, vp]),
        "pfop_linear_qkv": (C.c_int, [i32, vp, vp, vp, i32, i32, i32, i32, f32, vp, i32, i32, i32, i32,
                                      vp, vp, vp, vp]),
        "pfop_attention": (C.c_int, [i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]),
        "pfop_rmsnorm": (C.c_int, [vp, i32, i32, i32, vp, f32, vp, vp, vp]),
        "pfop_embed": (C.c_int, [i32, vp, vp, i32, i32, i32, f32, vp, i32, vp, vp, vp]),
        "pfop_kv_copy": (C.c_int, [i32, vp, i64, vp, i64, i32, i64, vp, vp]),
        "pfop_last_error": (C.c_char_p, []),
        "pfop_attention_split_noalloc": (C.c_int, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
        "pfop_linear_bench": (C.c_int, [i32, vp, i32, i32, i32, i32, vp, i32, i32, vp, i32, i32,
                                        C.POINTER(C.c_float), vp]),
        "pfop_attention_bench": (C.c_int, [i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, i64, i32, i32,
                                           C.POINTER(C.c_float), vp]),
        "pfop_kv_copy_bench": (C.c_int, [i32, vp, i64, vp, i64, i32, i64, vp, i64, i32, i32,
                                         C.POINTER(C.c_float), vp]),
        "pfop_linear_row": (C.c_int, [i32, vp, i32, i32, i32, vp, vp, i32, C.POINTER(C.c_float), vp]),
        "pfop_linear_wait_test": (C.c_int, [i32, vp, i32, i32, i32, vp, i32, i32, vp, i32, vp]),
        "pfop_set_gemm_pairs": (C.c_int, [i32]),
        "pfop_qkv_row_order": (i32, [i32, i32, i32, i32, vp, i32]),
        "pfop_repack_q4": (i64, [vp, i32, i32, i32, vp, i64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a) -> int | None:
    """Address of a numpy array, a torch tensor or an int; None stays None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()


def _buffer(a, what: str, dtype: str | None = None, min_elems: int = 0) -> int | None:
    """Byte size of a numpy array or torch tensor handed to the library (None
    for a raw address), after checking what the library cannot see behind a
    pointer: contiguity, element type and element count."""
    if a is None or isinstance(a, int):
        return None
    if isinstance(a, np.ndarray):
        ok, n, dt, nbytes = a.flags["C_CONTIGUOUS"], a.size, str(a.dtype), a.nbytes
    else:
        ok, n, dt = a.is_contiguous(), a.numel(), str(a.dtype).replace("torch.", "")
        nbytes = n * a.element_size()
    if not ok:
        raise ValueError(f"{what}: buffer must be contiguous")
    if dtype is not None and dt != dtype:
        raise ValueError(f"{what}: element type must be {dtype}, got {dt}")
    if n < min_elems:
        raise ValueError(f"{what}: needs at least {min_elems} elements, got {n}")
    return nbytes


def _stream(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check_op(rc: int):
    if rc != PF_OK:
        raise PrefillError(rc, load().pfop_last_error().decode())


# ---------------------------------------------------------------------------
# model description from a config dict


def make_desc(cfg: dict, max_ctx: int, ubatch_max: int, prune: bool = True, n_seq_max: int = 1,
              embeddings: bool = False, layer_inp=None):
    """layer_inp: None, or n_layer + 1 flags requesting the hidden state
    entering each layer (the last one: the final hidden state)."""
    kv_src = (C.c_int32 * cfg["n_layer"])(*cfg["kv_src"])
    inp = None
    if layer_inp is not None:
        if len(layer_inp) != cfg["n_layer"] + 1:
            raise ValueError("layer_inp needs n_layer + 1 flags")
        inp = (C.c_int32 * (cfg["n_layer"] + 1))(*[1 if f else 0 for f in layer_inp])
    d = ModelDesc(
        n_layer=cfg["n_layer"], n_layer_kv_from_start=cfg["n_layer_kv_from_start"],
        d_model=cfg["d_model"], n_head=cfg["n_head"], n_head_kv=cfg["n_head_kv"],
        head_dim=cfg["head_dim"], ffn_dim=cfg["ffn_dim"], vocab=cfg["vocab"],
        ple_dim=cfg["ple_dim"], ffn_kind=PF_FFN_GEGLU if cfg["ffn"] == "geglu" else PF_FFN_SWIGLU,
        wtype=PF_W_Q4_0 if cfg["wtype"] == "q4_0" else PF_W_F32, rms_eps=cfg["rms_eps"],
        rope_base=cfg["rope_base"], kv_src=C.cast(kv_src, C.POINTER(C.c_int32)), max_ctx=max_ctx,
        ubatch_max=ubatch_max, prune_shared_enable=1 if prune else 0, n_seq_max=n_seq_max,
        embeddings=1 if embeddings else 0,
        embd_layer_inp=C.cast(inp, C.POINTER(C.c_int32)) if inp is not None else None)
    d._keep = (kv_src, inp)
    return d


def prune_predicate(cfg: dict, prune: bool = True, n_seq_max: int = 1, embeddings: bool = False,
                    layer_inp=None) -> bool:
    d = make_desc(cfg, 16, 16, prune, n_seq_max, embeddings, layer_inp)
    rc = load().prefill_prune_predicate(C.byref(d))
    if rc < 0:
        raise PrefillError(rc, "bad description")
    return bool(rc)


def kv_image_bytes_for(n_layers_written: int, n_pos: int, kv_dim: int) -> int:
    return int(load().prefill_kv_image_bytes_for(n_layers_written, n_pos, kv_dim))


def kv_file_check(path: str, n_layers_written: int, kv_dim: int, max_ctx: int) -> tuple[int, int]:
    """(status, positions) of a KV image file checked on the host only."""
    n = C.c_int64(-1)
    rc = load().prefill_kv_file_check(os.fsencode(path), n_layers_written, kv_dim, max_ctx, C.byref(n))
    return rc, n.value


def prefill_with_cache(ctx: "PrefillContext", tokens, ubatch: int, logits, path: str) -> int:
    """The PicoLM flow for a fixed prompt prefix (KV cache article, "usage"):
    if `path` holds a valid image of the prompt's first positions, restore it
    and prefill only the rest; otherwise prefill everything and save the
    cache to `path`.  Returns how many prompt positions came from the file.
    Whether the file was made from the same prefix is the caller's contract
    (the image stores no tokens)."""
    n = len(tokens)
    ctx.reset()
    start = 0
    if os.path.exists(path):
        rc, n_file = kv_file_check(path, ctx.n_layers_written, ctx.kv_dim, ctx.max_ctx)
        if rc == PF_OK and 0 < n_file < n and ctx.kv_load_file(path, n_file) == PF_OK:
            start = n_file
    for i in range(start, n, ubatch):
        ctx.ubatch(tokens[i:i + ubatch], i, i + ubatch >= n, logits)
    if start == 0:
        ctx.sync()
        ctx.kv_save_file(path)
    return start


def kv_header_check(header: bytes, n_layers_written: int, kv_dim: int, n_pos: int, max_ctx: int,
                    image_bytes: int) -> int:
    buf = (C.c_uint8 * 16).from_buffer_copy(header[:16].ljust(16, b"\0"))
    return int(load().prefill_kv_header_check(buf, n_layers_written, kv_dim, n_pos, max_ctx, image_bytes))


def qkv_row_order(Hq: int, Hkv: int, hd: int, with_kv: bool = True):
    """Stored row order of a Q|K|V projection (host only): the source row of
    each stored row in [Wq; Wk; Wv], -1 for padding."""
    import numpy as np
    cap = ((Hq + 2 * Hkv) * hd + 127) // 128 * 128
    out = np.empty(cap, dtype=np.int32)
    n = int(load().pfop_qkv_row_order(Hq, Hkv, hd, 1 if with_kv else 0, out.ctypes.data, cap))
    if n < 0:
        raise PrefillError(n, load().pfop_last_error().decode())
    return out[:n]


def repack_q4(w, bn: int):
    """A Q4_0 matrix [N][K/32][18] in the library's stored tile layout (host
    only), as bytes."""
    import numpy as np
    w = np.ascontiguousarray(w, dtype=np.uint8)
    N, K = w.shape[0], w.shape[1] * 32
    need = int(load().pfop_repack_q4(w.ctypes.data, N, K, bn, None, 0))
    if need < 0:
        raise PrefillError(need, load().pfop_last_error().decode())
    out = np.empty(need, dtype=np.uint8)
    rc = int(load().pfop_repack_q4(w.ctypes.data, N, K, bn, out.ctypes.data, need))
    if rc != need:
        raise PrefillError(rc, load().pfop_last_error().decode())
    return out


# ---------------------------------------------------------------------------
# a prefill context


class PrefillContext:
    """One sequence on the current CUDA device (see prefill.h)."""

    def __init__(self, weights, max_ctx: int, ubatch_max: int, prune: bool = True, stream=None,
                 n_seq_max: int = 1, embeddings: bool = False, layer_inp=None):
        lib = load()
        cfg = weights.cfg
        self.cfg = cfg
        self._desc = make_desc(cfg, max_ctx, ubatch_max, prune, n_seq_max, embeddings, layer_inp)
        keep = []

        def p(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            keep.append(a)
            return a.ctypes.data

        layers = (LayerWeights * cfg["n_layer"])()
        for il, lw in enumerate(weights.layers):
            for k in LayerWeights._fields_:
                setattr(layers[il], k[0], p(lw[k[0]]))
        w = Weights(tok_embd=p(weights.tok_embd), ple_embd=p(weights.ple_embd),
                    out_norm=p(weights.out_norm), layers=C.cast(layers, C.POINTER(LayerWeights)))
        h = C.c_void_p()
        rc = lib.prefill_create(C.byref(self._desc), C.byref(w), _stream(stream), C.byref(h))
        if rc != PF_OK:
            raise PrefillError(rc, lib.prefill_last_error(None).decode())
        self._h = h
        self._lib = lib
        self.vocab = cfg["vocab"]
        self.max_ctx = max_ctx
        self.n_layers_written = min(cfg["n_layer_kv_from_start"], cfg["n_layer"])
        self.kv_dim = cfg["n_head_kv"] * cfg["head_dim"]

    def _check(self, rc):
        if rc != PF_OK:
            raise PrefillError(rc, self._lib.prefill_last_error(self._h).decode())

    def ubatch(self, tokens, pos0: int, is_last: bool, logits=None):
        """tokens: numpy int32 (host) or an int32 device tensor; logits: fp32
        device tensor [vocab] (needed when is_last)."""
        if isinstance(tokens, np.ndarray):
            tokens = np.ascontiguousarray(tokens, dtype=np.int32)
            n = len(tokens)
        else:
            _buffer(tokens, "tokens", "int32")
            n = tokens.numel()
        if is_last:
            _buffer(logits, "logits", "float32", self.cfg["vocab"])
        self._check(self._lib.prefill_ubatch(self._h, _ptr(tokens), n, pos0, 1 if is_last else 0,
                                             _ptr(logits)))

    def set_output(self, which: int, dst):
        """Hidden-state output buffer: which = PF_OUT_EMBD (the embeddings
        output) or a layer index in [0, n_layer]; dst an fp32 device tensor
        with ubatch_max x d_model elements, or None."""
        if dst is not None:
            _buffer(dst, "dst", "float32")
        self._check(self._lib.prefill_set_output(self._h, which, _ptr(dst)))

    def ubatch_seqs(self, tokens, runs, logits=None):
        """Several sequences in one ubatch: runs = [(seq_id, n_tokens,
        is_last), ...] in the order of their tokens; tokens: numpy int32
        (host) or an int32 device tensor holding the runs' tokens one after
        another; logits: fp32 device tensor [number of is_last runs, vocab]."""
        arr = (SeqRun * len(runs))(*[SeqRun(int(q), int(n), 1 if last else 0) for q, n, last in runs])
        if isinstance(tokens, np.ndarray):
            tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        else:
            _buffer(tokens, "tokens", "int32")
        n_last = sum(1 for r in runs if r[2])
        if n_last:
            _buffer(logits, "logits", "float32", n_last * self.cfg["vocab"])
        self._check(self._lib.prefill_ubatch_seqs(self._h, _ptr(tokens), arr, len(runs), _ptr(logits)))

    def graph_capture(self, tokens, pos0: int, is_last: bool, logits=None):
        """Record one ubatch (tokens: int32 device tensor) for graph_launch."""
        _buffer(tokens, "tokens", "int32")
        if is_last:
            _buffer(logits, "logits", "float32", self.cfg["vocab"])
        self._check(self._lib.prefill_graph_capture(self._h, _ptr(tokens), tokens.numel(), pos0,
                                                    1 if is_last else 0, _ptr(logits)))

    def graph_launch(self):
        self._check(self._lib.prefill_graph_launch(self._h))

    def seq_n_pos(self, seq_id: int) -> int:
        return int(self._lib.prefill_seq_n_pos(self._h, seq_id))

    def seq_reset(self, seq_id: int):
        self._check(self._lib.prefill_seq_reset(self._h, seq_id))

    def sync(self):
        self._check(self._lib.prefill_sync(self._h))

    def reset(self):
        self._check(self._lib.prefill_reset(self._h))

    @property
    def n_pos(self) -> int:
        return int(self._lib.prefill_n_pos(self._h))

    def set_prune(self, enable):
        """True / PF_PRUNE_ON, False / PF_PRUNE_OFF, or PF_PRUNE_OFF_PLAIN."""
        mode = enable if isinstance(enable, int) and not isinstance(enable, bool) else (1 if enable else 0)
        self._check(self._lib.prefill_set_prune(self._h, mode))

    @property
    def prune_active(self) -> bool:
        return bool(self._lib.prefill_prune_active(self._h))

    def kv_image_bytes(self, n_pos: int) -> int:
        return int(self._lib.prefill_kv_image_bytes(self._h, n_pos))

    def kv_save(self, dst, nbytes: int):
        size = _buffer(dst, "dst")
        if size is not None and nbytes > size:
            raise ValueError(f"dst: nbytes {nbytes} exceeds the buffer's {size} bytes")
        self._check(self._lib.kv_save(self._h, _ptr(dst), nbytes))

    def kv_load(self, src, nbytes: int, n_pos: int):
        size = _buffer(src, "src")
        if size is not None and nbytes > size:
            raise ValueError(f"src: nbytes {nbytes} exceeds the buffer's {size} bytes")
        self._check(self._lib.kv_load(self._h, _ptr(src), nbytes, n_pos))

    def kv_save_file(self, path: str):
        self._check(self._lib.kv_save_file(self._h, os.fsencode(path)))

    def kv_load_file(self, path: str, n_pos: int = -1) -> int:
        """Restore a KV image file; returns the status (0, or the refusal code,
        in which case the cache is unchanged and a full prefill is due)."""
        rc = self._lib.kv_load_file(self._h, os.fsencode(path), n_pos)
        if rc not in (PF_OK, PF_E_KV_MAGIC, PF_E_KV_SHAPE, PF_E_KV_RANGE, PF_E_IO):
            self._check(rc)
        return rc

    def set_timing(self, enable: bool):
        self._check(self._lib.prefill_set_timing(self._h, 1 if enable else 0))

    def stats(self) -> dict:
        st = Stats()
        self._check(self._lib.prefill_get_stats(self._h, C.byref(st)))
        return {name: dict(launches=st.launches[i], flops=st.flops[i], bytes=st.bytes[i],
                           timed=st.timed[i], ms=st.ms[i]) for i, name in enumerate(KC_NAMES)}

    def reset_stats(self):
        self._check(self._lib.prefill_reset_stats(self._h))

    def close(self):
        if getattr(self, "_h", None):
            self._lib.prefill_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
