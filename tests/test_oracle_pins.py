"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute: values
written by hand from a definition (tests/golden), closed forms, textbook
values, a published error bound, or a brute-force float64 loop on tiny
inputs.
"""
import math
import os
import struct

import numpy as np
import pytest

import oracle
from oracle.prefill import KVImageError, OracleContext, as_f32_matrix, rope_tables, rows_f32
from prefill_kv_shared_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _half_bits_to_f64(bits: int) -> float:
    """IEEE-754 binary16 decoded by its definition (independent of numpy)."""
    s = -1.0 if bits >> 15 else 1.0
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    if e == 0:
        return s * m * 2.0 ** -24
    assert e != 31
    return s * (1.0 + m / 1024.0) * 2.0 ** (e - 15)


# ---------------------------------------------------------------------------
# Q4_0


def test_q4_0_hand_built_block():
    rows = {r[0]: r[1:] for r in _golden_lines("q4_0_block.txt")}
    blk = np.array([int(b, 16) for b in rows["bytes"]], dtype=np.uint8).reshape(1, 1, 18)
    want = np.array([float(v) for v in rows["values"]])
    got = oracle.q4_0_decode(blk)[0]
    assert got.dtype == np.float32
    np.testing.assert_array_equal(got.astype(np.float64), want)


@pytest.mark.parametrize("dbits", [0x3800, 0x1A3C, 0x0003, 0x03FF, 0x2E66, 0x7BFF])
def test_q4_0_exact_for_every_nibble(dbits):
    """All 16 nibble values in both halves: decode == d*(n-8) in float64."""
    d = _half_bits_to_f64(dbits)
    nib = np.arange(32) % 16
    qs = (nib[:16] | (nib[16:][::-1] << 4)).astype(np.uint8)
    hi_vals = nib[16:][::-1]
    blk = np.concatenate([np.array([dbits & 0xFF, dbits >> 8], dtype=np.uint8), qs]).reshape(1, 1, 18)
    got = oracle.q4_0_decode(blk)[0].astype(np.float64)
    want = np.array([d * (n - 8) for n in nib[:16]] + [d * (n - 8) for n in hi_vals])
    np.testing.assert_array_equal(got, want)


def test_q4_0_matrix_layout():
    """Row r, column c of a decoded matrix is element c%32 of block c//32 of row r."""
    rng = np.random.default_rng(5)
    w = synth.draw_q4_0(rng, 3, 64)
    m = as_f32_matrix(w)
    assert m.shape == (3, 64)
    for r in range(3):
        for c in (0, 15, 16, 31, 32, 47, 48, 63):
            b = w[r, c // 32]
            d = _half_bits_to_f64(int(b[0]) | (int(b[1]) << 8))
            j = c % 32
            n = (b[2 + j] & 0xF) if j < 16 else (b[2 + j - 16] >> 4)
            assert float(m[r, c]) == d * (int(n) - 8)


def test_q4_0_row_gather():
    """The embedding gather picks whole rows by token id (repeats and the
    last row included), each decoded by the definition."""
    rng = np.random.default_rng(8)
    table = synth.draw_q4_0(rng, 5, 64)
    ids = np.array([4, 0, 4, 2])
    got = rows_f32(table, ids)
    assert got.shape == (4, 64) and got.dtype == np.float32
    for t, r in enumerate(ids):
        for c in range(64):
            b = table[r, c // 32]
            d = _half_bits_to_f64(int(b[0]) | (int(b[1]) << 8))
            j = c % 32
            n = (b[2 + j] & 0xF) if j < 16 else (b[2 + j - 16] >> 4)
            assert float(got[t, c]) == d * (int(n) - 8)


# ---------------------------------------------------------------------------
# per-row operations


@pytest.mark.parametrize("c", [0.5, 3.0, -2.0])
def test_rmsnorm_constant_vector(c):
    rng = np.random.default_rng(0)
    g = rng.normal(0, 0.02, 64).astype(np.float32)
    x = np.full((2, 64), c, dtype=np.float32)
    eps = 1e-6
    want = c / math.sqrt(c * c + eps) * (1.0 + g.astype(np.float64))
    got = oracle.rmsnorm(x, g, eps)
    np.testing.assert_allclose(got[0], want, rtol=1e-6)
    np.testing.assert_allclose(got[1], want, rtol=1e-6)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (4, 256)).astype(np.float32)
    g = np.zeros(256, dtype=np.float32)
    y = oracle.rmsnorm(x, g, 0.0)
    np.testing.assert_allclose(np.sqrt((y.astype(np.float64) ** 2).mean(-1)), 1.0, rtol=1e-5)
    np.testing.assert_allclose(oracle.rmsnorm(7.0 * x, g, 0.0), y, rtol=1e-5, atol=1e-6)


def test_rope_golden_pairs():
    rows = _golden_lines("rope_pairs.txt")
    for r in rows:
        vals = [float(v) for v in r]
        x = np.array(vals[:4], dtype=np.float32).reshape(1, 1, 4)
        got = oracle.rope_neox(x, np.array([1]), 10000.0)[0, 0]
        np.testing.assert_allclose(got, vals[4:], rtol=1e-6, atol=1e-7)


def test_rope_position_zero_is_identity_and_norms_kept():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(3, 2, 64)).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope_neox(x, np.zeros(3, int), 10000.0), x)
    y = oracle.rope_neox(x, np.array([5, 100, 7777]), 10000.0)
    half = 32
    n_in = x[..., :half] ** 2 + x[..., half:] ** 2
    n_out = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-5, atol=1e-6)


def test_rope_scores_depend_on_offset_only():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(1, 1, 256)).astype(np.float32)
    k = rng.normal(size=(1, 1, 256)).astype(np.float32)
    def score(pq, pk):
        a = oracle.rope_neox(q, np.array([pq]), 10000.0).astype(np.float64)
        b = oracle.rope_neox(k, np.array([pk]), 10000.0).astype(np.float64)
        return float((a * b).sum())
    s0 = score(50, 13)
    assert abs(score(87, 50) - s0) < 1e-4 * max(1.0, abs(s0))
    assert abs(score(50 + 4096, 13 + 4096) - s0) < 1e-3 * max(1.0, abs(s0))
    assert abs(score(51, 13) - s0) > 1e-3  # the offset matters


def test_rope_table_fp64_angle():
    cos, sin = rope_tables(np.array([32767]), 256, 10000.0)
    assert abs(float(cos[0, 0]) - math.cos(32767.0)) < 1e-7
    assert abs(float(sin[0, 127]) - math.sin(32767.0 * 10000.0 ** (-254 / 256))) < 1e-7


def test_gelu_tanh_within_published_bound_of_exact_gelu():
    """The tanh form stays within about 4.7e-4 of x*Phi(x) everywhere."""
    erf = pytest.importorskip("scipy.special").erf
    x = np.linspace(-12, 12, 200001).astype(np.float32)
    exact = 0.5 * x.astype(np.float64) * (1.0 + erf(x.astype(np.float64) / math.sqrt(2.0)))
    dev = np.abs(oracle.gelu_tanh(x).astype(np.float64) - exact)
    assert dev.max() < 5.0e-4
    assert dev.max() > 4.0e-4   # the cubic term is there (without it: ~2e-2)
    assert oracle.gelu_tanh(np.float32(0.0)) == 0.0
    assert abs(float(oracle.gelu_tanh(np.float32(1.0))) - 0.8411919906082768) < 1e-6


def test_silu_values():
    assert oracle.silu(np.float32(0.0)) == 0.0
    assert abs(float(oracle.silu(np.float32(1.0))) - 0.7310585786300049) < 1e-6
    assert abs(float(oracle.silu(np.float32(30.0))) - 30.0) < 1e-5
    assert abs(float(oracle.silu(np.float32(-30.0)))) < 1e-10


# ---------------------------------------------------------------------------
# attention


def _attention_brute(q, k, v, pos):
    M, Hq, hd = q.shape
    n, Hkv, _ = k.shape
    out = np.zeros((M, Hq, hd))
    for m in range(M):
        for h in range(Hq):
            g = (h * Hkv) // Hq
            s = []
            for j in range(n):
                if j <= pos[m]:
                    s.append(sum(float(q[m, h, i]) * float(k[j, g, i]) for i in range(hd)) / math.sqrt(hd))
            mx = max(s)
            e = [math.exp(a - mx) for a in s]
            z = sum(e)
            for j in range(len(s)):
                for i in range(hd):
                    out[m, h, i] += e[j] / z * float(v[j, g, i])
    return out


def test_attention_brute_force():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(3, 4, 8)).astype(np.float32)
    k = rng.normal(size=(6, 2, 8)).astype(np.float16)
    v = rng.normal(size=(6, 2, 8)).astype(np.float16)
    pos = np.array([0, 3, 5])
    got = oracle.attention(q, k, v, pos)
    np.testing.assert_allclose(got, _attention_brute(q, k, v, pos), rtol=1e-5, atol=1e-6)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(2, 2, 16)).astype(np.float32)
    v = rng.normal(size=(5, 1, 16)).astype(np.float16)
    k = rng.normal(size=(5, 1, 16)).astype(np.float16)
    # position 0 sees only key 0: output is V0
    o = oracle.attention(q, k, v, np.array([0, 0]))
    np.testing.assert_allclose(o[:, 0], np.broadcast_to(v[0, 0].astype(np.float32), (2, 16)), rtol=1e-6)
    # equal keys: uniform weights, output is the mean of the visible values
    keq = np.broadcast_to(k[:1], k.shape).copy()
    o = oracle.attention(q, keq, v, np.array([2, 4]))
    np.testing.assert_allclose(o[0, 1], v[:3, 0].astype(np.float64).mean(0), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(o[1, 0], v[:5, 0].astype(np.float64).mean(0), rtol=1e-5, atol=1e-6)
    # keys after the row's position change nothing
    k2 = k.copy(); v2 = v.copy()
    k2[3:] = 9.0; v2[3:] = -9.0
    np.testing.assert_array_equal(oracle.attention(q, k, v, np.array([1, 2])),
                                  oracle.attention(q, k2, v2, np.array([1, 2])))


# ---------------------------------------------------------------------------
# predicate and KV image


def test_prune_predicate_table():
    for r in _golden_lines("prune_predicate.txt"):
        L, S, nseq, emb, idx, want = (int(v) for v in r)
        inp = None
        if idx >= 0:
            inp = [False] * (L + 1)
            inp[idx] = True
        assert oracle.prune_shared(L, S, n_seq_max=nseq, embeddings=bool(emb),
                                   embeddings_layer_inp=inp) == bool(want), r


def test_kv_image_size_matches_article():
    kv = {r[0]: int(r[1]) for r in _golden_lines("kv_image_size.txt")}
    got = oracle.kv_image_bytes(kv["layers"], kv["n_pos"], kv["kv_dim"])
    assert got - 16 == kv["body_bytes"]
    assert round((got - 16) / 1024) == 550


def _kv_fixture():
    """The worked-example image of tests/golden/kv_image_small.txt, assembled
    in the fixture's own row order, and its cache contents by position."""
    rows = _golden_lines("kv_image_small.txt")
    hdr = {r[0]: r[1] for r in rows if r[0] not in ("K", "V")}
    n, L, kv = int(hdr["n_pos"]), int(hdr["n_layers"]), int(hdr["kv_dim"])
    body = [r for r in rows if r[0] in ("K", "V")]
    img = hdr["magic"].encode() + struct.pack("<iii", n, L, kv)
    cache = {"K": np.zeros((L, n, kv)), "V": np.zeros((L, n, kv))}
    for r in body:
        vals = [float(x) for x in r[3:]]
        assert len(vals) == kv
        img += np.array(vals, dtype="<f2").tobytes()
        cache[r[0]][int(r[1]), int(r[2])] = vals
    return img, n, L, kv, cache


def _kv_oracle(L, kv, max_ctx):
    cfg = dict(n_layer=L + 1, n_layer_kv_from_start=L, n_head=2, n_head_kv=1, head_dim=kv)
    return OracleContext(cfg, None, max_ctx)


def test_kv_image_layout_matches_worked_example():
    """The oracle's image is byte for byte the worked example (keys of every
    layer and position first, then values), and restoring a prefix of it
    reads back those positions."""
    img, n, L, kv, cache = _kv_fixture()
    o = _kv_oracle(L, kv, 8)
    o.K[:, :n, 0, :] = cache["K"]
    o.V[:, :n, 0, :] = cache["V"]
    o.n_pos = n
    assert o.kv_save() == img
    assert len(img) == oracle.kv_image_bytes(L, n, kv)
    r = _kv_oracle(L, kv, 8)
    r.kv_load(img, 2)
    assert r.n_pos == 2
    np.testing.assert_array_equal(r.K[:, :2, 0, :].astype(np.float64), cache["K"][:, :2])
    np.testing.assert_array_equal(r.V[:, :2, 0, :].astype(np.float64), cache["V"][:, :2])
    assert not r.K[:, 2:].any() and not r.V[:, 2:].any()


# ---------------------------------------------------------------------------
# whole model on a micro configuration


MICRO = dict(name="micro", n_layer=3, n_layer_kv_from_start=2, d_model=8, n_head=2,
             n_head_kv=1, head_dim=4, ffn_dim=8, ffn="geglu", vocab=11, ple_dim=4,
             rms_eps=1e-6, rope_base=10000.0, kv_src=[-1, -1, 1], wtype="f32")


def _model_brute(cfg, w, tokens, states=None):
    """Every step as float64 scalar loops, read straight from the method:
    pre-norm layers, Q/K/V projections, half-split RoPE, FP16 K/V, causal
    GQA attention over the own or the source layer's cache (query head h
    reads KV head h // (n_head / n_head_kv)), output projection, GeGLU or
    SwiGLU feed-forward, then the per-layer-embedding block when the model
    has one (ple_dim > 0).  With `states` a
    dict, also the rows entering each layer (states[il]), the final rows
    (states[n_layer]) and their output-normed form (states["embd"])."""
    D, L, S, P = cfg["d_model"], cfg["n_layer"], cfg["n_layer_kv_from_start"], cfg["ple_dim"]
    Hq, Hkv, hd, F = cfg["n_head"], cfg["n_head_kv"], cfg["head_dim"], cfg["ffn_dim"]
    T = len(tokens)

    def lin(Wm, vec):  # Wm [out, in]
        return [sum(float(Wm[o][i]) * vec[i] for i in range(len(vec))) for o in range(len(Wm))]

    def norm(vec, g):
        ms = sum(a * a for a in vec) / len(vec)
        r = 1.0 / math.sqrt(ms + cfg["rms_eps"])
        return [vec[i] * r * (1.0 + float(g[i])) for i in range(len(vec))]

    def rot(vec, p):
        half = hd // 2
        out = list(vec)
        for i in range(half):
            th = p * cfg["rope_base"] ** (-2.0 * i / hd)
            a, b = vec[i], vec[i + half]
            out[i] = a * math.cos(th) - b * math.sin(th)
            out[i + half] = a * math.sin(th) + b * math.cos(th)
        return out

    def gelu(a):
        return 0.5 * a * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (a + 0.044715 * a ** 3)))

    def silu(a):
        return a / (1.0 + math.exp(-a))

    act = gelu if cfg["ffn"] == "geglu" else silu

    f16 = lambda a: float(np.float16(a))
    x = [[float(w.tok_embd[t][i]) for i in range(D)] for t in tokens]
    ple = [[[float(w.ple_embd[t][il * P + p]) / math.sqrt(P) for p in range(P)]
            for il in range(L)] for t in tokens] if P > 0 else None
    cache = {}
    for il in range(L):
        lw = w.layers[il]
        if states is not None:
            states[il] = [list(r) for r in x]
        ys = [norm(x[t], lw["attn_norm"]) for t in range(T)]
        qs = []
        for t in range(T):
            qv = lin(lw["wq"], ys[t])
            qs.append([rot(qv[h * hd:(h + 1) * hd], t) for h in range(Hq)])
        if il < S:
            K, Vv = [], []
            for t in range(T):
                kv_ = lin(lw["wk"], ys[t]); vv = lin(lw["wv"], ys[t])
                K.append([[f16(a) for a in rot(kv_[g * hd:(g + 1) * hd], t)] for g in range(Hkv)])
                Vv.append([[f16(a) for a in vv[g * hd:(g + 1) * hd]] for g in range(Hkv)])
            cache[il] = (K, Vv)
            src = il
        else:
            src = cfg["kv_src"][il]
        K, Vv = cache[src]
        for t in range(T):
            o = []
            for h in range(Hq):
                g = h // (Hq // Hkv)
                s = [sum(qs[t][h][i] * K[j][g][i] for i in range(hd)) / math.sqrt(hd) for j in range(t + 1)]
                mx = max(s); e = [math.exp(a - mx) for a in s]; z = sum(e)
                o += [sum(e[j] / z * Vv[j][g][i] for j in range(t + 1)) for i in range(hd)]
            proj = lin(lw["wo"], o)
            x[t] = [x[t][i] + proj[i] for i in range(D)]
        for t in range(T):
            y = norm(x[t], lw["ffn_norm"])
            gg = lin(lw["w_gate"], y); uu = lin(lw["w_up"], y)
            h = [act(gg[f]) * uu[f] for f in range(F)]
            dn = lin(lw["w_down"], h)
            x[t] = [x[t][i] + dn[i] for i in range(D)]
            if P == 0:
                continue
            gate = lin(lw["ple_gate"], x[t])
            gp = [gelu(gate[p]) * ple[t][il][p] for p in range(P)]
            pp = lin(lw["ple_proj"], gp)
            x[t] = [x[t][i] + pp[i] for i in range(D)]
    if states is not None:
        states[L] = [list(r) for r in x]
        states["embd"] = [norm(r, w.out_norm) for r in x]
    y = norm(x[T - 1], w.out_norm)
    return np.array(lin(w.tok_embd, y))


def _micro_weights(scale=0.3, base=MICRO):
    cfg = dict(base)
    w = synth.make_weights(cfg, seed=11)
    # larger weights so every term moves the output visibly
    w.tok_embd = w.tok_embd * 40
    if w.ple_embd is not None:
        w.ple_embd = w.ple_embd * 40
    for lw in w.layers:
        for k, v in lw.items():
            if v is not None and v.ndim == 2:
                lw[k] = (v * (scale / 0.02)).astype(np.float32)
    return cfg, w


def test_micro_model_matches_brute_force():
    cfg, w = _micro_weights()
    tokens = np.array([3, 7, 0, 10, 5], dtype=np.int32)
    ctx = OracleContext(cfg, w, max_ctx=16)
    got = ctx.ubatch(tokens, is_last=True)
    want = _model_brute(cfg, w, tokens)
    np.testing.assert_allclose(got, want, rtol=2e-4, atol=2e-4 * np.abs(want).max())


def test_micro_model_hidden_states_match_brute_force():
    """The hidden states the oracle hands out (the rows entering a layer, the
    final rows, the embeddings output) against the float64 loops; asking
    for a state at or past the first KV-shared layer keeps every row there
    even with pruning asked for."""
    cfg, w = _micro_weights()
    tokens = np.array([3, 7, 0, 10, 5], dtype=np.int32)
    states = {}
    _model_brute(cfg, w, tokens, states)
    L = cfg["n_layer"]
    req = [False, True, True, True]
    cap = {}
    OracleContext(cfg, w, max_ctx=16).ubatch(tokens, is_last=True, prune=True, embeddings=True,
                                             embd_layer_inp=req, capture=cap)
    for key in (1, 2, L, "embd"):
        want = np.array(states[key])
        assert cap[key].shape == want.shape, key
        np.testing.assert_allclose(cap[key], want, rtol=2e-4, atol=2e-4 * np.abs(want).max())
    assert 0 not in cap


def test_micro_model_brute_force_catches_planted_mistake(monkeypatch):
    """A planted error in the oracle (wrong KV source layer) must break the pin."""
    cfg, w = _micro_weights()
    tokens = np.array([3, 7, 0, 10, 5], dtype=np.int32)
    bad = dict(cfg, kv_src=[-1, -1, 0])
    got = OracleContext(bad, w, max_ctx=16).ubatch(tokens, is_last=True)
    want = _model_brute(cfg, w, tokens)
    assert np.abs(got - want).max() > 1e-2 * np.abs(want).max()


# Two KV heads (query heads 0-1 read KV head 0, 2-3 read KV head 1),
# SwiGLU, no per-layer embeddings, and KV-shared layers that read the last
# writing layer of their own parity (layer 2 reads 0, layer 3 reads 1).
MICRO_GQA = dict(name="micro-gqa", n_layer=4, n_layer_kv_from_start=2, d_model=16, n_head=4,
                 n_head_kv=2, head_dim=4, ffn_dim=12, ffn="swiglu", vocab=13, ple_dim=0,
                 rms_eps=1e-6, rope_base=10000.0, kv_src=[-1, -1, 0, 1], wtype="f32")


def test_micro_gqa_swiglu_model_matches_brute_force():
    cfg, w = _micro_weights(base=MICRO_GQA)
    tokens = np.array([3, 12, 0, 7, 5, 9, 1], dtype=np.int32)
    want = _model_brute(cfg, w, tokens)
    got = OracleContext(cfg, w, max_ctx=16).ubatch(tokens, is_last=True)
    np.testing.assert_allclose(got, want, rtol=2e-4, atol=2e-4 * np.abs(want).max())
    # the pruned ordering over ragged ubatches (positions continue across
    # them; the intermediate ubatches stop before the first KV-shared layer)
    got = OracleContext(cfg, w, max_ctx=16).prefill(tokens, ubatch=3, prune=True)
    np.testing.assert_allclose(got, want, rtol=2e-4, atol=2e-4 * np.abs(want).max())


def test_micro_gqa_brute_force_catches_planted_head_mapping(monkeypatch):
    """A planted error in the oracle (query head h reading KV head h % n_head_kv
    instead of h // (n_head / n_head_kv)) must break the pin."""
    import oracle.prefill as op
    cfg, w = _micro_weights(base=MICRO_GQA)
    tokens = np.array([3, 12, 0, 7, 5, 9, 1], dtype=np.int32)
    want = _model_brute(cfg, w, tokens)
    real = op.attention
    perm = np.array([0, 2, 1, 3])  # its own inverse

    def planted(q, k, v, pos):
        return real(q[:, perm], k, v, pos)[:, perm]

    monkeypatch.setattr(op, "attention", planted)
    got = OracleContext(cfg, w, max_ctx=16).ubatch(tokens, is_last=True)
    assert np.abs(got - want).max() > 1e-2 * np.abs(want).max()


# ---------------------------------------------------------------------------
# whole-model invariants on the tiny configuration


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.config("tiny")
    return cfg, synth.make_weights(cfg)


def test_pruned_row_equals_unpruned_row(tiny):
    cfg, w = tiny
    tok = synth.make_tokens(cfg, 64)
    a = OracleContext(cfg, w, 128).ubatch(tok, True, prune=False)
    b = OracleContext(cfg, w, 128).ubatch(tok, True, prune=True)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-5 * np.abs(a).max())


@pytest.mark.parametrize("ub", [16, 7, 1])
def test_ubatch_split_invariance(tiny, ub):
    """The final row does not depend on how the prompt is cut into ubatches:
    16 (even), 7 (a ragged last ubatch of one token) and 1 (token by token,
    the form generation takes after the prompt)."""
    cfg, w = tiny
    tok = synth.make_tokens(cfg, 64)
    a = OracleContext(cfg, w, 128).prefill(tok, 64)
    b = OracleContext(cfg, w, 128).prefill(tok, ub, prune=True)
    c = OracleContext(cfg, w, 128).prefill(tok, ub, prune=False)
    # a different split rounds the fp32 sums differently, which can move an
    # FP16 cache entry by one unit: 1e-4 of the largest logit covers that
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-4 * np.abs(a).max())
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-4 * np.abs(a).max())


def test_empty_or_oversized_ubatch_is_refused(tiny):
    cfg, w = tiny
    a = OracleContext(cfg, w, 16)
    with pytest.raises(ValueError):
        a.ubatch(np.zeros(0, dtype=np.int32), True)
    with pytest.raises(ValueError):
        a.ubatch(synth.make_tokens(cfg, 17), True)
    assert a.n_pos == 0


def test_kv_restore_then_suffix_equals_full(tiny):
    cfg, w = tiny
    prefix = synth.make_tokens(cfg, 40, seed=1)
    suffix = synth.make_tokens(cfg, 12, seed=2)
    full = OracleContext(cfg, w, 128)
    want = full.prefill(np.concatenate([prefix, suffix]), 64)
    a = OracleContext(cfg, w, 128)
    a.prefill(prefix, 64)
    img = a.kv_save()
    assert len(img) == oracle.kv_image_bytes(2, 40, 64)
    b = OracleContext(cfg, w, 128)
    b.kv_load(img, 40)
    assert b.n_pos == 40
    got = b.ubatch(suffix, True)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-4 * np.abs(want).max())
    # a prefix of the image restores the same cached positions
    c = OracleContext(cfg, w, 128)
    c.kv_load(img, 25)
    np.testing.assert_array_equal(c.K[:, :25], a.K[:, :25])
    np.testing.assert_array_equal(c.V[:, :25], a.V[:, :25])


def test_kv_load_refusals_leave_state(tiny):
    cfg, w = tiny
    a = OracleContext(cfg, w, 64)
    a.prefill(synth.make_tokens(cfg, 20), 64)
    img = a.kv_save()
    b = OracleContext(cfg, w, 64)
    bad_magic = b"KVCQ" + img[4:]
    bad_shape = img[:8] + struct.pack("<i", 3) + img[12:]
    for blob, n, code in [(bad_magic, 10, "magic"), (bad_shape, 10, "shape"),
                          (img, 21, "range"), (img[:100], 10, "range")]:
        with pytest.raises(KVImageError) as e:
            b.kv_load(blob, n)
        assert e.value.code == code
        assert b.n_pos == 0 and not b.K.any()
    small = OracleContext(cfg, w, 16)
    with pytest.raises(KVImageError):
        small.kv_load(img, 20)


def test_all_layers_write_means_no_pruning():
    cfg = synth.scaled_config("tinyllama", n_layer=2, n_layer_kv_from_start=2, d_model=64,
                              n_head=4, n_head_kv=2, head_dim=16, ffn_dim=128, vocab=97)
    w = synth.make_weights(cfg)
    tok = synth.make_tokens(cfg, 10)
    a = OracleContext(cfg, w, 16).ubatch(tok, True, prune=False)
    b = OracleContext(cfg, w, 16).ubatch(tok, True, prune=True)
    np.testing.assert_array_equal(a, b)
