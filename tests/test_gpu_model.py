"""Whole prefill through the C ABI against the CPU oracle.

Acceptance: the output row's logits within 2e-2 * max|oracle logit| and the
same argmax as the oracle, and the pruned pass bit-identical to the
unpruned one.  Every model-level comparison records the GPU and oracle
argmax, the oracle's top-two gap and the error (printed, and appended as a
JSON line to the file named by PF_PARITY_LOG when that is set)."""
import json
import os

import numpy as np
import pytest

from oracle.prefill import OracleContext
from prefill_kv_shared_gb300 import binding, synth
from tests.gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu

TOL = 2e-2


def check_logits(got, want, case=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all()
    tol = TOL * np.abs(want).max()
    err = np.abs(got - want).max()
    top = np.sort(want)[::-1]
    rec = {"case": case, "gpu_argmax": int(np.argmax(got)), "oracle_argmax": int(np.argmax(want)),
           "oracle_top2_gap": float(top[0] - top[1]), "max_err": float(err), "tol": float(tol),
           "gpu_logit_at_oracle_argmax": float(got[int(np.argmax(want))])}
    print("parity", json.dumps(rec))
    path = os.environ.get("PF_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    assert err <= tol, f"max|err| {err:.4g} > {tol:.4g} ({rec})"
    assert rec["gpu_argmax"] == rec["oracle_argmax"], f"argmax differs from the oracle's ({rec})"
    return err / np.abs(want).max()


def run_gpu(weights, tokens, ubatch, prune, max_ctx=None, ctx=None):
    """prune: True, False or binding.PF_PRUNE_OFF_PLAIN."""
    cfg = weights.cfg
    own = ctx is None
    if own:
        ctx = binding.PrefillContext(weights, max_ctx=max_ctx or len(tokens), ubatch_max=ubatch, prune=bool(prune))
        if prune is binding.PF_PRUNE_OFF_PLAIN:
            ctx.set_prune(prune)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    chunks = synth.split_ubatches(tokens, ubatch)
    pos = ctx.n_pos
    for i, c in enumerate(chunks):
        ctx.ubatch(c, pos, i == len(chunks) - 1, logits)
        pos += len(c)
    ctx.sync()
    out = logits.cpu().numpy()
    if own:
        ctx.close()
    return out


@pytest.fixture(scope="module")
def gpu():
    need_gpu()
    from prefill_kv_shared_gb300 import build
    build.build()
    binding.load()


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.config("tiny")
    return synth.make_weights(cfg)


@pytest.fixture(scope="module")
def e2b():
    return synth.make_weights(synth.config("e2b"))


def test_tiny_matches_oracle(gpu, tiny):
    tok = synth.make_tokens(tiny.cfg, 64)
    want = OracleContext(tiny.cfg, tiny, 128).ubatch(tok, True)
    on = run_gpu(tiny, tok, 64, True)
    off = run_gpu(tiny, tok, 64, False)
    check_logits(on, want, "tiny-64")
    np.testing.assert_array_equal(on, off)


def test_tiny_ubatches_and_ragged(gpu, tiny):
    tok = synth.make_tokens(tiny.cfg, 61, seed=7)
    want = OracleContext(tiny.cfg, tiny, 128).prefill(tok, 16)
    on = run_gpu(tiny, tok, 16, True, max_ctx=128)
    off = run_gpu(tiny, tok, 16, False, max_ctx=128)
    check_logits(on, want, "tiny-61-ragged")
    np.testing.assert_array_equal(on, off)


def test_tiny_device_tokens(gpu, tiny):
    tok = synth.make_tokens(tiny.cfg, 64)
    host = run_gpu(tiny, tok, 64, True)
    ctx = binding.PrefillContext(tiny, max_ctx=64, ubatch_max=64)
    logits = torch.empty(tiny.cfg["vocab"], dtype=torch.float32, device="cuda")
    ctx.ubatch(torch.from_numpy(tok).cuda(), 0, True, logits)
    ctx.sync()
    np.testing.assert_array_equal(logits.cpu().numpy(), host)
    ctx.reset()
    bad = torch.from_numpy(tok).cuda()
    bad[5] = tiny.cfg["vocab"]
    ctx.ubatch(bad, 0, True, logits)
    with pytest.raises(binding.PrefillError) as e:
        ctx.sync()
    assert e.value.code == binding.PF_E_DEVICE_TOKEN
    ctx.close()


def test_e2b_512_matches_oracle(gpu, e2b):
    tok = synth.make_tokens(e2b.cfg, 512)
    on = run_gpu(e2b, tok, 512, True)
    off = run_gpu(e2b, tok, 512, False)
    np.testing.assert_array_equal(on, off)
    want = OracleContext(e2b.cfg, e2b, 512).ubatch(tok, True, prune=True)
    check_logits(on, want, "e2b-512")
    # the plain unpruned pass (every row through the prefill kernels) meets
    # the same acceptance; its bits may differ from the pruned pass's
    plain = run_gpu(e2b, tok, 512, binding.PF_PRUNE_OFF_PLAIN)
    check_logits(plain, want, "e2b-512 plain unpruned")


def test_e2b_2048_matches_oracle(gpu, e2b):
    """Four ubatches of 512: the first three stop before the KV-shared
    layers, the last carries one row through them.  Against the oracle's
    plain definition (every row through every layer), run once."""
    tok = synth.make_tokens(e2b.cfg, 2048)
    on = run_gpu(e2b, tok, 512, True)
    want = OracleContext(e2b.cfg, e2b, 2048).prefill(tok, 512, prune=False)
    check_logits(on, want, "e2b-2048")


@pytest.fixture(scope="module")
def e4b_scaled():
    # full E4B widths (d_model 2560, 8/2 heads of 256, GeGLU 10240, vocab
    # 32768, per-layer embedding 256), 6 layers: 0-3 write, 4 and 5 read
    # the last writing layer of their parity (2 and 3)
    return synth.make_weights(synth.scaled_config("e4b", n_layer=6, n_layer_kv_from_start=4))


def test_e4b_scaled_matches_oracle(gpu, e4b_scaled):
    """Two KV heads and the parity rule for the KV source, in ubatches of
    1024 (the first stops before the KV-shared layers)."""
    w = e4b_scaled
    assert w.cfg["kv_src"] == [-1, -1, -1, -1, 2, 3]
    tok = synth.make_tokens(w.cfg, 2048)
    on = run_gpu(w, tok, 1024, True)
    off = run_gpu(w, tok, 1024, False)
    np.testing.assert_array_equal(on, off)
    want = OracleContext(w.cfg, w, 2048).prefill(tok, 1024, prune=False)
    check_logits(on, want, "e4b-scaled-6L-2048")


@pytest.mark.parametrize("n", [2048, 8192, 32768])
def test_e2b_prune_bit_identical(gpu, e2b, n):
    tok = synth.make_tokens(e2b.cfg, n)
    on = run_gpu(e2b, tok, 512, True)
    off = run_gpu(e2b, tok, 512, False)
    assert np.isfinite(on).all()
    np.testing.assert_array_equal(on, off)


@pytest.fixture(scope="module")
def e4b():
    return synth.make_weights(synth.config("e4b"))


@pytest.mark.parametrize("n", [8192, 32768])
def test_e4b_prune_bit_identical(gpu, e4b, n):
    tok = synth.make_tokens(e4b.cfg, n)
    on = run_gpu(e4b, tok, 1024, True)
    off = run_gpu(e4b, tok, 1024, False)
    assert np.isfinite(on).all()
    np.testing.assert_array_equal(on, off)


@pytest.fixture(scope="module")
def tinyllama():
    return synth.make_weights(synth.config("tinyllama"))


def test_kv_restore_suffix_equals_full(gpu, tinyllama):
    """Cache a 500-token prefix as a KV image, restore it, prefill a 32-token
    suffix: the logits of the full 532-token prefill to rounding (the two runs
    cut the prompt into ubatches differently, and attention groups a row's
    key chunks by its launch's key count) and within tolerance of the
    oracle."""
    cfg = tinyllama.cfg
    prefix = synth.make_tokens(cfg, 500, seed=1)
    ctx = binding.PrefillContext(tinyllama, max_ctx=532, ubatch_max=512)
    assert not ctx.prune_active
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    ctx.ubatch(prefix, 0, False)
    nbytes = ctx.kv_image_bytes(500)
    assert nbytes == 16 + 2 * 22 * 500 * 256 * 2
    img = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ctx.kv_save(img, nbytes)
    ctx.sync()
    host_img = np.empty(nbytes, dtype=np.uint8)
    ctx.kv_save(host_img, nbytes)
    np.testing.assert_array_equal(host_img, img.cpu().numpy())
    orc = OracleContext(cfg, tinyllama, 532)
    orc.prefill(prefix, 512)
    for i in range(3):
        suffix = synth.make_tokens(cfg, 32, seed=2 + i)
        full = run_gpu(tinyllama, np.concatenate([prefix, suffix]), 512, True, max_ctx=532)
        ctx.reset()
        ctx.kv_load(img if i % 2 == 0 else host_img, nbytes, 500)
        assert ctx.n_pos == 500
        ctx.ubatch(suffix, 500, True, logits)
        ctx.sync()
        got = logits.cpu().numpy()
        assert np.abs(got - full).max() <= 2e-3 * np.abs(full).max()
        o2 = OracleContext(cfg, tinyllama, 532)
        o2.kv_load(orc.kv_save(), 500)
        check_logits(got, o2.ubatch(suffix, True), f"tinyllama-500+32 suffix {i}")
    ctx.close()


def test_kv_image_matches_oracle_image(gpu, tiny):
    """The GPU's KV image of a prefill against the oracle's image of the same
    prefill: the same header bytes, and a body whose FP16 keys and values
    (layer, position, element in the image's order) agree within the
    rounding the two computations differ by."""
    cfg = tiny.cfg
    tok = synth.make_tokens(cfg, 64)
    ctx = binding.PrefillContext(tiny, max_ctx=64, ubatch_max=64)
    ctx.ubatch(tok, 0, False)
    ctx.sync()
    n = ctx.kv_image_bytes(64)
    img = np.empty(n, dtype=np.uint8)
    ctx.kv_save(img, n)
    ctx.close()
    orc = OracleContext(cfg, tiny, 64)
    orc.ubatch(tok, False)
    want = np.frombuffer(orc.kv_save(), dtype=np.uint8)
    assert len(want) == n
    np.testing.assert_array_equal(img[:16], want[:16])
    got_b = img[16:].view(np.float16).astype(np.float64)
    want_b = want[16:].view(np.float16).astype(np.float64)
    assert np.abs(got_b - want_b).max() <= 2e-2 * np.abs(want_b).max()


def test_kv_partial_restore_matches_oracle_bytes(gpu, tiny):
    """Restore the first 3 positions of a 5-position image and save again:
    the GPU writes the same bytes as the oracle (a layout that put each
    layer's keys and values together would pick other positions)."""
    cfg = tiny.cfg
    L_w, kv = cfg["n_layer_kv_from_start"], cfg["n_head_kv"] * cfg["head_dim"]
    rng = np.random.default_rng(11)
    body = rng.normal(0, 1, 2 * L_w * 5 * kv).astype(np.float16)
    src = b"KVCP" + np.array([5, L_w, kv], dtype="<i4").tobytes() + body.tobytes()
    orc = OracleContext(cfg, tiny, 16)
    orc.kv_load(src, 3)
    want = orc.kv_save()
    ctx = binding.PrefillContext(tiny, max_ctx=16, ubatch_max=16)
    arr = np.frombuffer(src, dtype=np.uint8).copy()
    dev = torch.from_numpy(arr).cuda()
    ctx.kv_load(dev, len(arr), 3)
    n = ctx.kv_image_bytes(3)
    out = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ctx.kv_save(out, n)
    ctx.sync()
    ctx.close()
    assert out.cpu().numpy().tobytes() == want


def test_errors_leave_state(gpu, tiny):
    cfg = tiny.cfg
    ctx = binding.PrefillContext(tiny, max_ctx=64, ubatch_max=32)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    tok = synth.make_tokens(cfg, 40)
    with pytest.raises(binding.PrefillError) as e:
        ctx.ubatch(tok, 0, True, logits)          # more than ubatch_max
    assert e.value.code == binding.PF_E_ARG
    bad = tok[:10].copy()
    bad[3] = -1
    with pytest.raises(binding.PrefillError):
        ctx.ubatch(bad, 0, True, logits)          # token out of range
    ctx.ubatch(tok[:20], 0, False)
    with pytest.raises(binding.PrefillError):
        ctx.ubatch(tok[20:30], 5, True, logits)   # pos0 gap
    with pytest.raises(binding.PrefillError) as e:
        ctx.ubatch(tok[:0], 20, True, logits)       # empty ubatch
    assert e.value.code == binding.PF_E_ARG and ctx.n_pos == 20
    with pytest.raises(binding.PrefillError) as e:
        ctx.ubatch(tok[20:40], 20, True, None)      # last ubatch without logits
    assert e.value.code == binding.PF_E_ARG and ctx.n_pos == 20
    with pytest.raises(binding.PrefillError) as e:   # logits in host memory
        ctx.ubatch(tok[20:40], 20, True, np.empty(cfg["vocab"], dtype=np.float32))
    assert e.value.code == binding.PF_E_ARG and ctx.n_pos == 20
    ctx.ubatch(tok[20:40], 20, True, logits)
    with pytest.raises(binding.PrefillError) as e:
        ctx.ubatch(synth.make_tokens(cfg, 25), 40, True, logits)   # 40 + 25 > max_ctx 64
    assert e.value.code == binding.PF_E_ARG and ctx.n_pos == 40
    ctx.sync()
    n = ctx.kv_image_bytes(40)
    img = np.empty(n, dtype=np.uint8)
    ctx.kv_save(img, n)
    ctx.reset()
    for blob, npos, code in [(b"KVCQ" + img[4:].tobytes(), 10, binding.PF_E_KV_MAGIC),
                             (img[:8].tobytes() + np.int32(3).tobytes() + img[12:].tobytes(), 10, binding.PF_E_KV_SHAPE),
                             (img.tobytes(), 41, binding.PF_E_KV_RANGE),
                             (img[:200].tobytes(), 10, binding.PF_E_KV_RANGE)]:
        arr = np.frombuffer(blob, dtype=np.uint8).copy()
        with pytest.raises(binding.PrefillError) as e:
            ctx.kv_load(arr, len(arr), npos)
        assert e.value.code == code
        assert ctx.n_pos == 0
    ctx.close()


def test_kv_file_roundtrip_and_cached_prefill(gpu, tinyllama, tmp_path):
    """A KV image written to a file restores the same cache as the in-memory
    image (suffix logits bit for bit), and the cached-prefix flow (load when
    the file is valid, else full prefill and save) gives the full prefill's
    logits to rounding; a damaged file is refused with the state unchanged."""
    cfg = tinyllama.cfg
    prefix = synth.make_tokens(cfg, 500, seed=1)
    suffix = synth.make_tokens(cfg, 32, seed=2)
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    ctx = binding.PrefillContext(tinyllama, max_ctx=532, ubatch_max=512)
    ctx.ubatch(prefix, 0, False)
    path = str(tmp_path / "prefix.kvcp")
    ctx.kv_save_file(path)
    nbytes = ctx.kv_image_bytes(500)
    assert os.path.getsize(path) == nbytes
    img = np.empty(nbytes, dtype=np.uint8)
    ctx.kv_save(img, nbytes)
    assert open(path, "rb").read() == img.tobytes()
    assert binding.kv_file_check(path, 22, 256, 532) == (binding.PF_OK, 500)
    res = []
    for how in ("memory", "file"):
        ctx.reset()
        if how == "memory":
            ctx.kv_load(img, nbytes, 500)
        else:
            assert ctx.kv_load_file(path) == binding.PF_OK
        assert ctx.n_pos == 500
        ctx.ubatch(suffix, 500, True, logits)
        ctx.sync()
        res.append(logits.cpu().numpy().copy())
    np.testing.assert_array_equal(res[0], res[1])
    # a damaged file: refused, nothing changes
    bad = str(tmp_path / "bad.kvcp")
    with open(bad, "wb") as f:
        f.write(b"KVCQ" + img[4:].tobytes())
    ctx.reset()
    assert ctx.kv_load_file(bad) == binding.PF_E_KV_MAGIC
    assert ctx.n_pos == 0
    assert ctx.kv_load_file(str(tmp_path / "missing.kvcp")) == binding.PF_E_IO
    # the cached-prefix flow: first call prefills all and saves, second loads
    prompt = np.concatenate([prefix, suffix])
    cache = str(tmp_path / "flow.kvcp")
    full = run_gpu(tinyllama, prompt, 512, True, max_ctx=532)
    assert binding.prefill_with_cache(ctx, prompt[:500], 512, logits, cache) == 0
    ctx.sync()
    assert binding.kv_file_check(cache, 22, 256, 532)[1] == 500
    assert binding.prefill_with_cache(ctx, prompt, 512, logits, cache) == 500
    ctx.sync()
    got = logits.cpu().numpy()
    assert np.abs(got - full).max() <= 2e-3 * np.abs(full).max()
    ctx.close()


@pytest.mark.parametrize("name", ["tiny", "e2b"])
def test_decode_steps_match_oracle(gpu, tiny, e2b, name):
    """Generation after the prompt: one-token ubatches continue the cache
    (every layer takes the single-row attention), within tolerance of the
    oracle's continuation, and the same bits with pruning on and off."""
    w = tiny if name == "tiny" else e2b
    cfg = w.cfg
    n0, steps = (40, 6) if name == "tiny" else (300, 3)
    tok = synth.make_tokens(cfg, n0 + steps)
    orc = OracleContext(cfg, w, n0 + steps)
    orc.ubatch(tok[:n0], False)
    outs = {}
    for prune in (True, False):
        ctx = binding.PrefillContext(w, max_ctx=n0 + steps, ubatch_max=n0, prune=prune)
        logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
        ctx.ubatch(tok[:n0], 0, True, logits)
        got = []
        for i in range(n0, n0 + steps):
            ctx.ubatch(tok[i:i + 1], i, True, logits)
            ctx.sync()
            got.append(logits.cpu().numpy().copy())
        outs[prune] = got
        ctx.close()
    for a, b in zip(outs[True], outs[False]):
        np.testing.assert_array_equal(a, b)
    for i in range(steps):
        want = orc.ubatch(tok[n0 + i:n0 + i + 1], True)
        check_logits(outs[True][i], want, f"{name} decode step {i}")


def test_cli_cache_file_flow(gpu, tinyllama, tmp_path):
    """The command-line flow of the PicoLM cache article on the TinyLlama
    shape with a 25-token prompt: the first run prefills and writes the
    cache file, whose body is the article's 2 x 22 x 25 x 256 x 2 bytes
    (tests/golden/kv_image_size.txt); the second run restores 24 positions
    from it and prefills the last token, with the same first generated token
    and logits to rounding; a damaged file is refused and rewritten."""
    import io

    from prefill_kv_shared_gb300 import cli
    pin = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "kv_image_size.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, v = ln.split()
                pin[k] = int(v)
    path = str(tmp_path / "prompt.kvcp")
    args = cli.parse_args(["--model", "tinyllama", "--prompt-tokens", str(pin["n_pos"]), "--cache", path,
                           "--gen", "4"])
    log = io.StringIO()
    first = cli.run(args, weights=tinyllama, out=log)
    assert first["restored"] == 0
    assert os.path.getsize(path) - 16 == pin["body_bytes"]
    second = cli.run(args, weights=tinyllama, out=log)
    assert second["restored"] == pin["n_pos"] - 1
    assert "restored 24 prompt positions" in log.getvalue()
    assert second["first_token"] == first["first_token"]
    assert second["generated"] == first["generated"]
    a, b = first["logits"], second["logits"]
    assert np.abs(a - b).max() <= 2e-3 * np.abs(a).max()
    with open(path, "r+b") as f:
        f.write(b"XXXX")
    third = cli.run(args, weights=tinyllama, out=log)
    assert third["restored"] == 0 and "refused" in log.getvalue()
    assert os.path.getsize(path) - 16 == pin["body_bytes"]


def test_hidden_state_outputs_match_oracle(gpu, tiny):
    """Embeddings output and per-layer input hidden states (G4 section 1
    listing: requesting them at or past the first KV-shared layer turns the
    pruning off), ubatch by ubatch against the oracle; a request below the
    first KV-shared layer keeps the pruning and leaves the logits' bits."""
    cfg = tiny.cfg
    L, D = cfg["n_layer"], cfg["d_model"]
    tok = synth.make_tokens(cfg, 61, seed=5)
    cuts = [(0, 32), (32, 61)]
    req = [False, True, False, True, True]
    ctx = binding.PrefillContext(tiny, max_ctx=64, ubatch_max=32, embeddings=True, layer_inp=req)
    assert not ctx.prune_active
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    with pytest.raises(binding.PrefillError) as e:
        ctx.ubatch(tok[:32], 0, False)  # requested outputs without buffers
    assert e.value.code == binding.PF_E_ARG
    with pytest.raises(binding.PrefillError) as e:
        ctx.set_output(2, torch.empty(32 * D, device="cuda"))  # layer 2 was not requested
    assert e.value.code == binding.PF_E_ARG
    bufs = {k: torch.full((32, D), float("nan"), device="cuda") for k in (1, 3, L, binding.PF_OUT_EMBD)}
    for k, b in bufs.items():
        ctx.set_output(k, b)
    orc = OracleContext(cfg, tiny, 64)
    for a, b in cuts:
        cap = {}
        want_logits = orc.ubatch(tok[a:b], b == 61, embeddings=True, embd_layer_inp=req, capture=cap)
        ctx.ubatch(tok[a:b], a, b == 61, logits)
        ctx.sync()
        for k, buf in bufs.items():
            got = buf[:b - a].cpu().numpy()
            want = cap["embd" if k == binding.PF_OUT_EMBD else k]
            assert got.shape == want.shape
            assert np.abs(got - want).max() <= 2e-2 * np.abs(want).max(), (k, a)
    check_logits(logits.cpu().numpy(), want_logits, "tiny-61 with hidden-state outputs")
    ctx.close()
    # a request below the first KV-shared layer: pruning stays on, logits unchanged
    ref = run_gpu(tiny, tok, 32, True, max_ctx=64)
    req1 = [False, True, False, False, False]
    c1 = binding.PrefillContext(tiny, max_ctx=64, ubatch_max=32, layer_inp=req1)
    assert c1.prune_active
    buf = torch.empty((32, D), device="cuda")
    c1.set_output(1, buf)
    orc = OracleContext(cfg, tiny, 64)
    for a, b in cuts:
        cap = {}
        orc.ubatch(tok[a:b], b == 61, prune=True, embd_layer_inp=req1, capture=cap)
        c1.ubatch(tok[a:b], a, b == 61, logits)
        c1.sync()
        assert np.abs(buf[:b - a].cpu().numpy() - cap[1]).max() <= 2e-2 * np.abs(cap[1]).max()
    np.testing.assert_array_equal(logits.cpu().numpy(), ref)
    c1.close()


def _multi_seq_check(w, ubatches, n_seq, max_ctx, ubatch_max, case):
    """ubatches: [[(seq, tokens, is_last), ...], ...].  Runs them through one
    context with pruning on and off; every finishing sequence's logits must
    match its own oracle run (each sequence alone), and the two modes must
    agree bit for bit."""
    cfg = w.cfg
    outs = {}
    for prune in (True, False):
        ctx = binding.PrefillContext(w, max_ctx=max_ctx, ubatch_max=ubatch_max, n_seq_max=n_seq, prune=prune)
        got = []
        for ub in ubatches:
            toks = np.concatenate([t for _, t, _ in ub]).astype(np.int32)
            runs = [(q, len(t), last) for q, t, last in ub]
            n_last = sum(1 for r in runs if r[2])
            lg = torch.full((max(n_last, 1), cfg["vocab"]), float("nan"), device="cuda")
            ctx.ubatch_seqs(toks, runs, lg if n_last else None)
            ctx.sync()
            got += [lg[j].cpu().numpy().copy() for j in range(n_last)]
        outs[prune] = got
        ctx.close()
    for a, b in zip(outs[True], outs[False]):
        np.testing.assert_array_equal(a, b)
    oracles = {}
    want = []
    for ub in ubatches:
        for q, t, last in ub:
            o = oracles.setdefault(q, OracleContext(cfg, w, max_ctx))
            r = o.ubatch(t, bool(last))
            if last:
                want.append(r)
    assert len(want) == len(outs[True])
    for j, (g, wnt) in enumerate(zip(outs[True], want)):
        check_logits(g, wnt, f"{case} output {j}")


def test_multi_sequence_ubatches_match_oracle(gpu, tiny):
    """Three sequences sharing one cache and one ubatch (ragged runs, a
    sequence that finishes in the first ubatch, two that finish in the
    second): each finishing sequence's logits against the oracle run on that
    sequence alone, and the per-sequence gather bit-identical to the
    unpruned pass."""
    cfg = tiny.cfg
    a = synth.make_tokens(cfg, 20, seed=31)
    b = synth.make_tokens(cfg, 14, seed=32)
    c = synth.make_tokens(cfg, 25, seed=33)
    ubatches = [[(1, b[:9], False), (0, a[:12], False), (2, c, True)],
                [(0, a[12:], True), (1, b[9:], True)]]
    _multi_seq_check(tiny, ubatches, 3, 32, 64, "tiny multi-sequence")


def test_multi_sequence_e2b_4x128(gpu, e2b):
    cfg = e2b.cfg
    ubatches = [[(q, synth.make_tokens(cfg, 128, seed=40 + q), True) for q in range(4)]]
    _multi_seq_check(e2b, ubatches, 4, 128, 512, "e2b 4x128 multi-sequence")


def test_multi_sequence_refusals(gpu, tiny):
    cfg = tiny.cfg
    ctx = binding.PrefillContext(tiny, max_ctx=32, ubatch_max=40, n_seq_max=2)
    t = synth.make_tokens(cfg, 30, seed=3)
    lg = torch.empty((2, cfg["vocab"]), device="cuda")
    for runs in ([(0, 5, True), (0, 5, True)],          # one sequence twice
                 [(2, 5, True)],                        # seq_id past n_seq_max
                 [(0, 25, False), (1, 20, True)],       # more than ubatch_max tokens
                 [(0, 0, True)]):                       # an empty run
        with pytest.raises(binding.PrefillError) as e:
            ctx.ubatch_seqs(t[:sum(r[1] for r in runs)] if sum(r[1] for r in runs) <= 30 else
                            np.concatenate([t, t])[:sum(r[1] for r in runs)], runs, lg)
        assert e.value.code == binding.PF_E_ARG
    ctx.ubatch_seqs(t[:30], [(1, 30, False)])
    ctx.sync()
    assert ctx.seq_n_pos(1) == 30 and ctx.seq_n_pos(0) == 0
    with pytest.raises(binding.PrefillError):
        ctx.ubatch_seqs(t[:5], [(1, 5, True)], lg)     # 30 + 5 > max_ctx 32
    ctx.seq_reset(1)
    assert ctx.seq_n_pos(1) == 0
    ctx.close()


def test_graph_replay_matches_stream_launches(gpu, e2b):
    """A recorded E2B-512 ubatch replayed as one CUDA graph gives the logits
    of the stream launches bit for bit, replay after replay, for whatever
    the recorded token buffer holds; replays need the recorded position."""
    cfg = e2b.cfg
    s = torch.cuda.Stream()
    ctx = binding.PrefillContext(e2b, max_ctx=512, ubatch_max=512, stream=s)
    toks = [torch.from_numpy(synth.make_tokens(cfg, 512, seed=q)).cuda() for q in (1, 9)]
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    want = []
    for t in toks:
        ctx.reset()
        ctx.ubatch(t, 0, True, logits)
        ctx.sync()
        want.append(logits.cpu().numpy().copy())
    buf = toks[0].clone()
    ctx.reset()
    with pytest.raises(binding.PrefillError) as e:
        ctx.graph_capture(torch.from_numpy(np.zeros(4, np.int32)), 0, True, logits)  # host tokens
    assert e.value.code == binding.PF_E_ARG
    ctx.graph_capture(buf, 0, True, logits)
    assert ctx.n_pos == 0
    for rep in range(2):
        for q, t in enumerate(toks):
            buf.copy_(t)
            torch.cuda.synchronize()
            ctx.reset()
            ctx.graph_launch()
            assert ctx.n_pos == 512
            ctx.sync()
            np.testing.assert_array_equal(logits.cpu().numpy(), want[q])
    with pytest.raises(binding.PrefillError) as e:
        ctx.graph_launch()  # the recorded ubatch starts at position 0
    assert e.value.code == binding.PF_E_ARG
    ctx.close()
