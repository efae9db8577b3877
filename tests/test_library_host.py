"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol the headers declare, and its host-only helpers agree with the
pages' facts and the oracle."""
import os
import re
import struct
import subprocess

import pytest

import oracle
from prefill_kv_shared_gb300 import binding, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    from prefill_kv_shared_gb300 import build
    build.build()
    return binding.load()


def _declared_functions():
    names = set()
    for h in ("prefill.h", "prefill_ops.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M):
            name = m.group(1)
            if name not in ("defined",):
                names.add(name)
    return names


def test_headers_are_plain_c():
    for h in ("prefill.h", "prefill_ops.h"):
        r = subprocess.run(["gcc", "-fsyntax-only", "-std=c99", "-Wall", "-Werror", "-x", "c",
                            os.path.join(ROOT, "include", h)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_plain_c_client(lib, tmp_path):
    """A C99 program (tests/c_abi_client.c) compiled against include/prefill.h
    and linked with the library: the host-only calls answer as the pages fix
    them and, without a GPU, creating a context fails with PF_E_CUDA and a
    message (no host fallback)."""
    exe = str(tmp_path / "c_abi_client")
    libdir = os.path.dirname(binding.LIB_PATH)
    name = os.path.basename(binding.LIB_PATH)[3:-3]
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_client.c"), "-L", libdir, "-l" + name,
                        "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    args = [exe]
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        args.append("nogpu")
    r = subprocess.run(args, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, f"check {r.returncode} failed: {r.stdout} {r.stderr}"
    assert r.stdout.strip().endswith("ok")


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "prefill_ubatch" in declared and "kv_load" in declared and "pfop_attention" in declared
    assert declared == set(binding.EXPORTS), declared ^ set(binding.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = declared - exported
    assert not missing, missing


def test_kv_image_size_pin(lib):
    kv = {}
    for ln in open(os.path.join(GOLDEN, "kv_image_size.txt")):
        if ln.strip() and not ln.startswith("#"):
            k, v = ln.split()
            kv[k] = int(v)
    n = binding.kv_image_bytes_for(kv["layers"], kv["n_pos"], kv["kv_dim"])
    assert n - 16 == kv["body_bytes"]
    assert n == oracle.kv_image_bytes(kv["layers"], kv["n_pos"], kv["kv_dim"])
    assert binding.kv_image_bytes_for(-1, 3, 4) == -1


def test_prune_predicate_matches_listing(lib):
    base = synth.config("e2b")
    for ln in open(os.path.join(GOLDEN, "prune_predicate.txt")):
        if not ln.strip() or ln.startswith("#"):
            continue
        L, S, nseq, emb, idx, want = (int(v) for v in ln.split())
        inp = None
        if idx >= 0:
            inp = [False] * (L + 1)
            inp[idx] = True
        cfg = dict(base, n_layer=L, n_layer_kv_from_start=S,
                   kv_src=[-1 if i < S else max(S - 1, 0) for i in range(L)])
        assert binding.prune_predicate(cfg, True, nseq, bool(emb), inp) == bool(want), ln
        assert oracle.prune_shared(L, S, n_seq_max=nseq, embeddings=bool(emb),
                                   embeddings_layer_inp=inp) == bool(want)
    assert binding.prune_predicate(base, prune=False) is False


def test_prune_predicate_agrees_with_the_oracle(lib):
    """The library's pruning condition and the oracle's agree on 500 seeded
    descriptions (layer counts, the first KV-shared layer, sequences,
    embeddings, sparse per-layer input requests, the on/off switch)."""
    import numpy as np

    base = synth.config("e2b")
    rng = np.random.default_rng(21)
    outcomes = set()
    for _ in range(500):
        L = int(rng.integers(1, 41))
        S = int(rng.integers(1, L + 1))
        nseq = int(rng.choice([1, 1, 1, 2, 3]))
        emb = bool(rng.random() < 0.15)
        inp = None if rng.random() < 0.5 else [bool(f) for f in rng.random(L + 1) < 0.04]
        on = bool(rng.random() < 0.9)
        cfg = dict(base, n_layer=L, n_layer_kv_from_start=S,
                   kv_src=[-1 if i < S else S - 1 for i in range(L)])
        got = binding.prune_predicate(cfg, on, nseq, emb, inp)
        want = on and oracle.prune_shared(L, S, n_seq_max=nseq, embeddings=emb, embeddings_layer_inp=inp)
        assert got == want, (L, S, nseq, emb, inp, on)
        outcomes.add(got)
    assert outcomes == {True, False}


def _hdr(n, layers, kv, magic=b"KVCP"):
    return magic + struct.pack("<iii", n, layers, kv)


def test_kv_header_check(lib):
    size = binding.kv_image_bytes_for(22, 500, 256)
    ok = binding.kv_header_check(_hdr(500, 22, 256), 22, 256, 500, 2048, size)
    assert ok == binding.PF_OK
    assert binding.kv_header_check(_hdr(500, 22, 256), 22, 256, 25, 2048, size) == binding.PF_OK
    assert binding.kv_header_check(_hdr(500, 22, 256, b"KVCQ"), 22, 256, 500, 2048, size) == binding.PF_E_KV_MAGIC
    assert binding.kv_header_check(_hdr(500, 21, 256), 22, 256, 500, 2048, size) == binding.PF_E_KV_SHAPE
    assert binding.kv_header_check(_hdr(500, 22, 128), 22, 256, 500, 2048, size) == binding.PF_E_KV_SHAPE
    assert binding.kv_header_check(_hdr(500, 22, 256), 22, 256, 501, 2048, size) == binding.PF_E_KV_RANGE
    assert binding.kv_header_check(_hdr(500, 22, 256), 22, 256, 500, 499, size) == binding.PF_E_KV_RANGE
    assert binding.kv_header_check(_hdr(500, 22, 256), 22, 256, 500, 2048, size - 1) == binding.PF_E_KV_RANGE
    assert binding.kv_header_check(b"KV", 22, 256, 0, 2048, 2) == binding.PF_E_KV_MAGIC


def test_kv_header_check_agrees_with_the_oracle(lib, tmp_path):
    """The library's host checks of a KV image (in memory, and as a file
    restored whole) and the oracle's restore refuse the same images with the
    same class of error (PicoLM KV cache article, "rules": wrong magic, a
    layer or KV-width mismatch, or a position count beyond the image or the
    context), over 600 seeded cases that mix one or two faults."""
    import numpy as np
    from oracle.prefill import KVImageError, OracleContext

    L_w, kv = 2, 8
    cfg = dict(n_layer=3, n_layer_kv_from_start=L_w, n_head=1, n_head_kv=1, head_dim=kv)
    code = {"magic": binding.PF_E_KV_MAGIC, "shape": binding.PF_E_KV_SHAPE, "range": binding.PF_E_KV_RANGE}
    rng = np.random.default_rng(12)
    seen = set()
    for _ in range(600):
        n_img = int(rng.choice([-1, 0, 1, 5, 17]))
        l_img = int(rng.choice([L_w, L_w, L_w, 1, 3]))
        kv_img = int(rng.choice([kv, kv, kv, 4, 16]))
        magic = bytes(rng.choice([b"KVCP", b"KVCP", b"KVCP", b"KVCQ", b"kvcp"]))
        n_pos = int(rng.integers(-1, max(n_img, 0) + 3))
        max_ctx = int(rng.choice([4, 16, 64]))
        exact = 16 + 2 * max(l_img, 0) * max(n_img, 0) * max(kv_img, 0) * 2
        size = int(rng.choice([exact, exact, exact - 1, exact + 16, 2]))
        size = max(size, 0)
        img = (magic + struct.pack("<iii", n_img, l_img, kv_img)).ljust(size, b"\0")[:size]
        got = binding.kv_header_check(img, L_w, kv, n_pos, max_ctx, size)
        o = OracleContext(cfg, None, max_ctx=max_ctx)
        try:
            o.kv_load(img, n_pos)
            want = binding.PF_OK
        except KVImageError as e:
            want = code[e.code]
        assert got == want, (magic, n_img, l_img, kv_img, n_pos, max_ctx, size)
        seen.add(want)
        path = str(tmp_path / "img.kvcp")
        with open(path, "wb") as f:
            f.write(img)
        got_file, n_file = binding.kv_file_check(path, L_w, kv, max_ctx)
        try:
            OracleContext(cfg, None, max_ctx=max_ctx).kv_load(img, n_img)
            want_file = binding.PF_OK
        except KVImageError as e:
            want_file = code[e.code]
        assert got_file == want_file, ("file", magic, n_img, l_img, kv_img, max_ctx, size)
        if want_file == binding.PF_OK:
            assert n_file == n_img
    assert seen == {binding.PF_OK, *code.values()}


@pytest.mark.parametrize("Hq,Hkv,hd,with_kv", [(8, 1, 256, True), (8, 2, 256, True), (8, 1, 256, False),
                                             (4, 1, 64, True), (32, 4, 64, True), (2, 1, 128, True)])
def test_qkv_row_order_keeps_rope_pairs_in_a_tile(lib, Hq, Hkv, hd, with_kv):
    """The stored Q|K|V rows: every source row exactly once, the last tile
    padded, every RoPE pair (i, i + hd/2) of a Q or K head inside one
    128-row tile (the epilogue rotates a pair within its tile), V in order."""
    import numpy as np
    order = binding.qkv_row_order(Hq, Hkv, hd, with_kv)
    q, kv = Hq * hd, Hkv * hd
    n_src = q + (2 * kv if with_kv else 0)
    assert len(order) == (n_src + 127) // 128 * 128
    real = order[order >= 0]
    assert sorted(real.tolist()) == list(range(n_src))
    assert (order[len(real):] == -1).all()
    tile_of = {int(src): i // 128 for i, src in enumerate(order) if src >= 0}
    for src in range(q + (kv if with_kv else 0)):
        head, i = divmod(src, hd)
        partner = head * hd + (i + hd // 2) % hd
        assert tile_of[src] == tile_of[partner], (src, partner)
    if hd <= 128:
        assert (real == np.arange(n_src)).all()
    if with_kv:
        v_pos = [i for i, src in enumerate(order) if src >= q + kv]
        assert [int(order[i]) for i in v_pos] == list(range(q + kv, n_src))
    with pytest.raises(binding.PrefillError):
        binding.qkv_row_order(Hq, Hkv, 192, with_kv)


@pytest.mark.parametrize("N,K,bn", [(200, 128, 128), (200, 128, 192), (64, 64, 64), (300, 256, 256)])
def test_repack_q4_matches_documented_tile_layout(lib, N, K, bn):
    """The stored Q4_0 tiles, read back by the layout include/prefill_ops.h
    documents, decode to the source matrix (the oracle's decode), with zero
    rows padding the last tile."""
    import numpy as np
    rng = np.random.default_rng(N + K + bn)
    w = synth.draw_q4_0(rng, N, K)
    stored = binding.repack_q4(w, bn)
    n_tiles, nkb = (N + bn - 1) // bn, K // 64
    assert stored.size == n_tiles * nkb * bn * 36
    want = oracle.prefill.as_f32_matrix(w)
    got = np.zeros((n_tiles * bn, K), dtype=np.float32)
    for t in range(n_tiles):
        for kb in range(nkb):
            tile = stored[(t * nkb + kb) * bn * 36:(t * nkb + kb + 1) * bn * 36]
            for h in range(2):
                nib = tile[h * bn * 16:(h + 1) * bn * 16].reshape(bn, 16)
                sc = tile[bn * 32 + h * bn * 2:bn * 32 + (h + 1) * bn * 2].reshape(bn, 2)
                blocks = np.concatenate([sc, nib], axis=1).reshape(bn, 1, 18)
                got[t * bn:(t + 1) * bn, kb * 64 + h * 32:kb * 64 + h * 32 + 32] = oracle.q4_0_decode(blocks)[:, :32]
    np.testing.assert_array_equal(got[:N], want)
    assert not got[N:].any()


def test_stats_struct_matches_binding(tmp_path):
    """The ctypes mirror of prefill_stats has the header's class count and size."""
    import ctypes
    src = tmp_path / "s.c"
    src.write_text('#include <stdio.h>\n#include "prefill.h"\n'
                   'int main(void){printf("%d %d\\n", (int)PF_KC_COUNT, (int)sizeof(prefill_stats));return 0;}\n')
    exe = tmp_path / "s"
    r = subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    n, size = map(int, subprocess.run([str(exe)], capture_output=True, text=True).stdout.split())
    assert n == binding.KC_COUNT == len(binding.KC_NAMES)
    assert size == ctypes.sizeof(binding.Stats)


def test_kv_file_check_host_only(lib, tmp_path):
    """The file form of the KV image header check (PicoLM KV cache article,
    "file" and "rules"): a valid file gives its position count; a wrong
    magic, a wrong shape, a short file, a count beyond the context and a
    missing file are refused."""
    import numpy as np
    L_w, n, kv = 3, 40, 64
    hdr = b"KVCP" + np.array([n, L_w, kv], dtype="<i4").tobytes()
    body = bytes(2 * L_w * n * kv * 2)
    cases = {
        "ok": (hdr + body, binding.PF_OK),
        "magic": (b"KVCQ" + hdr[4:] + body, binding.PF_E_KV_MAGIC),
        "shape": (b"KVCP" + np.array([n, L_w + 1, kv], dtype="<i4").tobytes() + body, binding.PF_E_KV_SHAPE),
        "short": (hdr + body[:-2], binding.PF_E_KV_RANGE),
    }
    for name, (blob, code) in cases.items():
        p = tmp_path / (name + ".kvcp")
        p.write_bytes(blob)
        rc, npos = binding.kv_file_check(str(p), L_w, kv, 100)
        assert rc == code, name
        if code == binding.PF_OK:
            assert npos == n
    p = tmp_path / "ok.kvcp"
    assert binding.kv_file_check(str(p), L_w, kv, 39)[0] == binding.PF_E_KV_RANGE  # beyond the context
    assert binding.kv_file_check(str(tmp_path / "none.kvcp"), L_w, kv, 100)[0] == binding.PF_E_IO


def test_prefill_with_cache_flow_decisions(tmp_path):
    """The cached-prefix flow (PicoLM KV cache article, "usage"): a missing or
    refused file means a full prefill and a save; a valid file of the first
    n positions means a restore and a prefill of the rest only."""
    import numpy as np

    class FakeCtx:
        n_layers_written, kv_dim, max_ctx = 3, 64, 100

        def __init__(self, load_rc):
            self.calls, self.load_rc = [], load_rc

        def reset(self):
            self.calls.append(("reset",))

        def kv_load_file(self, path, n):
            self.calls.append(("load", n))
            return self.load_rc

        def ubatch(self, tok, pos0, is_last, logits):
            self.calls.append(("ubatch", pos0, len(tok), bool(is_last)))

        def sync(self):
            pass

        def kv_save_file(self, path):
            self.calls.append(("save",))

    tok = np.arange(50, dtype=np.int32)
    path = str(tmp_path / "p.kvcp")
    ctx = FakeCtx(binding.PF_OK)
    assert binding.prefill_with_cache(ctx, tok, 32, None, path) == 0  # no file yet
    assert ctx.calls == [("reset",), ("ubatch", 0, 32, False), ("ubatch", 32, 18, True), ("save",)]
    # a valid 40-position image of this model
    hdr = b"KVCP" + np.array([40, 3, 64], dtype="<i4").tobytes()
    with open(path, "wb") as f:
        f.write(hdr + bytes(2 * 3 * 40 * 64 * 2))
    ctx = FakeCtx(binding.PF_OK)
    assert binding.prefill_with_cache(ctx, tok, 32, None, path) == 40
    assert ctx.calls == [("reset",), ("load", 40), ("ubatch", 40, 10, True)]
    # the restore refused (e.g. the context changed): full prefill and save
    ctx = FakeCtx(binding.PF_E_KV_RANGE)
    assert binding.prefill_with_cache(ctx, tok, 32, None, path) == 0
    assert ctx.calls[-1] == ("save",) and ("ubatch", 0, 32, False) in ctx.calls
    # an image as long as the prompt cannot leave a row to prefill: ignored
    with open(path, "wb") as f:
        f.write(b"KVCP" + np.array([50, 3, 64], dtype="<i4").tobytes() + bytes(2 * 3 * 50 * 64 * 2))
    ctx = FakeCtx(binding.PF_OK)
    assert binding.prefill_with_cache(ctx, tok, 32, None, path) == 0
    assert ("load", 50) not in ctx.calls


def test_product_package_never_touches_the_oracle():
    """The library's Python side is marshalling only: no module of the
    package imports the oracle (which is test infrastructure)."""
    pkg = os.path.join(ROOT, "prefill_kv_shared_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            src = open(os.path.join(pkg, name)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), name


def test_missing_library_raises():
    code = ("import sys; from prefill_kv_shared_gb300 import binding\n"
            "try:\n    binding.load('/nonexistent/libprefill_kv_shared.so')\n"
            "except RuntimeError as e:\n    print('raised', e)\n    sys.exit(0)\n"
            "sys.exit(3)\n")
    r = subprocess.run([os.sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "CUDA library not found" in r.stdout, r.stdout + r.stderr


def test_no_gpu_means_an_error_not_a_fallback(lib):
    """Without a CUDA device the context refuses to be created (PF_E_CUDA):
    nothing of the pass runs on the host."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = synth.config("tiny")
    w = synth.make_weights(cfg)
    with pytest.raises(binding.PrefillError) as e:
        binding.PrefillContext(w, max_ctx=64, ubatch_max=32)
    assert e.value.code == binding.PF_E_CUDA


@pytest.mark.parametrize("kw", [dict(ubatch_max=1 << 21), dict(max_ctx=1 << 27),
                                dict(ubatch_max=1 << 20, cfg=dict(d_model=4096)),
                                dict(max_ctx=1 << 24, cfg=dict(n_head=16, n_head_kv=16, head_dim=256))])
def test_oversized_descriptions_refused_before_any_cuda_call(lib, kw):
    """Sizes whose element counts would pass 2^31 (the kernels index rows,
    weights and a layer's cache with 32-bit integers) are refused with
    PF_E_ARG by the description check, which runs before the first CUDA
    call (so this holds on a machine without a GPU too)."""
    cfg = dict(synth.config("tiny"))
    cfg.update(kw.get("cfg", {}))
    w = synth.make_weights(synth.config("tiny"))
    w.cfg = cfg
    with pytest.raises(binding.PrefillError) as e:
        binding.PrefillContext(w, max_ctx=kw.get("max_ctx", 64), ubatch_max=kw.get("ubatch_max", 32))
    assert e.value.code == binding.PF_E_ARG, str(e.value)


def test_attention_entry_points_refuse_empty_head_counts(lib):
    """Zero query or KV heads are argument errors (PF_E_ARG), found before
    any CUDA call or any division by the head-group size."""
    import ctypes as C
    fake = C.c_void_p(256)  # never dereferenced: the argument check fails first
    us = C.c_float(0.0)
    for hq, hkv in ((0, 1), (8, 0), (0, 0)):
        for mode in (0, 1):
            assert lib.pfop_attention(mode, fake, fake, fake, 1, hq, hkv, 64, 0, 1, fake, None) == binding.PF_E_ARG
            assert lib.pfop_attention_bench(mode, fake, fake, fake, 1, hq, hkv, 64, 0, 1, fake, None, 0, 0, 1,
                                            C.byref(us), None) == binding.PF_E_ARG
        assert lib.pfop_attention_split_noalloc(fake, fake, fake, hq, hkv, 64, 0, 1, fake, None) == binding.PF_E_ARG


@pytest.mark.parametrize("cache_off,img_off,cache_seg,img_seg,copy", [
    (8, 0, 256, 512, 512), (0, 4, 256, 512, 512), (0, 0, 252, 512, 512), (0, 0, 256, 520, 512),
    (0, 0, 256, 512, 504)])
def test_kv_copy_refuses_unaligned_layouts(lib, cache_off, img_off, cache_seg, img_seg, copy):
    """The KV copy kernel moves 16-byte vectors: misaligned pointers, cache
    strides or byte counts are argument errors, found before any CUDA call."""
    import ctypes as C
    base = 1 << 20  # never dereferenced
    us = C.c_float(0.0)
    args = (C.c_void_p(base + cache_off), cache_seg, C.c_void_p(base + img_off), img_seg, 2, copy)
    assert lib.pfop_kv_copy(1, *args, None, None) == binding.PF_E_ARG
    assert lib.pfop_kv_copy_bench(1, *args, None, 0, 0, 1, C.byref(us), None) == binding.PF_E_ARG


def test_binding_checks_buffers_it_can_see():
    """The binding refuses buffers the library could overrun behind a bare
    pointer: wrong element type, too few elements, non-contiguous views."""
    import numpy as np
    import torch
    assert binding._buffer(None, "x") is None and binding._buffer(4096, "x") is None
    assert binding._buffer(np.zeros(10, np.float32), "x", "float32", 10) == 40
    assert binding._buffer(torch.zeros(10, dtype=torch.int32), "x", "int32") == 40
    bad = [(np.zeros(10, np.float64), "float32", 10), (np.zeros(9, np.float32), "float32", 10),
           (np.zeros((4, 4), np.float32)[:, 0], "float32", 4), (torch.zeros(10, dtype=torch.int64), "int32", 0),
           (torch.zeros(4, 4)[:, 1], "float32", 4)]
    for arr, dt, n in bad:
        with pytest.raises(ValueError):
            binding._buffer(arr, "x", dt, n)
