"""Kernel-by-kernel parity of the CUDA path against the CPU oracle, through
the op-level C ABI (include/prefill_ops.h).  Sizes span several tiles and a
ragged tail; each GEMM is checked twice: tightly against the same arithmetic
in float64 on the bf16 operands the tensor cores see, and against the
oracle's exact Q4_0 decode within the bf16 rounding bound."""
import math

import numpy as np
import pytest

import oracle
from oracle.prefill import as_f32_matrix
from prefill_kv_shared_gb300 import binding, synth
from tests.gpu_util import bf16_round, gpu_q4_weights, need_gpu, padded_a, rel_err, torch

pytestmark = pytest.mark.gpu

Q4, F32 = binding.PF_W_Q4_0, binding.PF_W_F32


@pytest.fixture(scope="module")
def lib():
    need_gpu()
    from prefill_kv_shared_gb300 import build
    build.build()
    return binding.load()


def _weights(wtype, rng, N, K):
    if wtype == Q4:
        w = synth.draw_q4_0(rng, N, K)
        return w, gpu_q4_weights(w), as_f32_matrix(w)
    w = rng.normal(0, 0.05, (N, K)).astype(np.float32)
    return w, bf16_round(w), w


def _A(rng, M, K, scale=1.0):
    return bf16_round(rng.normal(0, scale, (M, K)).astype(np.float32))


GEMM_CASES = [
    (Q4, 1, 128, 64, 128),
    (Q4, 7, 256, 192, 256),
    (Q4, 130, 384, 256, 128),
    (Q4, 300, 200, 1536, 128),
    (Q4, 512, 512, 6144, 128),
    (Q4, 257, 512, 2048, 256),
    (F32, 64, 256, 256, 128),
    (F32, 200, 384, 512, 256),
    (Q4, 512, 256, 1536, 64),
    (Q4, 3, 192, 512, 64),
    (F32, 100, 128, 256, 64),
    (Q4, 1000, 2560, 256, 128),   # 160 tiles of 128 x 128: two M tiles per CTA
    (F32, 1000, 2560, 128, 128),
]


@pytest.mark.parametrize("wtype,M,N,K,bn", GEMM_CASES)
def test_linear_f32(lib, wtype, M, N, K, bn):
    rng = np.random.default_rng(M * 7 + N + K)
    w, w_gpu, w_exact = _weights(wtype, rng, N, K)
    A = _A(rng, M, K)
    a, R = padded_a(A)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    binding.check_op(lib.pfop_linear_f32(wtype, w.ctypes.data, N, K, bn, a.data_ptr(), R, M, out.data_ptr(), None))
    got = out.cpu().numpy()
    ref_tc = A.astype(np.float64) @ w_gpu.astype(np.float64).T
    ref_exact = A.astype(np.float64) @ w_exact.astype(np.float64).T
    assert np.isfinite(got).all()
    assert rel_err(got, ref_tc) < 2e-5
    assert rel_err(got, ref_exact) < 2e-2


@pytest.mark.parametrize("wtype,bn,N,M", [(Q4, 64, 256, 512), (Q4, 128, 256, 512), (Q4, 256, 256, 512),
                                          (F32, 128, 256, 512), (Q4, 128, 2560, 1024), (Q4, 128, 19200, 300)])
def test_linear_row_independent_of_m(lib, wtype, bn, N, M):
    """A row's result is bit-identical whether the launch carries M rows or 1
    (M = 1024 over 2560 columns takes two M tiles per CTA; 300 rows over 150
    tiles take the general persistent form, one row the one-unit form)."""
    rng = np.random.default_rng(3)
    K = 1536
    w, _, _ = _weights(wtype, rng, N, K)
    A = _A(rng, M, K)
    a, R = padded_a(A)
    full = torch.empty((M, N), dtype=torch.float32, device="cuda")
    binding.check_op(lib.pfop_linear_f32(wtype, w.ctypes.data, N, K, bn, a.data_ptr(), R, M, full.data_ptr(), None))
    for row in (0, 129, M - 1):
        a1, R1 = padded_a(A[row:row + 1])
        one = torch.empty((1, N), dtype=torch.float32, device="cuda")
        binding.check_op(lib.pfop_linear_f32(wtype, w.ctypes.data, N, K, bn, a1.data_ptr(), R1, 1, one.data_ptr(), None))
        assert torch.equal(one[0], full[row])


def test_linear_resid_and_bf16_copy(lib):
    rng = np.random.default_rng(11)
    M, N, K = 150, 384, 512
    w, w_gpu, _ = _weights(Q4, rng, N, K)
    A = _A(rng, M, K)
    a, R = padded_a(A)
    x0 = rng.normal(0, 1, (M, N)).astype(np.float32)
    x = torch.from_numpy(x0).cuda()
    xb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_linear_resid(Q4, w.ctypes.data, N, K, a.data_ptr(), R, M, x.data_ptr(), xb.data_ptr(), None))
    want = x0.astype(np.float64) + A.astype(np.float64) @ w_gpu.astype(np.float64).T
    got = x.cpu().numpy()
    assert rel_err(got, want) < 2e-5
    assert torch.equal(xb, x.to(torch.bfloat16))


@pytest.mark.parametrize("act,wtype", [(0, Q4), (1, Q4), (0, F32)])
def test_linear_glu(lib, act, wtype):
    _check_glu(lib, act, wtype, 140, 256, 512)


@pytest.mark.parametrize("M", [100, 300])
def test_linear_glu_192_row_tiles(lib, M):
    """F = 576 (a multiple of 96, not of 128): Q4_0 gate/up interleaved in
    192-row tiles; one and two 128-row M tiles per CTA."""
    _check_glu(lib, 0, Q4, M, 576, 512)


def _check_glu(lib, act, wtype, M, F, K):
    rng = np.random.default_rng(5 + act + M)
    wg, wg_gpu, wg_exact = _weights(wtype, rng, F, K)
    wu, wu_gpu, wu_exact = _weights(wtype, rng, F, K)
    A = _A(rng, M, K, scale=8.0 if wtype == Q4 else 1.0)
    a, R = padded_a(A)
    h = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_linear_glu(wtype, wg.ctypes.data, wu.ctypes.data, F, K, act, a.data_ptr(), R, M,
                                         h.data_ptr(), None))
    got = h.float().cpu().numpy()
    fn = oracle.gelu_tanh if act == 0 else oracle.silu
    g = (A @ wg_gpu.T).astype(np.float32)
    u = (A @ wu_gpu.T).astype(np.float32)
    assert rel_err(got, fn(g) * u) < 1e-2
    ge = (A @ wg_exact.T).astype(np.float32)
    ue = (A @ wu_exact.T).astype(np.float32)
    assert rel_err(got, fn(ge) * ue) < 3e-2


def test_linear_ple(lib):
    rng = np.random.default_rng(21)
    M, P, K, L = 130, 256, 1536, 3
    w, w_gpu, _ = _weights(Q4, rng, P, K)
    A = _A(rng, M, K, scale=8.0)
    a, R = padded_a(A)
    ple_all = bf16_round(rng.normal(0, 1, (M, L, P)).astype(np.float32))
    ple = torch.from_numpy(ple_all).cuda().to(torch.bfloat16)
    il = 1
    out = torch.empty((M, P), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_linear_ple(Q4, w.ctypes.data, P, K, a.data_ptr(), R, M,
                                         ple.data_ptr() + il * P * 2, L * P, out.data_ptr(), None))
    want = oracle.gelu_tanh((A @ w_gpu.T).astype(np.float32)) * ple_all[:, il, :]
    assert rel_err(out.float().cpu().numpy(), want) < 1e-2


@pytest.mark.parametrize("Hq,Hkv,hd,K,M,pos0,with_kv", [
    (8, 1, 256, 1536, 200, 0, True),
    (8, 2, 256, 512, 64, 37, True),
    (4, 1, 64, 256, 64, 0, True),
    (32, 4, 64, 512, 40, 500, True),
    (8, 1, 256, 1536, 1, 777, False),
])
def test_linear_qkv_rope(lib, Hq, Hkv, hd, K, M, pos0, with_kv):
    rng = np.random.default_rng(Hq + hd + M)
    q, kv = Hq * hd, Hkv * hd
    wq, wq_gpu, _ = _weights(Q4, rng, q, K)
    wk, wk_gpu, _ = _weights(Q4, rng, kv, K)
    wv, wv_gpu, _ = _weights(Q4, rng, kv, K)
    A = _A(rng, M, K, scale=8.0)
    a, R = padded_a(A)
    max_ctx = pos0 + M + 3
    qo = torch.empty((M, q), dtype=torch.float16, device="cuda")
    kc = torch.zeros((max_ctx, kv), dtype=torch.float16, device="cuda")
    vc = torch.zeros((max_ctx, kv), dtype=torch.float16, device="cuda")
    binding.check_op(lib.pfop_linear_qkv(Q4, wq.ctypes.data, wk.ctypes.data if with_kv else None,
                                         wv.ctypes.data if with_kv else None, Hq, Hkv, hd, K, 10000.0,
                                         a.data_ptr(), R, M, pos0, max_ctx, qo.data_ptr(), kc.data_ptr(),
                                         vc.data_ptr(), None))
    pos = pos0 + np.arange(M)
    qref = oracle.rope_neox((A @ wq_gpu.T).astype(np.float32).reshape(M, Hq, hd), pos, 10000.0).reshape(M, q)
    assert rel_err(qo.float().cpu().numpy(), qref) < 2e-3
    if with_kv:
        kref = oracle.rope_neox((A @ wk_gpu.T).astype(np.float32).reshape(M, Hkv, hd), pos, 10000.0).reshape(M, kv)
        vref = (A @ wv_gpu.T).astype(np.float32)
        kcn = kc.float().cpu().numpy()
        vcn = vc.float().cpu().numpy()
        assert rel_err(kcn[pos0:pos0 + M], kref) < 2e-3
        assert rel_err(vcn[pos0:pos0 + M], vref) < 2e-3
        assert not kcn[:pos0].any() and not kcn[pos0 + M:].any()
    else:
        assert not kc.any() and not vc.any()


ATTN_CASES = [
    (64, 4, 1, 64, 0, 64),
    (37, 8, 1, 256, 100, 137),
    (200, 8, 2, 256, 0, 200),
    (5, 32, 4, 64, 500, 505),
    (512, 8, 1, 256, 0, 512),
]


def _attn_inputs(rng, M, Hq, Hkv, hd, kv_len):
    q = rng.normal(0, 1, (M, Hq, hd)).astype(np.float16)
    k = rng.normal(0, 1, (kv_len + 5, Hkv, hd)).astype(np.float16)
    v = rng.normal(0, 1, (kv_len + 5, Hkv, hd)).astype(np.float16)
    k[kv_len:] = np.float16(np.nan)  # rows beyond the cache's valid range must not be read
    v[kv_len:] = np.float16(np.nan)
    return q, k, v


@pytest.mark.parametrize("M,Hq,Hkv,hd,pos_base,kv_len", ATTN_CASES)
def test_attention_prefill(lib, M, Hq, Hkv, hd, pos_base, kv_len):
    rng = np.random.default_rng(M + hd + kv_len)
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, hd, kv_len)
    tq, tk, tv = (torch.from_numpy(t).cuda() for t in (q, k, v))
    out = torch.empty((M, Hq * hd), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_attention(0, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), M, Hq, Hkv, hd, pos_base,
                                        kv_len, out.data_ptr(), None))
    want = oracle.attention(q.astype(np.float32), k[:kv_len], v[:kv_len], pos_base + np.arange(M))
    got = out.float().cpu().numpy().reshape(M, Hq, hd)
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() < 1e-2


@pytest.mark.parametrize("Hq,Hkv,hd,kv_len,pos", [
    (8, 1, 256, 512, 511), (8, 1, 256, 8192, 8191), (8, 2, 256, 1000, 999), (4, 1, 64, 64, 63),
    (32, 4, 64, 532, 531), (8, 1, 256, 1, 0), (8, 1, 256, 3000, 1234), (8, 2, 256, 32768, 32767),
    (8, 1, 256, 20000, 9500), (16, 1, 64, 200, 130)])
def test_attention_split_matches_oracle(lib, Hq, Hkv, hd, kv_len, pos):
    """The single-row form (the output row of the KV-shared layers): keys
    [0, pos] of a cache holding kv_len positions, against the oracle, and the
    same bits on a second call."""
    rng = np.random.default_rng(kv_len + hd + pos)
    q, k, v = _attn_inputs(rng, 1, Hq, Hkv, hd, kv_len)
    tq, tk, tv = (torch.from_numpy(t).cuda() for t in (q, k, v))
    outs = []
    for _ in range(2):
        one = torch.zeros((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
        binding.check_op(lib.pfop_attention(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 1, Hq, Hkv, hd, pos,
                                            kv_len, one.data_ptr(), None))
        outs.append(one)
    want = oracle.attention(q.astype(np.float32), k[:kv_len], v[:kv_len], np.array([pos]))
    got = outs[0].float().cpu().numpy().reshape(1, Hq, hd)
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() < 1e-2
    assert torch.equal(outs[0], outs[1])


def test_attention_split_ignores_keys_past_the_row(lib):
    """Keys after the row's position change nothing, bit for bit."""
    rng = np.random.default_rng(77)
    Hq, Hkv, hd, kv_len, pos = 8, 1, 256, 4096, 2500
    q, k, v = _attn_inputs(rng, 1, Hq, Hkv, hd, kv_len)
    k2, v2 = k.copy(), v.copy()
    k2[pos + 1:] = rng.normal(0, 3, k2[pos + 1:].shape).astype(np.float16)
    v2[pos + 1:] = rng.normal(0, 3, v2[pos + 1:].shape).astype(np.float16)
    res = []
    for kk, vv in ((k, v), (k2, v2)):
        tq, tk, tv = (torch.from_numpy(t).cuda() for t in (q, kk, vv))
        one = torch.zeros((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
        binding.check_op(lib.pfop_attention(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 1, Hq, Hkv, hd, pos,
                                            kv_len, one.data_ptr(), None))
        res.append(one)
    assert torch.equal(res[0], res[1])


def test_rmsnorm_gather_and_copy(lib):
    rng = np.random.default_rng(8)
    T, D = 70, 1536
    x = rng.normal(0, 2, (T, D)).astype(np.float32)
    g = rng.normal(0, 0.02, D).astype(np.float32)
    tx = torch.from_numpy(x).cuda()
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_rmsnorm(tx.data_ptr(), 0, T, D, g.ctypes.data, 1e-6, y.data_ptr(), None, None))
    want = oracle.rmsnorm(x, g, 1e-6)
    assert rel_err(y.float().cpu().numpy(), want) < 8e-3
    y1 = torch.empty((1, D), dtype=torch.bfloat16, device="cuda")
    xc = torch.empty((1, D), dtype=torch.float32, device="cuda")
    binding.check_op(lib.pfop_rmsnorm(tx.data_ptr(), T - 1, 1, D, g.ctypes.data, 1e-6, y1.data_ptr(), xc.data_ptr(),
                                      None))
    assert torch.equal(y1[0], y[T - 1])
    assert torch.equal(xc[0], tx[T - 1])


@pytest.mark.parametrize("wtype", [Q4, F32])
def test_embed_and_ple(lib, wtype):
    rng = np.random.default_rng(9)
    V, D, L, P, T = 300, 256, 3, 64, 40
    q4 = wtype == Q4
    tab = synth.draw_q4_0(rng, V, D) if q4 else rng.normal(0, 0.02, (V, D)).astype(np.float32)
    ptab = synth.draw_q4_0(rng, V, L * P) if q4 else rng.normal(0, 0.02, (V, L * P)).astype(np.float32)
    tok = rng.integers(0, V, T).astype(np.int32)
    ttok = torch.from_numpy(tok).cuda()
    x = torch.empty((T, D), dtype=torch.float32, device="cuda")
    ple = torch.empty((T, L * P), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(P)
    binding.check_op(lib.pfop_embed(wtype, tab.ctypes.data, ptab.ctypes.data, V, D, L * P, scale, ttok.data_ptr(), T,
                                    x.data_ptr(), ple.data_ptr(), None))
    np.testing.assert_array_equal(x.cpu().numpy(), oracle.prefill.rows_f32(tab, tok))
    want = bf16_round(oracle.prefill.rows_f32(ptab, tok) * np.float32(scale))
    np.testing.assert_array_equal(ple.float().cpu().numpy(), want)
    bad = torch.tensor([1, V, 2], dtype=torch.int32, device="cuda")
    rc = lib.pfop_embed(wtype, tab.ctypes.data, None, V, D, 0, 1.0, bad.data_ptr(), 3, x.data_ptr(), None, None)
    assert rc == binding.PF_E_DEVICE_TOKEN


def test_kv_copy_roundtrip(lib):
    rng = np.random.default_rng(10)
    L_w, max_ctx, kv, n = 3, 100, 256, 37
    cache = torch.from_numpy(rng.normal(0, 1, (2, L_w, max_ctx, kv)).astype(np.float16)).cuda()
    img = torch.zeros(16 + 2 * L_w * n * kv * 2, dtype=torch.uint8, device="cuda")
    hdr = np.frombuffer(b"KVCP" + np.array([n, L_w, kv], dtype="<i4").tobytes(), dtype=np.int32).copy()
    seg = n * kv * 2
    binding.check_op(lib.pfop_kv_copy(0, cache.data_ptr(), max_ctx * kv, img.data_ptr(), seg, 2 * L_w, seg,
                                      hdr.ctypes.data, None))
    raw = img.cpu().numpy().tobytes()
    assert raw[:4] == b"KVCP" and np.frombuffer(raw[4:16], "<i4").tolist() == [n, L_w, kv]
    body = np.frombuffer(raw[16:], dtype=np.float16).reshape(2, L_w, n, kv)
    np.testing.assert_array_equal(body, cache[:, :, :n].cpu().numpy())
    back = torch.zeros_like(cache)
    k = 20  # restore a prefix of the image
    binding.check_op(lib.pfop_kv_copy(1, back.data_ptr(), max_ctx * kv, img.data_ptr(), seg, 2 * L_w, k * kv * 2,
                                      None, None))
    assert torch.equal(back[:, :, :k], cache[:, :, :k])
    assert not back[:, :, k:].any()


def test_attention_bench_runs_the_same_kernels(lib):
    """The timing entry point leaves the same single-row output as the plain
    call (bit for bit) and reports a positive time, with and without the L2
    scrub."""
    import ctypes as C
    rng = np.random.default_rng(11)
    Hq, Hkv, hd, kv_len = 8, 1, 256, 3000
    q, k, v = _attn_inputs(rng, 1, Hq, Hkv, hd, kv_len)
    tq, tk, tv = (torch.from_numpy(t).cuda() for t in (q, k, v))
    ref = torch.empty((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
    binding.check_op(lib.pfop_attention(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 1, Hq, Hkv, hd, kv_len - 1,
                                        kv_len, ref.data_ptr(), None))
    scrub = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    for sc, nb in ((scrub.data_ptr(), scrub.numel()), (None, 0)):
        out = torch.zeros_like(ref)
        us = C.c_float(0.0)
        binding.check_op(lib.pfop_attention_bench(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 1, Hq, Hkv, hd,
                                                  kv_len - 1, kv_len, out.data_ptr(), sc, nb, 1, 3, C.byref(us),
                                                  None))
        assert us.value > 0
        assert torch.equal(out, ref)
    assert lib.pfop_attention_bench(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 2, Hq, Hkv, hd, kv_len - 2,
                                    kv_len, ref.data_ptr(), None, 0, 0, 1, C.byref(us), None) == binding.PF_E_ARG


def test_kv_copy_bench_restores_exactly(lib):
    import ctypes as C
    rng = np.random.default_rng(12)
    L_w, n, kv = 4, 300, 256
    seg = n * kv * 2
    img = torch.from_numpy(rng.integers(0, 256, 16 + 2 * L_w * seg, dtype=np.uint8)).cuda()
    cache = torch.zeros((2, L_w, n, kv), dtype=torch.float16, device="cuda")
    scrub = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    us = C.c_float(0.0)
    binding.check_op(lib.pfop_kv_copy_bench(1, cache.data_ptr(), n * kv, img.data_ptr(), seg, 2 * L_w, seg,
                                            scrub.data_ptr(), scrub.numel(), 1, 2, C.byref(us), None))
    assert us.value > 0
    got = cache.cpu().numpy().view(np.uint8).reshape(-1)
    np.testing.assert_array_equal(got, img[16:].cpu().numpy())


@pytest.mark.parametrize("wtype,N,K,bn", [(Q4, 1536, 6144, 64), (Q4, 2560, 1536, 128), (Q4, 12288, 1536, 256),
                                          (Q4, 200, 256, 64), (Q4, 32768, 1536, 128), (F32, 384, 512, 128),
                                          (F32, 256, 1024, 256), (Q4, 12288, 1536, 192), (Q4, 500, 512, 192)])
def test_linear_row_stream(lib, wtype, N, K, bn):
    """The one-token projection (CUDA cores, fp32): against float64 on the
    exact Q4_0 decode (its weights are exact in fp32, no bf16 rounding), the
    same bits on a repeated call, ragged N included."""
    rng = np.random.default_rng(N + K + bn)
    w, w_gpu, w_exact = _weights(wtype, rng, N, K)
    A = _A(rng, 1, K)
    a = torch.from_numpy(A).cuda().bfloat16()
    outs = []
    for _ in range(2):
        out = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        binding.check_op(lib.pfop_linear_row(wtype, w.ctypes.data, N, K, bn, a.data_ptr(), out.data_ptr(), 0, None,
                                             None))
        outs.append(out)
    got = outs[0].cpu().numpy()
    ref = A.astype(np.float64)[0] @ (w_exact if wtype == Q4 else w_gpu).astype(np.float64).T
    assert np.isfinite(got).all()
    assert rel_err(got, ref) < 2e-5
    assert torch.equal(outs[0], outs[1])
