"""The tensor-core GEMM in 2-CTA pairs (tcgen05 .cta_group::2): each CTA of a
cluster stages its own 128 rows of A and half of the Q4_0 weight tile, and one
MMA covers 256 rows.  Checked against float64 on the bf16 operands the tensor
cores see and against the oracle's exact Q4_0 decode, bit for bit against the
same GEMM on single CTAs without a k-split (every output element comes from
the same MMA sequence over k), and through every fused epilogue.  Shapes cover ragged M,
one and two 256-row MMA tiles per pair, several work units per pair (the
persistent loop and its accumulator buffers) and all three tile widths."""
import ctypes

import numpy as np
import pytest

import tests.test_gpu_ops as base
from oracle.prefill import as_f32_matrix
from prefill_kv_shared_gb300 import binding, synth
from tests.gpu_util import bf16_round, gpu_q4_weights, need_gpu, padded_a, rel_err, torch

pytestmark = pytest.mark.gpu

Q4 = binding.PF_W_Q4_0


@pytest.fixture(scope="module")
def lib():
    need_gpu()
    from prefill_kv_shared_gb300 import build
    build.build()
    lib = binding.load()
    yield lib
    lib.pfop_set_gemm_pairs(0)


@pytest.fixture
def pairs(lib):
    binding.check_op(lib.pfop_set_gemm_pairs(1))
    yield
    binding.check_op(lib.pfop_set_gemm_pairs(0))


def _gemm(lib, mode, w, N, K, bn, a, R, M):
    binding.check_op(lib.pfop_set_gemm_pairs(mode))
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    binding.check_op(lib.pfop_linear_f32(Q4, w.ctypes.data, N, K, bn, a.data_ptr(), R, M, out.data_ptr(), None))
    return out


def _gemm_split(lib, split, w, N, K, bn, a, R, M):
    """One launch through the timing entry point: split 1 = single CTAs
    without a k-split, -1 = CTA pairs."""
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    us = ctypes.c_float()
    binding.check_op(lib.pfop_linear_bench(Q4, w.ctypes.data, N, K, bn, split, a.data_ptr(), R, M, out.data_ptr(), 0,
                                           1, ctypes.byref(us), None))
    return out


PAIR_CASES = [
    (1, 256, 512, 128),
    (7, 384, 1536, 256),
    (130, 384, 512, 128),
    (256, 512, 1536, 128),
    (300, 576, 1536, 192),
    (513, 512, 2048, 256),
    (512, 2560, 1536, 128),
    (1000, 2560, 256, 128),   # 80 units of 256 rows: two MMA tiles per pair
    (200, 25600, 256, 128),   # 200 units on the pairs: several per pair, two accumulator buffers
    (300, 25600, 256, 128),   # two MMA tiles per unit, several units per pair
    (250, 19200, 256, 192),
    (600, 12288, 256, 256),   # one accumulator buffer (512 TMEM columns), several units per pair
]


@pytest.mark.parametrize("M,N,K,bn", PAIR_CASES)
def test_pairs_match_single_ctas(lib, M, N, K, bn):
    rng = np.random.default_rng(M * 3 + N + K + bn)
    w = synth.draw_q4_0(rng, N, K)
    A = bf16_round(rng.normal(0, 1, (M, K)).astype(np.float32))
    a, R = padded_a(A)
    try:
        got = _gemm(lib, 1, w, N, K, bn, a, R, M)
    finally:
        lib.pfop_set_gemm_pairs(0)
    g = got.cpu().numpy()
    assert np.isfinite(g).all()
    assert rel_err(g, A.astype(np.float64) @ gpu_q4_weights(w).astype(np.float64).T) < 2e-5
    assert rel_err(g, A.astype(np.float64) @ as_f32_matrix(w).astype(np.float64).T) < 2e-2
    # the same bits as single CTAs over the same k-order (no k-split), and as
    # the timing entry point's pair launch
    assert torch.equal(got, _gemm_split(lib, 1, w, N, K, bn, a, R, M))
    assert torch.equal(got, _gemm_split(lib, -1, w, N, K, bn, a, R, M))


def test_glu_in_pairs(lib, pairs):
    base._check_glu(lib, 0, Q4, 300, 1536, 512)  # 256-row gate/up tiles
    base._check_glu(lib, 1, Q4, 140, 576, 512)   # 192-row tiles


@pytest.mark.parametrize("Hq,Hkv,hd,K,M,pos0,with_kv", [
    (8, 1, 256, 1536, 200, 0, True),
    (32, 4, 64, 512, 300, 500, True),
    (8, 1, 256, 1536, 1, 777, False),
])
def test_qkv_rope_in_pairs(lib, pairs, Hq, Hkv, hd, K, M, pos0, with_kv):
    base.test_linear_qkv_rope(lib, Hq, Hkv, hd, K, M, pos0, with_kv)


def test_resid_and_ple_in_pairs(lib, pairs):
    base.test_linear_resid_and_bf16_copy(lib)
    base.test_linear_ple(lib)


@pytest.mark.parametrize("bn,N,M", [(128, 2560, 1024), (256, 256, 512), (192, 576, 300)])
def test_row_independent_of_m_in_pairs(lib, pairs, bn, N, M):
    base.test_linear_row_independent_of_m(lib, Q4, bn, N, M)
