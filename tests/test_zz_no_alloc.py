"""The allocation-free single-row attention (pfop_attention_split_noalloc).

It serves callers that may not allocate device memory when this step runs
(a memory budget already handed out, a server that allows no allocation
after start-up, an embedder whose own allocator owns the device); its
scratch is one fixed array inside the library.  It runs the same kernels
with the same cut of the keys into ranges as the allocating entry point
(pfop_attention, split mode), so the two must agree bit for bit, on two
calls in a row that reuse the shared array, and both must match the oracle
within the attention tolerance of the other GPU tests.  This file is
collected last on purpose."""
import numpy as np
import pytest

from oracle import prefill as oracle
from prefill_kv_shared_gb300 import binding
from tests.gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu

TOL = 1e-2  # the attention parity tolerance of the other GPU tests


@pytest.fixture(scope="module")
def lib():
    need_gpu()
    from prefill_kv_shared_gb300 import build
    build.build()
    return binding.load()


def _inputs(seed, Hq, Hkv, hd, kv_len):
    rng = np.random.default_rng(seed)
    q = rng.normal(0, 1, (1, Hq * hd)).astype(np.float16)
    k = rng.normal(0, 1, (kv_len, Hkv * hd)).astype(np.float16)
    v = rng.normal(0, 1, (kv_len, Hkv * hd)).astype(np.float16)
    return q, k, v


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 1, 256), (32, 4, 64)])
def test_noalloc_matches_allocating_entry_point_twice(lib, Hq, Hkv, hd):
    # the second call is shorter, so stale range states of the first call
    # remain in the shared array past the ones it writes
    for call, (seed, kv_len) in enumerate([(1, 1500), (2, 700)]):
        q, k, v = _inputs(seed, Hq, Hkv, hd, kv_len)
        tq, tk, tv = (torch.from_numpy(t).cuda() for t in (q, k, v))
        want = torch.empty((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
        got = torch.full((1, Hq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.check_op(lib.pfop_attention(1, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), 1, Hq, Hkv, hd,
                                            kv_len - 1, kv_len, want.data_ptr(), None))
        binding.check_op(lib.pfop_attention_split_noalloc(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), Hq, Hkv, hd,
                                                          kv_len - 1, kv_len, got.data_ptr(), None))
        assert torch.equal(got, want), f"call {call}: differs from the allocating entry point"
        ref = oracle.attention(q.reshape(1, Hq, hd).astype(np.float32), k.reshape(kv_len, Hkv, hd),
                               v.reshape(kv_len, Hkv, hd), np.array([kv_len - 1]))
        err = np.abs(got.float().cpu().numpy().reshape(1, Hq, hd) - ref).max()
        assert np.isfinite(err) and err <= TOL, f"call {call}: max |err| {err} against the oracle"


def test_noalloc_refuses_requests_beyond_the_array(lib):
    # 4096 query heads of 256 over 256 KV heads: one cluster of key ranges
    # per KV head, whose folded states need 256 * (16 * 256 + 32) floats,
    # more than the 2^19 the array holds.  The buffers are full size for the
    # request, so even a call that wrongly went ahead would stay inside them.
    Hq, Hkv, hd, kv_len = 4096, 256, 256, 64
    q, k, v = (torch.from_numpy(t).cuda() for t in _inputs(3, Hq, Hkv, hd, kv_len))
    out = torch.empty((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
    rc = lib.pfop_attention_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), Hq, Hkv, hd, kv_len - 1, kv_len,
                                          out.data_ptr(), None)
    assert rc == binding.PF_E_ARG
    assert b"scratch" in lib.pfop_last_error()


def test_noalloc_refuses_shapes_the_kernels_do_not_take(lib):
    # refused on the host with PF_E_ARG; the buffers are large enough for
    # every request below, so nothing reaches memory it does not own
    q, k, v = (torch.from_numpy(t).cuda() for t in _inputs(4, 8, 2, 256, 256))
    out = torch.empty(8 * 256, dtype=torch.bfloat16, device="cuda")
    for Hq, Hkv, hd in [(8, 2, 128), (6, 4, 64), (8, 3, 64)]:
        rc = lib.pfop_attention_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), Hq, Hkv, hd, 10, 64,
                                              out.data_ptr(), None)
        assert rc == binding.PF_E_ARG, (Hq, Hkv, hd)
    rc = lib.pfop_attention_split_noalloc(q.data_ptr() + 2, k.data_ptr(), v.data_ptr(), 8, 2, 64, 10, 64,
                                          out.data_ptr(), None)
    assert rc == binding.PF_E_ARG and b"aligned" in lib.pfop_last_error()
