"""The allocation-free single-row attention (pfop_attention_split_noalloc).

It serves callers that may not allocate device memory when this step runs;
its scratch is one fixed array inside the library.  Its results must match
the allocating entry point (pfop_attention, split mode) within the
tolerance the attention tests use, on two calls in a row that reuse the
shared array.  This file is collected last on purpose."""
import numpy as np
import pytest

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
    q = torch.from_numpy(rng.normal(0, 1, (1, Hq * hd)).astype(np.float16)).cuda()
    k = torch.from_numpy(rng.normal(0, 1, (kv_len, Hkv * hd)).astype(np.float16)).cuda()
    v = torch.from_numpy(rng.normal(0, 1, (kv_len, Hkv * hd)).astype(np.float16)).cuda()
    return q, k, v


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 1, 256), (32, 4, 64)])
def test_noalloc_matches_allocating_entry_point_twice(lib, Hq, Hkv, hd):
    for call, (seed, kv_len) in enumerate([(1, 1500), (2, 700)]):
        q, k, v = _inputs(seed, Hq, Hkv, hd, kv_len)
        want = torch.empty((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
        got = torch.full((1, Hq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.check_op(lib.pfop_attention(1, q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, Hq, Hkv, hd,
                                            kv_len - 1, kv_len, want.data_ptr(), None))
        binding.check_op(lib.pfop_attention_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), Hq, Hkv, hd,
                                                          kv_len - 1, kv_len, got.data_ptr(), None))
        diff = (got.float() - want.float()).abs().max().item()
        assert np.isfinite(diff) and diff <= TOL, f"call {call}: max |diff| {diff}"


def test_noalloc_refuses_requests_beyond_the_array(lib):
    # 16 query heads of 256 on one KV head, keys cut into 148 ranges: the
    # range states need 16 * 148 * 260 floats, more than the 2^19 the array
    # holds.  The buffers are full size for the request, so even a call that
    # wrongly went ahead would stay inside them.
    Hq, Hkv, hd, kv_len = 16, 1, 256, 148 * 64
    q, k, v = _inputs(3, Hq, Hkv, hd, kv_len)
    out = torch.empty((1, Hq * hd), dtype=torch.bfloat16, device="cuda")
    rc = lib.pfop_attention_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), Hq, Hkv, hd, kv_len - 1, kv_len,
                                          out.data_ptr(), None)
    assert rc == binding.PF_E_ARG
    assert b"scratch" in lib.pfop_last_error()
