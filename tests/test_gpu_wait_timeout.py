"""The failure path of the kernels' bounded waits, made to run on purpose.

Every wait of the tensor-core GEMM on a pipeline barrier gives up after a
bound (about 2 s of SM clock), records the cause in the device error word
and lets the kernel unwind: copies already issued are drained, TMEM is freed,
and the host sees PF_E_DEVICE_TIMEOUT instead of a hung GPU.  Here the copy
producer of the only CTA withholds one pipeline stage (it issues nothing
more, so no copy is left in flight), the consumers' waits for that stage run
out, and the call must come back with the timeout status; afterwards the
same GPU context must compute the plain GEMM correctly.  No fault, trap or
endless wait is involved: the kernel returns on its own."""
import time

import numpy as np
import pytest

from oracle.prefill import as_f32_matrix
from prefill_kv_shared_gb300 import binding, synth
from tests.gpu_util import bf16_round, gpu_q4_weights, need_gpu, padded_a, rel_err, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    need_gpu()
    from prefill_kv_shared_gb300 import build
    build.build()
    return binding.load()


def test_withheld_copy_times_out_and_context_stays_usable(lib):
    rng = np.random.default_rng(21)
    # one 128 x 128 tile, K = 1536: 24 k-blocks in 12 pipeline stages; the
    # first three stages' weight copies are issued before the main loop, so
    # stage 5 is withheld from inside it
    N, K, M, bn = 128, 1536, 128, 128
    w = synth.draw_q4_0(rng, N, K)
    A = bf16_round(rng.normal(0, 1, (M, K)).astype(np.float32))
    a, R = padded_a(A)
    out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    rc = lib.pfop_linear_wait_test(binding.PF_W_Q4_0, w.ctypes.data, N, K, bn, a.data_ptr(), R, M, out.data_ptr(),
                                   5, None)
    took = time.perf_counter() - t0
    assert rc == binding.PF_E_DEVICE_TIMEOUT, lib.pfop_last_error()
    assert b"bounded wait" in lib.pfop_last_error()
    assert took < 30.0
    # the context is intact: the plain GEMM on the same GPU gives the right result
    ref = A.astype(np.float64) @ gpu_q4_weights(w).astype(np.float64).T
    for stage in (-1, 1000):  # no stage withheld; a stage past the last one
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.pfop_linear_wait_test(binding.PF_W_Q4_0, w.ctypes.data, N, K, bn, a.data_ptr(), R, M,
                                       out.data_ptr(), stage, None)
        assert rc == binding.PF_OK, lib.pfop_last_error()
        got = out.cpu().numpy()
        assert np.isfinite(got).all() and rel_err(got, ref) < 2e-5
    assert rel_err(got, A.astype(np.float64) @ as_f32_matrix(w).astype(np.float64).T) < 2e-2
