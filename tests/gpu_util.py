"""Helpers for the GPU tests (torch for device memory only)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")


def to_bf16(x: np.ndarray):
    """fp32 numpy -> bf16 torch tensor on the GPU (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda().to(torch.bfloat16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def padded_a(A: np.ndarray, rows: int | None = None):
    """A [M, K] as a bf16 device buffer with at least 128 rows (zeros after M)."""
    M, K = A.shape
    R = rows or max(128, (M + 127) // 128 * 128)
    buf = torch.zeros((R, K), dtype=torch.bfloat16, device="cuda")
    buf[:M] = to_bf16(A)
    return buf, R


def gpu_q4_weights(blocks: np.ndarray) -> np.ndarray:
    """The values the GEMM multiplies for Q4_0 weights: the scale rounded to
    bf16, times (nibble - 8), rounded to bf16."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float32)
    d = bf16_round(d)
    qs = blocks[..., 2:18]
    n = np.concatenate([(qs & 0xF), (qs >> 4)], axis=-1).astype(np.float32) - 8.0
    w = bf16_round(d[..., None] * n)
    return w.reshape(*blocks.shape[:-2], blocks.shape[-2] * 32)


def rel_err(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))
