"""Helpers shared by the GPU parity tests (argument marshalling and tolerance checks)."""
import numpy as np
import pytest

# Tolerances (stated with the workloads): O max abs 2e-2 and mean abs 2e-3 against the
# float64 oracle, LSE max abs 1e-2; masks and CSR indices bit-exact.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-2


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def to_dev(bits: np.ndarray):
    """uint16 bf16 bit patterns -> torch.bfloat16 CUDA tensor (same bits)."""
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bf16_to_f64(t) -> np.ndarray:
    """CUDA bf16 tensor -> float64 numpy (exact)."""
    torch = torch_cuda()
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def assert_attention_close(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
                           what: str = ""):
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    err = np.abs(o_gpu - o_ref)
    both_inf = np.isneginf(lse_gpu) & np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), np.isneginf(lse_ref)), f"{what}: empty-row pattern differs"
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(lse_gpu - lse_ref))
    msg = f"{what}: O max {err.max():.3e} mean {err.mean():.3e}, LSE max {lerr.max():.3e}"
    assert err.max() <= O_MAX_ABS, msg
    assert err.mean() <= O_MEAN_ABS, msg
    assert lerr.max() <= LSE_MAX_ABS, msg
    return err.max(), err.mean(), lerr.max()
