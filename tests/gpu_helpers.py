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


# Gradients (dQ, dK, dV) against the float64 oracle, relative to each tensor's scale:
# max abs error <= 2e-2 * max |ref| and mean abs error <= 5e-3 * mean |ref|. Derivation:
# the kernel rounds P and dS to bf16 for the tensor core and the outputs to bf16 (unit
# roundoff u = 2^-9 each), and forms D = rowsum(dO * O) from the bf16 forward output, so
# each gradient element carries a few u of relative error about its own scale; 2e-2 is
# about 10 u on the worst element, 5e-3 about 2.5 u on average.
GRAD_MAX_REL = 2e-2
GRAD_MEAN_REL = 5e-3


def assert_grad_close(g_gpu: np.ndarray, g_ref: np.ndarray, what: str = ""):
    assert g_gpu.shape == g_ref.shape
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite gradient"
    err = np.abs(g_gpu - g_ref)
    scale_max = max(float(np.abs(g_ref).max()), 1e-30)
    scale_mean = max(float(np.abs(g_ref).mean()), 1e-30)
    msg = (f"{what}: max err {err.max():.3e} (scale {scale_max:.3e}), mean err {err.mean():.3e} "
           f"(scale {scale_mean:.3e})")
    assert err.max() <= GRAD_MAX_REL * scale_max, msg
    assert err.mean() <= GRAD_MEAN_REL * scale_mean, msg
    return err.max() / scale_max, err.mean() / scale_mean
