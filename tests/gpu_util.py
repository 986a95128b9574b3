"""Helpers shared by the GPU tests: moving seeded inputs to the device and
comparing against the oracle."""
import numpy as np
import torch

LOGP_ATOL = 2e-3      # nats: max |logp_gpu - logp_oracle|
GRAD_REL_L2 = 1e-2    # relative L2 error of dH and dW against the oracle


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    nb = float(np.linalg.norm(b))
    return float(np.linalg.norm(np.asarray(a, np.float64) - b)) / (nb if nb > 0 else 1.0)


def assert_logp_close(gpu: np.ndarray, ref: np.ndarray, atol=LOGP_ATOL):
    gpu = np.asarray(gpu, np.float64)
    err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    assert np.all(np.isfinite(gpu)), "non-finite logp"
    assert err <= atol, f"max |dlogp| = {err:.3e} > {atol}"
    return err


def assert_grad_close(gpu: np.ndarray, ref: np.ndarray, tol=GRAD_REL_L2, what="grad"):
    e = rel_l2(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"non-finite {what}"
    assert e <= tol, f"{what}: relative L2 {e:.3e} > {tol}"
    return e
