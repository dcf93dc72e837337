"""Helpers for the GPU parity tests: numpy bit patterns <-> CUDA tensors."""
import numpy as np
import torch

DEV = "cuda:0"

_VIEW = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32, np.dtype(np.uint8): np.uint8,
         np.dtype(np.int32): np.int32, np.dtype(np.float32): np.float32, np.dtype(np.float16): np.float16,
         np.dtype(np.int16): np.int16, np.dtype(np.int64): np.int64}


def dev(a) -> torch.Tensor:
    """numpy array -> CUDA tensor with the same bytes (uint16/uint32 travel as int16/int32)."""
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(_VIEW[a.dtype])).to(DEV)


def host(t: torch.Tensor, dtype) -> np.ndarray:
    """CUDA tensor -> numpy array reinterpreted as ``dtype``."""
    return t.cpu().numpy().view(dtype)


def empty(shape, dtype=torch.int16) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=DEV)


def zeros_bytes(n: int) -> torch.Tensor:
    return torch.zeros(max(int(n), 16), dtype=torch.uint8, device=DEV)


def pinned(a) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(_VIEW[a.dtype])).pin_memory()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    u = t.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def assert_attn_close(got, want, max_abs=2e-2, mean_abs=2e-3, what=""):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= max_abs, f"{what}: max-abs {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean-abs {err.mean():.3e} > {mean_abs}"
    return err.max(), err.mean()
