"""Shared helpers of the GPU parity tests (host <-> device marshalling and the
comparison rules)."""
import numpy as np
import torch

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev_bits(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """uint16 storage bits -> device tensor of the half type."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).to(device)


def dev(x, device="cuda"):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device)


def integer_rows(rng, n, dim, lo=-3, hi=3):
    """Small integers: exact in f16 / bf16 and in every fp32 partial sum."""
    return rng.integers(lo, hi + 1, size=(n, dim)).astype(np.float64)


def assert_scores(got: torch.Tensor, ref: np.ndarray, lq: int):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-3 * max(lq, 1)), f"max |score diff| {err.max()} > 1e-3 * Lq"


def assert_argmax(got: torch.Tensor, ref: np.ndarray, gap: np.ndarray):
    got = got.cpu().numpy()
    assert got.shape == ref.shape
    clear = gap >= 1e-3
    bad = clear & (got != ref)
    assert not bad.any(), f"{bad.sum()} argmax mismatches where the top-2 gap >= 1e-3"
    # sentinels are decided by the masks alone and must agree everywhere
    assert np.array_equal(got == -1, ref == -1)


def assert_grad(got: torch.Tensor, ref: np.ndarray):
    got = got.cpu().numpy().astype(np.float64)
    floor = 1e-2 * np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    tol = 1e-3 * np.maximum(np.abs(ref), floor)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} gradient entries beyond 1e-3 relative (max |d| {np.abs(got - ref).max()})"


def assert_grad_rounded(got: torch.Tensor, ref: np.ndarray, dtype: str):
    """Gradients returned in the input's 16-bit type: the fp32 kernel result
    (within the gradient tolerance of ref) is rounded once more, so allow one
    unit in the last place of that type on top of the tolerance."""
    got = got.float().cpu().numpy().astype(np.float64)
    floor = 1e-2 * np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    mant = {"f16": 10, "bf16": 7}[dtype]
    mag = np.maximum(np.abs(ref), np.finfo(np.float64).tiny)
    ulp = np.exp2(np.floor(np.log2(mag)) - mant)
    tol = 1e-3 * np.maximum(np.abs(ref), floor) + ulp
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} gradient entries beyond 1e-3 relative + 1 ulp (max |d| {np.abs(got - ref).max()})"
