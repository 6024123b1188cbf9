"""Tolerance check and sampled-entry selection shared by the GPU parity tests.

Bar (per output tensor, and per shard slice of dA, dB, da): relative Frobenius error
<= 5e-3 and max abs error <= 2e-2 * max|ref|, the GPU result upconverted to fp64.
"""
import numpy as np
import torch

REL_FRO = 5e-3
MAX_ABS_FRAC = 2e-2


def errors(gpu, ref) -> tuple[float, float, float]:
    g = gpu.detach().to("cpu", torch.float64).numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    d = g - r
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
    mx = float(np.abs(r).max()) if r.size else 0.0
    return float(rel), float(np.abs(d).max()) if d.size else 0.0, mx


def assert_close(name: str, gpu, ref, rel_fro: float = REL_FRO, max_abs_frac: float = MAX_ABS_FRAC) -> None:
    rel, mad, mx = errors(gpu, ref)
    assert np.isfinite(rel) and rel <= rel_fro, f"{name}: rel Frobenius error {rel:.3e} > {rel_fro}"
    assert mad <= max_abs_frac * mx + 1e-30, f"{name}: max abs error {mad:.3e} > {max_abs_frac} * {mx:.3e}"


# One rounding of a normally distributed value to bf16 leaves a relative Frobenius error of
# about 1.7e-3 (the RMS of a uniform error of half an 8-bit-mantissa ulp, relative to the
# value). Independent roundings along a chain of n bf16 stores add in quadrature.
BF16_ROUNDING_REL = 1.7e-3


def bf16_chain_tol(n: int) -> tuple[float, float]:
    """Bar for an output that passes through n bf16 roundings: twice the expected relative
    Frobenius error sqrt(n) * 1.7e-3, and the same max abs error bound as every other
    output, 2e-2 * max|ref|."""
    rel = 2.0 * BF16_ROUNDING_REL * float(np.sqrt(n))
    return rel, MAX_ABS_FRAC


def sample_rows_cols(T: int, f: int, t: int, seed: int = 1234, n: int = 64):
    """64 seeded tokens plus the first and last; 64 seeded MLP columns plus the first and
    last column of every shard."""
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(T, size=min(n, T), replace=False), [0, T - 1]]))
    fs = f // t
    edges = np.array([[i * fs, (i + 1) * fs - 1] for i in range(t)]).ravel()
    cols = np.unique(np.concatenate([rng.choice(f, size=min(n, f), replace=False), edges]))
    return rows.astype(np.int64), cols.astype(np.int64)
