"""Pins for the oracle's bias + dropout + residual-add step: its Philox4x32-10 against a
library implementation, mask statistics, special cases, and finite differences."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rand(T, h, f, seed):
    rng = np.random.default_rng(seed)
    return {"X": rng.standard_normal((T, h)), "A": rng.standard_normal((h, f)) * 0.5,
            "a": rng.standard_normal(f) * 0.3, "B": rng.standard_normal((f, h)) * 0.5,
            "b": rng.standard_normal(h) * 0.3}


_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def k(out_ptr, c_ptr, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * i)
    c1 = tl.load(c_ptr + 4 * i + 1)
    c2 = tl.load(c_ptr + 4 * i + 2)
    c3 = tl.load(c_ptr + 4 * i + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + 4 * i, a)
    tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c)
    tl.store(out_ptr + 4 * i + 3, d)

cases = json.loads(sys.argv[1])
res = []
for seed, ctrs in cases:
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.int32)  # two's complement bit patterns
    out = torch.zeros(len(ctrs), dtype=torch.int32)
    k[(1,)](out, c, seed, N=len(ctrs) // 4)
    res.append([v & 0xFFFFFFFF for v in out.tolist()])
print(json.dumps(res))
"""


def test_philox_matches_library_implementation():
    """Triton's philox (tl.philox, run by its CPU interpreter) is an independent library
    implementation of the same Philox4x32-10; both must agree word for word."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(7)
    cases = []
    for seed in (0, 1, 0x123456789ABCDEF0, 0xFFFFFFFFFFFFFFFF):
        ctrs = [0, 0, 0, 0, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF]
        ctrs += [int(v) for v in rng.integers(0, 2**32, size=8, dtype=np.uint64)]
        cases.append((seed, ctrs))
    import json
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX, json.dumps(cases)], capture_output=True,
                       text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.skip(f"triton interpreter unavailable: {r.stderr[-300:]}")
    lib = json.loads(r.stdout.strip().splitlines()[-1])
    for (seed, ctrs), got in zip(cases, lib):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(0, len(ctrs), 4):
            assert oracle.philox4x32_10(ctrs[i:i + 4], key) == tuple(got[i:i + 4]), (seed, ctrs[i:i + 4])


def test_dropout_mask_statistics_and_determinism():
    for p in (0.1, 0.5, 0.9):
        keep = oracle.dropout_keep(512, 1024, p, seed=1234, offset=5)
        n = keep.size
        frac_drop = 1.0 - keep.mean()
        assert abs(frac_drop - p) < 5 * np.sqrt(p * (1 - p) / n), (p, frac_drop)
        # columns and rows are not stuck
        assert keep.mean(0).std() < 0.1 and keep.mean(1).std() < 0.1
    a = oracle.dropout_keep(64, 64, 0.3, seed=9, offset=0)
    assert np.array_equal(a, oracle.dropout_keep(64, 64, 0.3, seed=9, offset=0))
    assert not np.array_equal(a, oracle.dropout_keep(64, 64, 0.3, seed=9, offset=1))
    assert not np.array_equal(a, oracle.dropout_keep(64, 64, 0.3, seed=10, offset=0))
    assert oracle.dropout_keep(8, 16, 0.0, seed=3).all()
    with pytest.raises(ValueError):
        oracle.dropout_keep(8, 16, 1.0, seed=3)


def test_mask_element_is_its_philox_word():
    """Element e = r*h + c takes word e % 4 of Philox on counter (e // 4, offset)."""
    T, h, p, seed, offset = 3, 24, 0.4, 0xDEADBEEFCAFE, 77
    keep = oracle.dropout_keep(T, h, p, seed, offset)
    p24 = int(np.floor(p * 2**24))
    for e in range(T * h):
        q = e // 4
        words = oracle.philox4x32_10([q & 0xFFFFFFFF, q >> 32, offset & 0xFFFFFFFF, offset >> 32],
                                     [seed & 0xFFFFFFFF, seed >> 32])
        assert keep.flat[e] == int((words[e % 4] >> 8) >= p24)


def test_no_dropout_is_residual_plus_block():
    inp = _rand(5, 8, 16, seed=1)
    rng = np.random.default_rng(2)
    R, dZ = rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    out = oracle.fwd_bwd_residual_dropout(dict(inp, dY=dZ), R, dZ, p=0.0, seed=4)
    _, _, Y = oracle.forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"])
    np.testing.assert_allclose(out["Z"], R + Y, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(out["dY"], dZ)


@pytest.mark.parametrize("p", [0.2, 0.6])
def test_dropout_block_finite_differences(p):
    T, h, f = 3, 4, 8
    inp = _rand(T, h, f, seed=3)
    rng = np.random.default_rng(4)
    R, dZ = rng.standard_normal((T, h)), rng.standard_normal((T, h))
    seed, offset = 99, 3
    out = oracle.fwd_bwd_residual_dropout(dict(inp, dY=dZ), R, dZ, p=p, seed=seed, offset=offset)
    assert 0 < out["keep"].sum() < T * h  # both kept and dropped elements occur

    def loss(d, Rr):
        keep = oracle.dropout_keep(T, h, p, seed, offset)
        _, _, Y = oracle.forward(d["X"], d["A"], d["a"], d["B"], d["b"])
        return float((oracle.residual_dropout(Y, Rr, keep, p) * dZ).sum())

    grads = {"X": out["dX"], "A": out["dA"], "a": out["da"], "B": out["dB"], "b": out["db"]}
    for name, g in grads.items():
        base = inp[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            hi = dict(inp); hi[name] = base.copy(); hi[name][idx] += eps
            lo = dict(inp); lo[name] = base.copy(); lo[name][idx] -= eps
            fd[idx] = (loss(hi, R) - loss(lo, R)) / (2 * eps)
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-7, err_msg=name)
    fdR = np.empty_like(R)
    for idx in np.ndindex(R.shape):
        hi = R.copy(); hi[idx] += 1e-6
        lo = R.copy(); lo[idx] -= 1e-6
        fdR[idx] = (loss(inp, hi) - loss(inp, lo)) / 2e-6
    np.testing.assert_allclose(out["dR"], fdR, rtol=1e-6, atol=1e-7)
