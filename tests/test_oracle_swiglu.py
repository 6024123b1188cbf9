"""Pins for the oracle's SwiGLU block: SiLU against the library routine, torch autograd,
finite differences and the shard-sum invariant."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(T, h, f, seed):
    rng = np.random.default_rng(seed)
    return {"X": rng.standard_normal((T, h)), "A": rng.standard_normal((h, f)) * 0.5,
            "Wg": rng.standard_normal((h, f)) * 0.5, "B": rng.standard_normal((f, h)) * 0.5,
            "dY": rng.standard_normal((T, h))}


def test_silu_against_library_and_closed_forms():
    xs = np.linspace(-12, 12, 481)
    ref = torch.nn.functional.silu(torch.tensor(xs)).numpy()
    np.testing.assert_allclose(oracle.silu(xs), ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu([0.0])[0] == 0.0 and abs(oracle.silu_grad([0.0])[0] - 0.5) < 1e-15
    np.testing.assert_allclose(oracle.silu([40.0]), [40.0], rtol=1e-15)
    assert abs(oracle.silu([-40.0])[0]) < 1e-15
    eps = 1e-6
    fd = (oracle.silu(xs + eps) - oracle.silu(xs - eps)) / (2 * eps)
    np.testing.assert_allclose(oracle.silu_grad(xs), fd, atol=1e-8)
    # x * sigma(x) with sigma written through tanh: sigma(x) = (1 + tanh(x/2)) / 2
    # (1 + tanh) cancels for very negative x in this form, hence the small absolute floor
    np.testing.assert_allclose(oracle.silu(xs), [x * 0.5 * (1 + math.tanh(x / 2)) for x in xs], rtol=1e-13,
                               atol=1e-15)


def test_swiglu_matches_torch_autograd():
    inp = _rand(5, 6, 12, seed=1)
    tt = {k: torch.tensor(v, requires_grad=k != "dY") for k, v in inp.items()}
    Y = (torch.nn.functional.silu(tt["X"] @ tt["A"]) * (tt["X"] @ tt["Wg"])) @ tt["B"]
    (Y * tt["dY"]).sum().backward()
    out = oracle.swiglu_fwd_bwd(inp)
    np.testing.assert_allclose(out["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    for k, g in (("dX", "X"), ("dA", "A"), ("dWg", "Wg"), ("dB", "B")):
        np.testing.assert_allclose(out[k], tt[g].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=k)


def test_swiglu_finite_differences():
    T, h, f = 3, 4, 8
    inp = _rand(T, h, f, seed=2)
    out = oracle.swiglu_fwd_bwd(inp)

    def loss(d):
        return float((oracle.swiglu_fwd_bwd(d)["Y"] * d["dY"]).sum())

    for name, gname in (("X", "dX"), ("A", "dA"), ("Wg", "dWg"), ("B", "dB")):
        base = inp[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            hi = dict(inp); hi[name] = base.copy(); hi[name][idx] += eps
            lo = dict(inp); lo[name] = base.copy(); lo[name][idx] -= eps
            fd[idx] = (loss(hi) - loss(lo)) / (2 * eps)
        np.testing.assert_allclose(out[gname], fd, rtol=1e-6, atol=1e-7, err_msg=gname)


def test_swiglu_shard_sum_invariant():
    """(SiLU(XA) * XWg) B = sum_i (SiLU(XA_i) * XWg_i) B_i: one sum for any t."""
    inp = _rand(6, 8, 16, seed=3)
    full = oracle.swiglu_fwd_bwd(inp)
    for t in (1, 2, 4, 8, 16):
        sh = oracle.swiglu_sharded(inp, t, parts=True)
        for k in ("Y", "dX", "dA", "dWg", "dB"):
            np.testing.assert_allclose(sh[k], full[k], rtol=1e-12, atol=1e-12, err_msg=f"{k} t={t}")
        np.testing.assert_allclose(sh["Y_part"].sum(0), full["Y"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sh["dX_part"].sum(0), full["dX"], rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.swiglu_sharded(inp, 3)


def test_swiglu_gate_of_zero_blocks_everything():
    inp = _rand(4, 6, 8, seed=4)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    out = oracle.swiglu_fwd_bwd(inp)
    np.testing.assert_array_equal(out["Y"], 0.0)
    np.testing.assert_array_equal(out["dA"], 0.0)
    np.testing.assert_array_equal(out["dB"], 0.0)


def test_swiglu_sampled_matches_full_on_bf16_inputs():
    from megatron_tensor_transformer_tcgen05_gb300.inputs import make_swiglu_inputs
    inp = make_swiglu_inputs(40, 24, 64, seed=3, sdy=1.0, sw=0.2)
    full = oracle.swiglu_fwd_bwd(inp)
    rows, cols = np.array([0, 9, 39]), np.array([0, 31, 32, 63])
    s = oracle.swiglu_sampled_bf16(inp, rows, cols)
    np.testing.assert_allclose(s["Y_rows"], full["Y"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dX_rows"], full["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dA_cols"], full["dA"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dWg_cols"], full["dWg"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dB_rows"], full["dB"][cols], rtol=1e-12, atol=1e-12)
