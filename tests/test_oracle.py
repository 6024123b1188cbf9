"""Pins for the fp64 CPU oracle: values the pages print, closed forms, invariants,
library special cases and finite differences. None of these needs a GPU."""
import math

import numpy as np
import pytest
import torch

import oracle
from golden_io import load
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_inputs, WORKLOADS

ACTS = ("gelu_tanh", "gelu_erf")


def _rand(T, h, f, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return {"X": rng.standard_normal((T, h)), "A": rng.standard_normal((h, f)) * 0.5 * scale,
            "a": rng.standard_normal(f) * 0.3, "B": rng.standard_normal((f, h)) * 0.5,
            "b": rng.standard_normal(h) * 0.3, "dY": rng.standard_normal((T, h))}


# ---- worked example printed on the page (ReLU, one token, two shards) ------------------

def test_worked_example_one_token_two_shards():
    g = load("relu_mlp_one_token_two_shards.txt")
    X, A, B = g["X"][None, :], g["A"], g["B"]
    a, b = np.zeros(4), np.zeros(2)
    dY = g["dZ"][None, :]
    H, G, Y = oracle.forward(X, A, a, B, b, act="relu")
    np.testing.assert_array_equal(H[0], g["XA"])
    np.testing.assert_array_equal(Y[0], g["Z"])
    bw = oracle.backward(X, A, B, H, G, dY, act="relu")
    np.testing.assert_array_equal(bw["dX"][0], g["dX"])
    np.testing.assert_array_equal(bw["dA"], g["dA"])
    np.testing.assert_array_equal(bw["dB"], g["dB"])
    np.testing.assert_array_equal(bw["da"], g["da"])
    np.testing.assert_array_equal(bw["db"], g["db"])
    # shard by shard: the printed per-GPU intermediate values
    np.testing.assert_array_equal(G[0, :2], g["shard0_Y"])
    np.testing.assert_array_equal(G[0, 2:], g["shard1_Y"])
    np.testing.assert_array_equal(bw["dH"][0, :2], g["shard0_dH"])
    np.testing.assert_array_equal(bw["dH"][0, 2:], g["shard1_dH"])
    sh = oracle.sharded({"X": X, "A": A, "a": a, "B": B, "b": b, "dY": dY}, 2, act="relu",
                        parts=True)
    np.testing.assert_array_equal(sh["Y_part"][0, 0], g["shard0_partial"])
    np.testing.assert_array_equal(sh["Y_part"][1, 0], g["shard1_partial"])
    np.testing.assert_array_equal(sh["dX_part"][0, 0], g["shard0_dX"])
    np.testing.assert_array_equal(sh["dX_part"][1, 0], g["shard1_dX"])
    np.testing.assert_array_equal(sh["Y"][0], g["Z"])
    np.testing.assert_array_equal(sh["dX"][0], g["dX"])
    # dG_i = dZ B_i^T (printed); dH_i = dG_i * relu'(H_i)
    np.testing.assert_array_equal((dY @ B.T)[0, :2], g["shard0_dG"])
    np.testing.assert_array_equal((dY @ B.T)[0, 2:], g["shard1_dG"])


def test_row_split_is_wrong():
    """A nonlinearity of partial sums is not the nonlinearity of the sum: splitting A by
    rows and activating each partial product gives the page's wrong [1,2,2,2], while the
    block's activation is [1,2,1,0]."""
    g = load("relu_mlp_one_token_two_shards.txt")
    X, A, B = g["X"], g["A"], g["B"]
    parts = [oracle.forward(X[k:k + 1][None, :], A[k:k + 1], np.zeros(4), B[:, :1], np.zeros(1),
                            act="relu")[1][0] for k in range(2)]
    np.testing.assert_array_equal(parts[0] + parts[1], g["row_split_relu_sum"])
    _, G, _ = oracle.forward(X[None, :], A, np.zeros(4), B, np.zeros(2), act="relu")
    assert not np.array_equal(G[0], g["row_split_relu_sum"])
    np.testing.assert_array_equal(G[0], g["XA"])  # ReLU leaves [1,2,1,0] unchanged


@pytest.mark.parametrize("t", [1, 2, 4])
def test_four_tokens_four_shards(t):
    g = load("relu_mlp_four_tokens_four_shards.txt")
    inp = {"X": g["X"], "A": g["A"], "a": np.zeros(4), "B": g["B"], "b": np.zeros(2), "dY": g["dZ"]}
    out = oracle.fwd_bwd(inp, act="relu")
    for k in ("H", "G", "dH", "dX", "dA", "dB", "da", "db"):
        np.testing.assert_array_equal(out[k], g[k], err_msg=k)
    np.testing.assert_array_equal(out["Y"], g["Z"])
    sh = oracle.sharded(inp, t, act="relu")
    for k in ("dX", "dA", "dB", "da", "db"):
        np.testing.assert_array_equal(sh[k], g[k], err_msg=k)
    np.testing.assert_array_equal(sh["Y"], g["Z"])
    # "split the tokens": each token's output depends on that token only
    for r in range(4):
        one = {k: (v[r:r + 1] if k in ("X", "dY") else v) for k, v in inp.items()}
        o1 = oracle.fwd_bwd(one, act="relu")
        np.testing.assert_array_equal(o1["Y"][0], g["Z"][r])
        np.testing.assert_array_equal(o1["dX"][0], g["dX"][r])


# ---- GELU: closed forms, the exact form against the library erf -------------------------

def test_gelu_closed_forms():
    xs = np.linspace(-6, 6, 241)
    for kind in ACTS:
        assert oracle.act([0.0], kind)[0] == 0.0
        assert abs(oracle.act_grad([0.0], kind)[0] - 0.5) < 1e-15
        g, gm = oracle.act(xs, kind), oracle.act(-xs, kind)
        np.testing.assert_allclose(g - gm, xs, atol=1e-13)  # gelu(x) - gelu(-x) = x
        big = np.array([20.0, 40.0])
        np.testing.assert_allclose(oracle.act(big, kind), big, rtol=1e-15)
        np.testing.assert_allclose(oracle.act(-big, kind), 0.0, atol=1e-30)
        np.testing.assert_allclose(oracle.act_grad(big, kind), 1.0, rtol=1e-15)
        np.testing.assert_allclose(oracle.act_grad(-big, kind), 0.0, atol=1e-30)


def test_gelu_erf_form_matches_library_erf():
    xs = np.linspace(-7, 7, 561)
    ref = np.array([0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))) for x in xs])
    np.testing.assert_allclose(oracle.act(xs, "gelu_erf"), ref, rtol=1e-14, atol=1e-300)


def test_gelu_tanh_form_close_to_exact_form():
    """The tanh form approximates x*Phi(x) within 5e-4 everywhere (the largest gap is
    about 4.7e-4 near |x| = 2.2); a wrong constant or a dropped cubic term breaks this."""
    xs = np.linspace(-8, 8, 3201)
    d = np.abs(oracle.act(xs, "gelu_tanh") - oracle.act(xs, "gelu_erf"))
    assert d.max() < 5e-4
    assert d.max() > 1e-4  # and it is the tanh form, not the exact one


@pytest.mark.parametrize("kind", ACTS)
def test_gelu_grad_matches_finite_difference(kind):
    xs = np.linspace(-5, 5, 201)
    eps = 1e-6
    fd = (oracle.act(xs + eps, kind) - oracle.act(xs - eps, kind)) / (2 * eps)
    np.testing.assert_allclose(oracle.act_grad(xs, kind), fd, atol=1e-8)


# ---- library special case: identity activation reduces the block to plain matmuls ------

def test_identity_activation_is_plain_matmuls():
    inp = _rand(5, 6, 12, seed=1)
    X, A, a, B, b, dY = (inp[k] for k in ("X", "A", "a", "B", "b", "dY"))
    out = oracle.fwd_bwd(inp, act="identity")
    H = X @ A + a
    np.testing.assert_allclose(out["Y"], H @ B + b, rtol=1e-12, atol=1e-12)
    dH = dY @ B.T
    np.testing.assert_allclose(out["dX"], dH @ A.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dA"], X.T @ dH, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dB"], H.T @ dY, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["da"], dH.sum(0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["db"], dY.sum(0), rtol=1e-12, atol=1e-12)


def test_torch_autograd_agrees_for_exact_gelu():
    """Library cross-check: torch's exact-GELU MLP and its autograd (fp64, CPU)."""
    inp = _rand(4, 6, 16, seed=2)
    tt = {k: torch.tensor(v, requires_grad=k != "dY") for k, v in inp.items()}
    Y = torch.nn.functional.gelu(tt["X"] @ tt["A"] + tt["a"]) @ tt["B"] + tt["b"]
    (Y * tt["dY"]).sum().backward()
    out = oracle.fwd_bwd(inp, act="gelu_erf")
    np.testing.assert_allclose(out["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    for k, g in (("dX", "X"), ("dA", "A"), ("da", "a"), ("dB", "B"), ("db", "b")):
        np.testing.assert_allclose(out[k], tt[g].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=k)


def test_torch_autograd_agrees_for_tanh_gelu():
    inp = _rand(4, 6, 16, seed=3)
    tt = {k: torch.tensor(v, requires_grad=k != "dY") for k, v in inp.items()}
    Y = torch.nn.functional.gelu(tt["X"] @ tt["A"] + tt["a"], approximate="tanh") @ tt["B"] + tt["b"]
    (Y * tt["dY"]).sum().backward()
    out = oracle.fwd_bwd(inp, act="gelu_tanh")
    np.testing.assert_allclose(out["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    for k, g in (("dX", "X"), ("dA", "A"), ("da", "a"), ("dB", "B"), ("db", "b")):
        np.testing.assert_allclose(out[k], tt[g].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=k)


# ---- invariants ------------------------------------------------------------------------

@pytest.mark.parametrize("act", ACTS + ("relu",))
def test_shard_sum_invariant_every_t(act):
    """GELU(XA)B = sum_i GELU(XA_i)B_i, and dX = sum_i dH_i A_i^T, for every t | f."""
    inp = _rand(6, 8, 16, seed=4)
    full = oracle.fwd_bwd(inp, act=act)
    for t in (1, 2, 4, 8, 16):
        sh = oracle.sharded(inp, t, act=act, parts=True)
        for k in ("Y", "dX", "dA", "da", "dB", "db"):
            np.testing.assert_allclose(sh[k], full[k], rtol=1e-12, atol=1e-12, err_msg=f"{k} t={t}")
        # the backward of a copy is a sum: dX is the sum of the shard dX's
        np.testing.assert_allclose(sh["dX_part"].sum(0), full["dX"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sh["Y_part"].sum(0) + inp["b"], full["Y"], rtol=1e-12, atol=1e-12)


def test_sharded_rejects_uneven_split():
    inp = _rand(2, 4, 12, seed=5)
    with pytest.raises(ValueError):
        oracle.sharded(inp, 5)


def test_db_is_colsum_of_dy_independent_of_weights():
    inp = _rand(7, 4, 8, seed=6)
    db0 = oracle.fwd_bwd(inp)["db"]
    inp2 = dict(inp, A=inp["A"] * -3.0, B=inp["B"] + 1.0, a=inp["a"] * 0)
    db1 = oracle.fwd_bwd(inp2)["db"]
    np.testing.assert_array_equal(db0, db1)
    np.testing.assert_allclose(db0, inp["dY"].sum(0), rtol=1e-14)


def test_empty_token_batch():
    inp = _rand(0, 4, 8, seed=7)
    out = oracle.fwd_bwd(inp)
    assert out["Y"].shape == (0, 4)
    np.testing.assert_array_equal(out["dA"], 0.0)
    np.testing.assert_array_equal(out["db"], 0.0)


# ---- finite differences ----------------------------------------------------------------

@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("t", [1, 2])
def test_central_finite_differences(act, t):
    """L = <dY, Y>; every entry of dX, dA, da, dB, db against a central difference."""
    T, h, f = 3, 4, 8
    inp = _rand(T, h, f, seed=10 + t)
    grads = oracle.sharded(inp, t, act=act)

    def loss(d):
        _, _, Y = oracle.forward(d["X"], d["A"], d["a"], d["B"], d["b"], act)
        return float((Y * d["dY"]).sum())

    for name, gname in (("X", "dX"), ("A", "dA"), ("a", "da"), ("B", "dB"), ("b", "db")):
        base = inp[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            hi = dict(inp); hi[name] = base.copy(); hi[name][idx] += eps
            lo = dict(inp); lo[name] = base.copy(); lo[name][idx] -= eps
            fd[idx] = (loss(hi) - loss(lo)) / (2 * eps)
        np.testing.assert_allclose(grads[gname], fd, rtol=1e-6, atol=1e-7, err_msg=gname)


# ---- the sampled-entry oracle equals the full one on the entries it picks --------------

def test_sampled_matches_full_on_bf16_inputs():
    inp = make_inputs(40, 24, 64, seed=3, sdy=1.0, sw=0.2)
    full = oracle.fwd_bwd(inp)
    rows = np.array([0, 7, 39])
    cols = np.array([0, 15, 16, 31, 63])
    s = oracle.sampled_bf16(inp, rows, cols)
    np.testing.assert_allclose(s["Y_rows"], full["Y"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dX_rows"], full["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dA_cols"], full["dA"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dB_rows"], full["dB"][cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["da"], full["da"][cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["db"], full["db"], rtol=1e-12, atol=1e-12)


# ---- the shared input generator --------------------------------------------------------

def test_input_generator_is_seeded_and_bf16():
    w = WORKLOADS["tiny"]
    a = make_inputs(w.T, w.h, w.f, seed=0, sdy=w.sdy)
    b = make_inputs(w.T, w.h, w.f, seed=0, sdy=w.sdy)
    c = make_inputs(w.T, w.h, w.f, seed=1, sdy=w.sdy)
    for k in a:
        assert a[k].dtype == torch.bfloat16
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["X"], c["X"])
    assert abs(float(a["A"].float().std()) - 0.02) < 0.002
    part = make_inputs(w.T, w.h, w.f, seed=0, sdy=w.sdy, rows=5)
    assert torch.equal(part["X"], a["X"][:5]) and torch.equal(part["A"], a["A"])
