"""Pins for the oracle's head-parallel attention block: torch autograd (a library routine),
finite differences, the head-shard-sum invariant, and the causal mask."""
import numpy as np
import pytest
import torch

import oracle


def _rand(b, s, h, a, d, seed):
    rng = np.random.default_rng(seed)
    hd = a * d
    return {"X": rng.standard_normal((b * s, h)), "Wq": rng.standard_normal((h, hd)) * 0.4,
            "Wk": rng.standard_normal((h, hd)) * 0.4, "Wv": rng.standard_normal((h, hd)) * 0.4,
            "Wo": rng.standard_normal((hd, h)) * 0.4, "dY": rng.standard_normal((b * s, h))}


@pytest.mark.parametrize("causal", [True, False])
def test_attention_matches_torch_autograd(causal):
    b, s, h, a, d = 2, 5, 6, 3, 4
    inp = _rand(b, s, h, a, d, seed=1)
    tt = {k: torch.tensor(v, requires_grad=k != "dY") for k, v in inp.items()}
    x = tt["X"].view(b, s, h)
    q = (x @ tt["Wq"]).view(b, s, a, d).transpose(1, 2)
    k = (x @ tt["Wk"]).view(b, s, a, d).transpose(1, 2)
    v = (x @ tt["Wv"]).view(b, s, a, d).transpose(1, 2)
    c = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    Y = c.transpose(1, 2).reshape(b * s, a * d) @ tt["Wo"]
    (Y * tt["dY"]).sum().backward()
    out = oracle.attn_fwd_bwd(inp, b, s, a, causal)
    np.testing.assert_allclose(out["Y"], Y.detach().numpy(), rtol=1e-11, atol=1e-12)
    for key, g in (("dX", "X"), ("dWq", "Wq"), ("dWk", "Wk"), ("dWv", "Wv"), ("dWo", "Wo")):
        np.testing.assert_allclose(out[key], tt[g].grad.numpy(), rtol=1e-10, atol=1e-11, err_msg=key)


def test_causal_mask_and_softmax_rows():
    b, s, h, a, d = 1, 6, 4, 2, 2
    out = oracle.attn_fwd_bwd(_rand(b, s, h, a, d, seed=2), b, s, a, causal=True)
    P = out["P"]
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=1e-14)
    assert np.all(np.triu(P[0, 0], 1) == 0.0)  # no query attends to a later key
    np.testing.assert_allclose(P[0, :, 0, 0], 1.0)  # the first token sees only itself


def test_attention_finite_differences():
    b, s, h, a, d = 1, 4, 3, 2, 2
    inp = _rand(b, s, h, a, d, seed=3)
    out = oracle.attn_fwd_bwd(inp, b, s, a, causal=True)

    def loss(dd):
        return float((oracle.attn_fwd_bwd(dd, b, s, a, causal=True)["Y"] * dd["dY"]).sum())

    for name, gname in (("X", "dX"), ("Wq", "dWq"), ("Wk", "dWk"), ("Wv", "dWv"), ("Wo", "dWo")):
        base = inp[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            hi = dict(inp); hi[name] = base.copy(); hi[name][idx] += eps
            lo = dict(inp); lo[name] = base.copy(); lo[name][idx] -= eps
            fd[idx] = (loss(hi) - loss(lo)) / (2 * eps)
        np.testing.assert_allclose(out[gname], fd, rtol=1e-6, atol=1e-7, err_msg=gname)


def test_head_shard_sum_invariant():
    """Heads split over t shards: Y = sum_i C_i Wo_i and dX = sum_i dX_i, for every t | a."""
    b, s, h, a, d = 2, 5, 6, 4, 3
    inp = _rand(b, s, h, a, d, seed=4)
    full = oracle.attn_fwd_bwd(inp, b, s, a)
    for t in (1, 2, 4):
        sh = oracle.attn_sharded(inp, b, s, a, t, parts=True)
        for k in ("Y", "dX", "dWq", "dWk", "dWv", "dWo"):
            np.testing.assert_allclose(sh[k], full[k], rtol=1e-12, atol=1e-12, err_msg=f"{k} t={t}")
        np.testing.assert_allclose(sh["Y_part"].sum(0), full["Y"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sh["dX_part"].sum(0), full["dX"], rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.attn_sharded(inp, b, s, a, 3)


def test_uniform_scores_closed_form():
    """Wq = 0 makes every score 0: causal softmax is then uniform over the keys j <= i, so
    C_i is the running mean of V over the sequence (non-causal: the mean of all of V), and
    Y = C Wo. With one token the block reduces to X Wv Wo."""
    b, s, h, a, d = 2, 7, 5, 2, 3
    inp = _rand(b, s, h, a, d, seed=5)
    inp["Wq"] = np.zeros_like(inp["Wq"])
    V = inp["X"] @ inp["Wv"]
    for causal in (True, False):
        out = oracle.attn_fwd_bwd(inp, b, s, a, causal)
        Vb = V.reshape(b, s, a * d)
        if causal:
            C = np.cumsum(Vb, axis=1) / np.arange(1, s + 1)[None, :, None]
        else:
            C = np.broadcast_to(Vb.mean(axis=1, keepdims=True), Vb.shape)
        np.testing.assert_allclose(out["C"], C.reshape(b * s, a * d), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(out["Y"], out["C"] @ inp["Wo"], rtol=1e-13, atol=1e-13)
        assert np.all(np.isfinite(out["dWq"]))
    one = _rand(3, 1, h, a, d, seed=6)
    out = oracle.attn_fwd_bwd(one, 3, 1, a)
    np.testing.assert_allclose(out["Y"], one["X"] @ one["Wv"] @ one["Wo"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["dWq"], 0.0, atol=1e-15)  # a lone score has zero softmax gradient
    np.testing.assert_allclose(out["dWk"], 0.0, atol=1e-15)


def test_lse_reproduces_the_probabilities():
    """L is the base-2 log-sum-exp of the scaled scores: 2^(S log2 e - L) gives back P."""
    b, s, h, a, d = 2, 6, 5, 2, 3
    inp = _rand(b, s, h, a, d, seed=7)
    out = oracle.attn_fwd_bwd(inp, b, s, a, causal=True)
    for bi in range(b):
        for hh in range(a):
            rows = slice(bi * s, (bi + 1) * s)
            cols = slice(hh * d, (hh + 1) * d)
            S = out["Q"][rows, cols] @ out["K"][rows, cols].T / np.sqrt(d)
            P = np.where(np.tril(np.ones((s, s))) > 0, np.exp2(S * np.log2(np.e) - out["L"][bi * a + hh][:, None]), 0)
            np.testing.assert_allclose(P, out["P"][bi, hh], rtol=1e-12, atol=1e-15)


def test_sampled_bf16_matches_the_full_oracle():
    """The sampled C and L agree with the full forward on bf16-representable inputs."""
    import torch
    from megatron_tensor_transformer_tcgen05_gb300.inputs import make_attn_inputs
    b, s, h, a, d = 2, 9, 16, 2, 4
    inp = make_attn_inputs(b, s, h, a, d, seed=3, sw=0.3)
    full = oracle.attn_fwd_bwd({k: v.double().numpy() for k, v in inp.items()}, b, s, a, causal=True)
    rows, heads = np.array([0, 4, 8, 9, 17]), np.array([1, 0])
    smp = oracle.attn_sampled_bf16(inp, b, s, a, rows, heads, causal=True)
    for ri, r in enumerate(rows):
        for hi, hh in enumerate(heads):
            np.testing.assert_allclose(smp["C"][ri, hi], full["C"][r, hh * d:(hh + 1) * d], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(smp["L"][ri, hi], full["L"][(r // s) * a + hh, r % s], rtol=1e-13)
    assert torch.is_tensor(inp["X"])
