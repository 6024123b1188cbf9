"""The device GELU and GELU' over every finite bf16 input, against the oracle's tanh-form GELU
("Efficient Large-Scale Language Model Training on GPU Clusters Using Megatron-LM", §3,
fused bias + GeLU; the MLP block's Y = GELU(XA)B).

The inputs make each epilogue evaluate its activation on all 65,280 finite bf16 values at
once, with nothing else in the way:
- forward: X has a single 1 per row (column 0) and A's row 0 holds the values, a = 0, so
  H = X A + a is exactly that row and G = GELU(H) comes straight from the bias + GELU
  epilogue;
- backward: dY and B each have a single 1 per row (column 0), so dG = dY B^T is exactly 1 and
  dH = dG GELU'(H) is the dH epilogue's GELU' of the saved H, rounded to bf16.

Bar, per value: the bf16 result lies between the bf16 roundings of ref - eps and ref + eps,
eps = 4e-5 |ref| + oracle_err(x) + 1e-30:
- 4e-5 |ref| is the fp32 evaluation's error: ex2.approx and the rounded coefficients give
  e = exp(-2u) a relative error up to ~2.5e-5 where z is near its largest (x near -9.75);
- oracle_err bounds the fp64 oracle's own error. It evaluates the definition as written, and
  1 + tanh u and 1 - tanh^2 u cancel for u << 0: an absolute error of a few 2^-53, times
  |x| and |u'(x)|, for |x| <= 10 (beyond, tanh u is exactly +-1 in fp64 and the exact values
  are below 1e-80);
- 1e-30: the values below -9.75 evaluate at -9.75, under 3.1e-35 in magnitude.
And at most 0.5% of the values whose bound (oracle_err + 1e-30) is under a thousandth of
the reference's magnitude may differ from the bf16 rounding of that reference at all (a difference needs the fp32 result
within eps of a rounding boundary)."""
import numpy as np
import pytest
import torch

import oracle
from megatron_tensor_transformer_tcgen05_gb300 import _lib, block
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod

pytestmark = pytest.mark.gpu

T, h, f, t = 128, 64, 65536, 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


def _every_bf16() -> torch.Tensor:
    """All 65,536 bf16 bit patterns in order, with the non-finite ones replaced by 0."""
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).copy()
    vals[((bits >> 7) & 0xFF) == 0xFF] = 0.0
    return torch.from_numpy(vals).to(torch.bfloat16)  # exact: the low 16 bits are zero


def _rne_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


def _oracle_err(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    du = 0.7978845608028654 * (1.0 + 3.0 * 0.044715 * np.minimum(ax, 10.0) ** 2)
    return np.where(ax <= 10.0, 2.0 ** -50 * (1.0 + ax) * (1.0 + du), 0.0)


def _check(name: str, got: torch.Tensor, x: np.ndarray, ref: np.ndarray) -> None:
    g = got.to("cpu", torch.float64).numpy()
    assert np.all(np.isfinite(g)), f"{name}: non-finite results"
    oerr = _oracle_err(x)
    eps = 4e-5 * np.abs(ref) + oerr + 1e-30
    lo, hi = _rne_bf16(ref - eps), _rne_bf16(ref + eps)
    bad = np.nonzero((g < lo) | (g > hi))[0]
    assert bad.size == 0, (f"{name}: {bad.size} values outside the bar, first at x = {x[bad[0]]:.6e}: "
                           f"got {g[bad[0]]:.9e}, oracle {ref[bad[0]]:.9e}")
    good = oerr + 1e-30 <= 1e-3 * np.abs(ref)
    off = np.count_nonzero((g != _rne_bf16(ref)) & good)
    assert off <= 0.005 * np.count_nonzero(good), f"{name}: {off} values differ from the rounded oracle value"


def _inputs(x: torch.Tensor) -> dict:
    bf = torch.bfloat16
    X = torch.zeros((T, h), dtype=bf)
    X[:, 0] = 1
    A = torch.zeros((h, f), dtype=bf)
    A[0] = x
    B = torch.zeros((f, h), dtype=bf)
    B[:, 0] = 1
    dY = torch.zeros((T, h), dtype=bf)
    dY[:, 0] = 1
    return {"X": X, "A": A, "a": torch.zeros(f, dtype=bf), "B": B, "b": torch.zeros(h, dtype=bf), "dY": dY}


def test_gelu_of_the_forward_epilogue_over_every_bf16():
    x = _every_bf16()
    dev = {k: v.cuda() for k, v in _inputs(x).items()}
    buf = block.empty_buffers(T, h, f, t)
    block.forward(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    H = buf["H"].cpu()
    # H is X A + a, one product per entry; the tensor core may flush subnormal operands,
    # so the reference is taken at the H the kernel produced (the same in every row)
    assert torch.equal(H, H[:1].expand(T, f)), "H rows differ"
    normal = (x.float().abs() >= 2.0 ** -126) | (x.float() == 0)
    assert torch.equal(H[0][normal], x[normal]), "H differs from the exact X A + a"
    G = buf["G"].cpu()
    assert torch.equal(G, G[:1].expand(T, f)), "G rows differ"
    h0 = H[0].double().numpy()
    _check("GELU", G[0], h0, oracle.act(h0))


def test_gelu_grad_of_the_dh_epilogue_over_every_bf16():
    x = _every_bf16()
    dev = {k: v.cuda() for k, v in _inputs(x).items()}
    buf = block.empty_buffers(T, h, f, t)
    buf["H"].copy_(x.cuda().expand(T, f))
    buf["G"].zero_()
    block.backward(dev, buf, t)
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    ws = buf["ws"]
    dH = ws[: T * f * 2].view(torch.bfloat16).view(T, f).cpu()  # dH = dG GELU'(H), dG = 1
    assert torch.equal(dH, dH[:1].expand(T, f)), "dH rows differ"
    xs = x.double().numpy()
    ref = oracle.act_grad(xs)
    _check("GELU'", dH[0], xs, ref)
    # da sums the fp32 dH of the 128 equal rows (before its bf16 rounding): 128 times the
    # fp32 GELU', exactly, as sums of equal values in pairs are exact
    da = buf["da"].cpu().double().numpy() / 128.0
    bad = np.nonzero(np.abs(da - ref) > 4e-5 * np.abs(ref) + _oracle_err(xs) + 1e-30)[0]
    assert bad.size == 0, f"da: {bad.size} columns off, first {bad[0]}: {da[bad[0]]:.9e} vs {ref[bad[0]]:.9e}"
