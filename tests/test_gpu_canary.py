"""Out-of-bounds write detection with guard bands, in place of a memory sanitizer.

Every output and workspace of a call is the middle of a larger device allocation: the
exact-size region the call may write, with GUARD bytes of a known pattern right before and
right after it. After the call (and a device status check) both bands must still hold the
pattern, and every input must be bit-for-bit unchanged. The shapes reach every hand-written
store of the library on ragged sizes and every branch of the GEMM launch planner: the split
tails' fp32 parts and their fixup (splitk_fixup_kernel), the dH epilogue's per-32-row column
sums (in the workspace) and the column-sum kernels (da, db), the attention block's L and D
(D in the workspace), the dropout backward, the SwiGLU epilogues, the GELU recompute's
forward and backward, and the allocation-free bias-gradient entry point. A one-element overrun past the
end of any output, or a write before its start, changes a guard byte and fails the test."""
import numpy as np
import pytest
import torch

from sweep_shapes import attn_sweep_shapes, mlp_sweep_shapes
from megatron_tensor_transformer_tcgen05_gb300 import _lib
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import make_attn_inputs, make_inputs, make_swiglu_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes on each side; keeps the region 256-byte aligned
PAT = 0xA5     # guard byte
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    _lib.lib()


class Guarded:
    """A device region of exactly nbytes (shape x dtype, or raw bytes), with GUARD bytes of
    PAT before and after it in the same allocation. The region itself starts filled with
    PAT too, so a call that leaves part of an output unwritten is caught by the parity
    tests, not hidden here."""

    def __init__(self, name, shape, dtype=torch.uint8):
        self.name = name
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape)) * itemsize
        self.raw = torch.full((GUARD + self.n + GUARD,), PAT, dtype=torch.uint8, device="cuda")
        assert self.raw.data_ptr() % 256 == 0
        self.t = self.raw[GUARD:GUARD + self.n].view(dtype).view(*shape)

    def check(self):
        for where, band in (("before", self.raw[:GUARD]), ("after", self.raw[GUARD + self.n:])):
            bad = torch.nonzero(band != PAT)
            assert bad.numel() == 0, (f"{self.name}: {bad.numel()} guard bytes {where} the {self.n}-byte region "
                                      f"overwritten, first at offset {int(bad[0])}")


def _guarded(spec: dict) -> dict:
    return {k: Guarded(k, *v) for k, v in spec.items()}


def _run_and_check(outs: dict, inputs: dict, fn):
    before = {k: v.clone() for k, v in inputs.items()}
    fn()
    torch.cuda.synchronize()
    assert _lib.mlp_tp_query_device_status() == 0, _lib.mlp_tp_last_device_where()
    for g in outs.values():
        g.check()
    for k, v in inputs.items():
        assert torch.equal(v, before[k]), f"input {k} was written"


# split tails in the forward and backward GEMMs (one CTA per tile, CTA pairs, clusters of two
# pairs, the bias + GELU and GELU' epilogues), as in the split-tail parity tests
SPLIT_SHAPES = [(128, 1024, 8192, 4), (512, 1024, 4096, 2), (2048, 256, 1024, 2), (512, 2048, 2048, 2),
                (512, 4096, 2048, 2)]
MLP_SHAPES = mlp_sweep_shapes() + SPLIT_SHAPES


def _mlp_outs(T, h, f, t, recompute=False):
    bf, f32 = torch.bfloat16, torch.float32
    ws = (_lib.mlp_tp_recompute_workspace_bytes if recompute else _lib.mlp_tp_workspace_bytes)(T, h, f, t)
    return _guarded({"H": ((T, f), bf), "G": ((T, f), bf), "Y": ((T, h), bf), "dX": ((T, h), bf),
                     "dA": ((h, f), bf), "dB": ((f, h), bf), "da": ((f,), f32), "db": ((h,), f32),
                     "ws": ((ws,),), "fws": ((_lib.mlp_tp_forward_workspace_bytes(),),)})


@pytest.mark.parametrize("T,h,f,t", MLP_SHAPES, ids=[f"T{T}-h{h}-f{f}-t{t}" for T, h, f, t in MLP_SHAPES])
def test_mlp_forward_backward_stay_in_bounds(T, h, f, t):
    inp = {k: v.cuda() for k, v in make_inputs(T, h, f, seed=T + f, sdy=1.0).items()}
    o = _mlp_outs(T, h, f, t)
    g = {k: v.t for k, v in o.items()}

    def call():
        _lib.mlp_tp_forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], T, h, f, t, g["H"], g["G"], g["Y"],
                            g["fws"], g["fws"].numel())
        _lib.mlp_tp_backward(inp["X"], inp["A"], inp["B"], g["H"], g["G"], inp["dY"], T, h, f, t, g["dX"], g["dA"],
                             g["dB"], g["da"], g["db"], g["ws"], g["ws"].numel())

    _run_and_check(o, inp, call)
    # the allocation-free bias gradients, from the dH the backward left in its workspace
    nb = _guarded({"da2": ((f,), torch.float32), "db2": ((h,), torch.float32)})
    dH = g["ws"][: T * f * 2].view(torch.bfloat16).view(T, f)
    _run_and_check(nb, {"dH": dH, "dY": inp["dY"]},
                   lambda: _lib.mlp_tp_bias_grads_noalloc(dH, inp["dY"], T, h, f, nb["da2"].t, nb["db2"].t))


@pytest.mark.parametrize("T,h,f,t", MLP_SHAPES[::3], ids=[f"T{T}-h{h}-f{f}-t{t}" for T, h, f, t in MLP_SHAPES[::3]])
def test_recompute_forward_backward_stay_in_bounds(T, h, f, t):
    """The GELU recompute: H-only forward and the backward from H (A operands transformed on chip)."""
    inp = {k: v.cuda() for k, v in make_inputs(T, h, f, seed=T + h, sdy=1.0).items()}
    o = _mlp_outs(T, h, f, t, recompute=True)
    del o["G"]
    g = {k: v.t for k, v in o.items()}
    _run_and_check(o, inp, lambda: _lib.mlp_tp_forward_recompute(
        inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], T, h, f, t, g["H"], g["Y"], g["fws"], g["fws"].numel()))
    H = g["H"].clone()
    _run_and_check(o, dict(inp, H=H), lambda: _lib.mlp_tp_backward_recompute(
        inp["X"], inp["A"], inp["B"], H, inp["dY"], T, h, f, t, g["dX"], g["dA"], g["dB"], g["da"], g["db"], g["ws"],
        g["ws"].numel()))


@pytest.mark.parametrize("T,h,f,t", [(300, 136, 512, 2), (1000, 2048, 4096, 4), (4096 - 40, 1024, 2048, 2)])
def test_dropout_output_step_stays_in_bounds(T, h, f, t):
    inp = {k: v.cuda() for k, v in make_inputs(T, h, f, seed=3, sdy=1.0).items()}
    R = torch.randn((T, h), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    bf = torch.bfloat16
    o = _guarded({"H": ((T, f), bf), "G": ((T, f), bf), "Z": ((T, h), bf), "dY": ((T, h), bf)})
    _run_and_check(o, dict(inp, R=R), lambda: (
        _lib.mlp_tp_forward_residual_dropout(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], R, T, h, f, t, 0.1,
                                             77, 5, o["H"].t, o["G"].t, o["Z"].t),
        _lib.mlp_tp_dropout_backward(inp["dY"], T, h, 0.1, 77, 5, o["dY"].t)))


@pytest.mark.parametrize("T,h,f,t", [(300, 136, 512, 2), (1000, 1024, 2048, 2), (600, 2048, 4096, 4)])
def test_swiglu_stays_in_bounds(T, h, f, t):
    inp = {k: v.cuda() for k, v in make_swiglu_inputs(T, h, f, seed=5).items()}
    bf = torch.bfloat16
    ws = _lib.mlp_tp_swiglu_workspace_bytes(T, h, f, t)
    o = _guarded({"Ha": ((T, f), bf), "Hg": ((T, f), bf), "U": ((T, f), bf), "Y": ((T, h), bf),
                  "dX": ((T, h), bf), "dA": ((h, f), bf), "dWg": ((h, f), bf), "dB": ((f, h), bf), "ws": ((ws,),),
                  "fws": ((_lib.mlp_tp_forward_workspace_bytes(),),)})
    g = {k: v.t for k, v in o.items()}
    _run_and_check(o, inp, lambda: (
        _lib.mlp_tp_swiglu_forward(inp["X"], inp["A"], inp["Wg"], inp["B"], T, h, f, t, g["Ha"], g["Hg"], g["U"],
                                   g["Y"], g["fws"], g["fws"].numel()),
        _lib.mlp_tp_swiglu_backward(inp["X"], inp["A"], inp["Wg"], inp["B"], g["Ha"], g["Hg"], g["U"], inp["dY"], T,
                                    h, f, t, g["dX"], g["dA"], g["dWg"], g["dB"], g["ws"], g["ws"].numel())))


ATTN_SHAPES = attn_sweep_shapes() + [(1, 1024, 2048, 16, 2, True)]


@pytest.mark.parametrize("b,s,h,a,t,causal", ATTN_SHAPES,
                         ids=[f"b{b}-s{s}-h{h}-a{a}-t{t}-{'causal' if c else 'full'}" for b, s, h, a, t, c in ATTN_SHAPES])
def test_attention_stays_in_bounds(b, s, h, a, t, causal):
    inp = make_attn_inputs(b, s, h, a, D, seed=s + a, sw=1.2 / np.sqrt(h), sdy=1.0)
    dev = {k: inp[k].cuda() for k in ("X", "Wqkv", "Wo", "dY")}
    T, hd = b * s, a * D
    bf = torch.bfloat16
    ws = _lib.mlp_tp_attn_workspace_bytes(b, s, h, a, D, t)
    o = _guarded({"QKV": ((T, 3 * hd), bf), "C": ((T, hd), bf), "L": ((b * a, s), torch.float32),
                  "Y": ((T, h), bf), "dX": ((T, h), bf), "dWqkv": ((h, 3 * hd), bf), "dWo": ((hd, h), bf),
                  "ws": ((ws,),), "fws": ((_lib.mlp_tp_forward_workspace_bytes(),),)})
    g = {k: v.t for k, v in o.items()}
    _run_and_check(o, dev, lambda: (
        _lib.mlp_tp_attn_forward(dev["X"], dev["Wqkv"], dev["Wo"], b, s, h, a, D, t, causal, g["QKV"], g["C"],
                                 g["L"], g["Y"], g["fws"], g["fws"].numel()),
        _lib.mlp_tp_attn_backward(dev["X"], dev["Wqkv"], dev["Wo"], g["QKV"], g["C"], g["L"], dev["dY"], b, s, h, a,
                                  D, t, causal, g["dX"], g["dWqkv"], g["dWo"], g["ws"], g["ws"].numel())))


def test_guard_check_catches_a_one_element_overrun():
    """The check itself: a copy one element longer than an output region trips the band."""
    o = Guarded("probe", (64,), torch.bfloat16)
    src = torch.ones(65, dtype=torch.bfloat16, device="cuda")
    o.raw[GUARD:GUARD + 130].copy_(src.view(torch.uint8))  # 65 elements into a 64-element region
    with pytest.raises(AssertionError, match="after"):
        o.check()
