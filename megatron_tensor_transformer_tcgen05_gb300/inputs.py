"""Seeded synthetic inputs and the workload table for the tensor-parallel MLP block.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's tests.
It holds no arithmetic of the block itself: it only draws normal random numbers,
scales them by a standard deviation and rounds them to bf16.

Recipe (per workload, one ``torch.Generator('cpu')`` seeded with ``seed``):
draw, in this order, X [T,h], A [h,f], a [f], B [f,h], b [h], dY [T,h] as
``torch.randn(..., dtype=float32) * sigma`` and round to bf16 (round to nearest even).
sigma is a standard deviation. The workloads are the GPT layer shapes of
"Efficient Large-Scale Language Model Training on GPU Clusters Using Megatron-LM",
§5 (Table 1 models, s = 2048 synthetic batches, MLP width f = 4h from §3 Fig 5a),
with micro-batches b chosen so that T = b*s tokens.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens (micro-batch x sequence length)
    h: int          # hidden width
    f: int          # MLP width (4h)
    t: int          # tensor-parallel shard count
    sx: float = 1.0     # std of X
    sw: float = 0.02    # std of A and B
    sbias: float = 0.01  # std of a and b
    sdy: float = 0.01   # std of dY
    desc: str = ""
    kind: str = "gelu"   # "gelu": Y = GELU(X A + a) B + b;  "swiglu": Y = (SiLU(X A) * X Wg) B

    @property
    def flops_fwd_bwd(self) -> int:
        """Matmul FLOPs of one forward + backward: 6 GEMMs of 2*T*h*f each (GELU block), or
        9 (SwiGLU block: X A, X Wg, U B; dU, dX over two K segments, dA, dWg, dB)."""
        return (18 if self.kind == "swiglu" else 12) * self.T * self.h * self.f


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    Workload("tiny", 128, 64, 256, 2, sdy=1.0,
             desc="tiny TP MLP block T=128 h=64 f=256 t=2"),
    Workload("gpt-1.7b-t1", 16384, 2304, 9216, 1,
             desc="GPT 1.7B-shaped layer T=16384 (8x2048) h=2304 f=9216 t=1"),
    Workload("gpt-1.7b-t2", 16384, 2304, 9216, 2,
             desc="GPT 1.7B-shaped layer T=16384 (8x2048) h=2304 f=9216 t=2"),
    Workload("gpt-18b", 8192, 6144, 24576, 8,
             desc="GPT 18B-shaped layer T=8192 (4x2048) h=6144 f=24576 t=8"),
    Workload("gpt3-175b", 4096, 12288, 49152, 8,
             desc="GPT-3 175B-shaped layer T=4096 (2x2048) h=12288 f=49152 t=8"),
    Workload("gpt-1t", 2048, 25600, 102400, 8, sw=0.006,
             desc="1T-shaped layer T=2048 (1x2048) h=25600 f=102400 t=8"),
    # SwiGLU variant at the GPT-3 175B layer shape, f = 8h/3 so that its three weight
    # matrices hold as many parameters as the GELU block's two.
    Workload("gpt3-175b-swiglu", 4096, 12288, 32768, 8, kind="swiglu",
             desc="SwiGLU MLP at the GPT-3 175B layer shape T=4096 h=12288 f=32768 (8h/3) t=8"),
]}

NAMES = ("X", "A", "a", "B", "b", "dY")


def shapes(T: int, h: int, f: int) -> dict[str, tuple[int, ...]]:
    return {"X": (T, h), "A": (h, f), "a": (f,), "B": (f, h), "b": (h,), "dY": (T, h)}


def make_inputs(T: int, h: int, f: int, *, seed: int = 0, sx: float = 1.0,
                sw: float = 0.02, sbias: float = 0.01, sdy: float = 0.01,
                rows: int | None = None) -> dict[str, torch.Tensor]:
    """Draw the six bf16 inputs on the CPU in the fixed order X, A, a, B, b, dY.

    ``rows`` (optional) keeps only the first ``rows`` tokens of X and dY; the draws are
    unchanged, so the kept rows are exactly those of the full workload.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    sig = {"X": sx, "A": sw, "a": sbias, "B": sw, "b": sbias, "dY": sdy}
    out: dict[str, torch.Tensor] = {}
    for name, shp in shapes(T, h, f).items():
        v = torch.randn(shp, generator=g, dtype=torch.float32)
        v.mul_(sig[name])
        v = v.to(torch.bfloat16)
        if rows is not None and name in ("X", "dY"):
            v = v[:rows].contiguous()
        out[name] = v
    return out


def make_workload_inputs(w: Workload, *, seed: int = 0, rows: int | None = None
                         ) -> dict[str, torch.Tensor]:
    return make_inputs(w.T, w.h, w.f, seed=seed, sx=w.sx, sw=w.sw, sbias=w.sbias,
                       sdy=w.sdy, rows=rows)


def make_swiglu_inputs(T: int, h: int, f: int, *, seed: int = 0, sx: float = 1.0, sw: float = 0.02,
                       sdy: float = 0.01) -> dict[str, torch.Tensor]:
    """Inputs of the SwiGLU block, drawn in the order X, A, Wg, B, dY (same recipe)."""
    g = torch.Generator("cpu").manual_seed(seed)
    shp = {"X": (T, h), "A": (h, f), "Wg": (h, f), "B": (f, h), "dY": (T, h)}
    sig = {"X": sx, "A": sw, "Wg": sw, "B": sw, "dY": sdy}
    out = {}
    for name, s in shp.items():
        v = torch.randn(s, generator=g, dtype=torch.float32)
        v.mul_(sig[name])
        out[name] = v.to(torch.bfloat16)
    return out


def make_any_inputs(w: Workload, *, seed: int = 0) -> dict[str, torch.Tensor]:
    if w.kind == "swiglu":
        return make_swiglu_inputs(w.T, w.h, w.f, seed=seed, sx=w.sx, sw=w.sw, sdy=w.sdy)
    return make_workload_inputs(w, seed=seed)


# ---- head-parallel attention block ----------------------------------------------------------

@dataclass(frozen=True)
class AttnWorkload:
    """Head-parallel self-attention at a GPT layer shape: b sequences of s tokens, hidden
    width h, a heads of width d = h / a, split over t shards; causal mask (GPT)."""
    name: str
    b: int
    s: int
    h: int
    a: int
    t: int
    causal: bool = True
    sx: float = 1.0
    sw: float = 0.02
    sdy: float = 0.01
    desc: str = ""
    kind: str = "attention"

    @property
    def d(self) -> int:
        return self.h // self.a

    @property
    def T(self) -> int:
        return self.b * self.s

    @property
    def flops_fwd_bwd(self) -> int:
        return attn_flops(self.b, self.s, self.h, self.a, self.d, self.causal)


def attn_flops(b: int, s: int, h: int, a: int, d: int, causal: bool) -> int:
    """Matmul FLOPs of one forward + backward of the attention block. Projections: X Wqkv
    and C Wo forward (8 T h (a d)), twice that backward. Attention core per head: Q K^T and
    P V forward (2 d FLOPs per query-key pair each), dP, dV, dQ, dK backward (2.5x the
    forward); when causal only the s (s + 1) / 2 unmasked pairs count."""
    pairs = s * (s + 1) // 2 if causal else s * s
    return 24 * b * s * h * a * d + 14 * b * a * pairs * d


ATTN_WORKLOADS: dict[str, AttnWorkload] = {w.name: w for w in [
    AttnWorkload("attn-tiny", 2, 200, 256, 2, 2, sw=0.08, sdy=1.0,
                 desc="tiny head-parallel attention b=2 s=200 h=256 a=2 d=128 t=2, causal"),
    AttnWorkload("attn-2k", 2, 2048, 2048, 16, 2,
                 desc="small head-parallel attention b=2 s=2048 h=2048 a=16 d=128 t=2, causal"),
    AttnWorkload("gpt-18b-attn", 4, 2048, 6144, 48, 8,
                 desc="GPT 18B-shaped attention b=4 s=2048 h=6144 a=48 d=128 t=8, causal"),
    AttnWorkload("gpt3-175b-attn", 2, 2048, 12288, 96, 8,
                 desc="GPT-3 175B-shaped attention b=2 s=2048 h=12288 a=96 d=128 t=8, causal"),
]}


def make_attn_inputs(b: int, s: int, h: int, a: int, d: int, *, seed: int = 0, sx: float = 1.0, sw: float = 0.02,
                     sdy: float = 0.01) -> dict[str, torch.Tensor]:
    """Inputs of the attention block, drawn in the order X, Wq, Wk, Wv, Wo, dY (same recipe).
    "Wqkv" is Wq, Wk and Wv side by side ([h, 3 a d]), the layout the C ABI takes."""
    g = torch.Generator("cpu").manual_seed(seed)
    T, hd = b * s, a * d
    shp = {"X": (T, h), "Wq": (h, hd), "Wk": (h, hd), "Wv": (h, hd), "Wo": (hd, h), "dY": (T, h)}
    sig = {"X": sx, "Wq": sw, "Wk": sw, "Wv": sw, "Wo": sw, "dY": sdy}
    out = {}
    for name, sh in shp.items():
        v = torch.randn(sh, generator=g, dtype=torch.float32)
        v.mul_(sig[name])
        out[name] = v.to(torch.bfloat16)
    out["Wqkv"] = torch.cat([out["Wq"], out["Wk"], out["Wv"]], dim=1).contiguous()
    return out


def make_attn_workload_inputs(w: AttnWorkload, *, seed: int = 0) -> dict[str, torch.Tensor]:
    return make_attn_inputs(w.b, w.s, w.h, w.a, w.d, seed=seed, sx=w.sx, sw=w.sw, sdy=w.sdy)
