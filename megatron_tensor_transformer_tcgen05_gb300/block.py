"""Device buffers and one-call helpers around the C ABI (allocation through PyTorch only).

A user with their own buffers calls the C-ABI names in ``_lib`` directly; these helpers
allocate the outputs and workspaces on the current CUDA device and call the same entry
points. No arithmetic of the block happens here. The backward workspace ("ws") starts
with the intermediates and ends with the split-tail region, whose last
mlp_tp_forward_workspace_bytes() bytes the forward reuses as its optional workspace
(the forward and backward of one buffer set run in stream order).
"""
from __future__ import annotations

import torch

from ._lib import (mlp_tp_backward, mlp_tp_forward, mlp_tp_forward_workspace_bytes, mlp_tp_workspace_bytes)


def _fwd_ws(buf: dict):
    """The forward's optional workspace: the tail of the backward workspace."""
    ws = buf["ws"]
    n = mlp_tp_forward_workspace_bytes()
    if ws.numel() < n:
        return None, 0
    off = (ws.numel() - n) // 256 * 256
    return ws[off:], ws.numel() - off


def empty_buffers(T: int, h: int, f: int, t: int, device="cuda") -> dict[str, torch.Tensor]:
    """Outputs of one forward + backward, and the backward's workspace."""
    bf, f32 = torch.bfloat16, torch.float32
    ws = mlp_tp_workspace_bytes(T, h, f, t)
    if ws == 0:
        raise ValueError(f"invalid sizes T={T} h={h} f={f} t={t}")
    return {
        "H": torch.empty((T, f), dtype=bf, device=device),
        "G": torch.empty((T, f), dtype=bf, device=device),
        "Y": torch.empty((T, h), dtype=bf, device=device),
        "dX": torch.empty((T, h), dtype=bf, device=device),
        "dA": torch.empty((h, f), dtype=bf, device=device),
        "dB": torch.empty((f, h), dtype=bf, device=device),
        "da": torch.empty((f,), dtype=f32, device=device),
        "db": torch.empty((h,), dtype=f32, device=device),
        "ws": torch.empty((ws,), dtype=torch.uint8, device=device),
    }


def forward(inp: dict, buf: dict, t: int, stream=None) -> None:
    T, h = inp["X"].shape
    f = inp["A"].shape[1]
    fws, fwn = _fwd_ws(buf)
    mlp_tp_forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], T, h, f, t,
                   buf["H"], buf["G"], buf["Y"], fws, fwn, stream)


def backward(inp: dict, buf: dict, t: int, stream=None) -> None:
    T, h = inp["X"].shape
    f = inp["A"].shape[1]
    mlp_tp_backward(inp["X"], inp["A"], inp["B"], buf["H"], buf["G"], inp["dY"], T, h, f, t,
                    buf["dX"], buf["dA"], buf["dB"], buf["da"], buf["db"], buf["ws"],
                    buf["ws"].numel(), stream)


def step(inp: dict, buf: dict, t: int, stream=None) -> None:
    """One forward + backward of the block."""
    forward(inp, buf, t, stream)
    backward(inp, buf, t, stream)


# ---- SwiGLU variant -----------------------------------------------------------------------

def empty_swiglu_buffers(T: int, h: int, f: int, t: int, device="cuda") -> dict[str, torch.Tensor]:
    from ._lib import mlp_tp_swiglu_workspace_bytes
    bf = torch.bfloat16
    ws = mlp_tp_swiglu_workspace_bytes(T, h, f, t)
    if ws == 0:
        raise ValueError(f"invalid sizes T={T} h={h} f={f} t={t}")
    out = {k: torch.empty((T, f), dtype=bf, device=device) for k in ("Ha", "Hg", "U")}
    out.update(Y=torch.empty((T, h), dtype=bf, device=device), dX=torch.empty((T, h), dtype=bf, device=device),
               dA=torch.empty((h, f), dtype=bf, device=device), dWg=torch.empty((h, f), dtype=bf, device=device),
               dB=torch.empty((f, h), dtype=bf, device=device), ws=torch.empty((ws,), dtype=torch.uint8, device=device))
    return out


def swiglu_forward(inp: dict, buf: dict, t: int, stream=None) -> None:
    from ._lib import mlp_tp_swiglu_forward
    T, h = inp["X"].shape
    f = inp["A"].shape[1]
    fws, fwn = _fwd_ws(buf)
    mlp_tp_swiglu_forward(inp["X"], inp["A"], inp["Wg"], inp["B"], T, h, f, t, buf["Ha"], buf["Hg"], buf["U"],
                          buf["Y"], fws, fwn, stream)


def swiglu_backward(inp: dict, buf: dict, t: int, stream=None) -> None:
    from ._lib import mlp_tp_swiglu_backward
    T, h = inp["X"].shape
    f = inp["A"].shape[1]
    mlp_tp_swiglu_backward(inp["X"], inp["A"], inp["Wg"], inp["B"], buf["Ha"], buf["Hg"], buf["U"], inp["dY"], T, h,
                           f, t, buf["dX"], buf["dA"], buf["dWg"], buf["dB"], buf["ws"], buf["ws"].numel(), stream)


def swiglu_step(inp: dict, buf: dict, t: int, stream=None) -> None:
    """One forward + backward of the SwiGLU block."""
    swiglu_forward(inp, buf, t, stream)
    swiglu_backward(inp, buf, t, stream)


# ---- head-parallel attention block ----------------------------------------------------------

def empty_attn_buffers(b: int, s: int, h: int, a: int, d: int, t: int, device="cuda") -> dict[str, torch.Tensor]:
    from ._lib import mlp_tp_attn_workspace_bytes
    bf = torch.bfloat16
    ws = mlp_tp_attn_workspace_bytes(b, s, h, a, d, t)
    if ws == 0 and b > 0:
        raise ValueError(f"invalid sizes b={b} s={s} h={h} a={a} d={d} t={t}")
    ws = max(ws, 256)
    T, hd = b * s, a * d
    return {"QKV": torch.empty((T, 3 * hd), dtype=bf, device=device), "C": torch.empty((T, hd), dtype=bf, device=device),
            "L": torch.empty((b * a, s), dtype=torch.float32, device=device),
            "Y": torch.empty((T, h), dtype=bf, device=device), "dX": torch.empty((T, h), dtype=bf, device=device),
            "dWqkv": torch.empty((h, 3 * hd), dtype=bf, device=device),
            "dWo": torch.empty((hd, h), dtype=bf, device=device),
            "ws": torch.empty((ws,), dtype=torch.uint8, device=device)}


def attn_forward(inp: dict, buf: dict, b: int, s: int, a: int, t: int, causal: bool = True, stream=None) -> None:
    from ._lib import mlp_tp_attn_forward
    h = inp["X"].shape[1]
    d = inp["Wqkv"].shape[1] // (3 * a)
    fws, fwn = _fwd_ws(buf)
    mlp_tp_attn_forward(inp["X"], inp["Wqkv"], inp["Wo"], b, s, h, a, d, t, causal, buf["QKV"], buf["C"], buf["L"],
                        buf["Y"], fws, fwn, stream)


def attn_backward(inp: dict, buf: dict, b: int, s: int, a: int, t: int, causal: bool = True, stream=None) -> None:
    from ._lib import mlp_tp_attn_backward
    h = inp["X"].shape[1]
    d = inp["Wqkv"].shape[1] // (3 * a)
    mlp_tp_attn_backward(inp["X"], inp["Wqkv"], inp["Wo"], buf["QKV"], buf["C"], buf["L"], inp["dY"], b, s, h, a, d,
                         t, causal, buf["dX"], buf["dWqkv"], buf["dWo"], buf["ws"], buf["ws"].numel(), stream)


def attn_step(inp: dict, buf: dict, b: int, s: int, a: int, t: int, causal: bool = True, stream=None) -> None:
    """One forward + backward of the attention block."""
    attn_forward(inp, buf, b, s, a, t, causal, stream)
    attn_backward(inp, buf, b, s, a, t, causal, stream)
