"""fp64 CPU oracle for the tensor-parallel MLP block (ctypes front end of mlp_oracle.c).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. The CUDA path does not import it, and it does not
import the CUDA path; the two share only the seeded input generator.

Every function returns float64 numpy arrays. Inputs may be numpy arrays or CPU torch
tensors; bf16 tensors convert to fp64 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mlp_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ACTS = {"gelu_tanh": 0, "gelu_erf": 1, "relu": 2, "identity": 3}


def build(force: bool = False) -> str:
    """Compile mlp_oracle.c into liboracle.so beside it (gcc, -O3, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_act.restype = ctypes.c_double
            lib.oracle_act.argtypes = [i32, ctypes.c_double]
            lib.oracle_act_grad.restype = ctypes.c_double
            lib.oracle_act_grad.argtypes = [i32, ctypes.c_double]
            lib.oracle_num_threads.restype = i32
            lib.oracle_set_num_threads.argtypes = [i32]
            lib.oracle_mlp_forward.restype = i32
            lib.oracle_mlp_forward.argtypes = [i64, i64, i64, i32] + [dp] * 8
            lib.oracle_mlp_backward.restype = i32
            lib.oracle_mlp_backward.argtypes = [i64, i64, i64, i32] + [dp] * 12
            lib.oracle_mlp_sharded.restype = i32
            lib.oracle_mlp_sharded.argtypes = [i64, i64, i64, i64, i32] + [dp] * 14
            lib.oracle_mlp_sampled_bf16.restype = i32
            lib.oracle_mlp_sampled_bf16.argtypes = ([i64, i64, i64, i32] + [dp] * 6 +
                                                    [i64, dp, i64, dp] + [dp] * 6)
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_philox4x32_10.argtypes = [dp, dp, dp]
            lib.oracle_dropout_keep.restype = i32
            lib.oracle_dropout_keep.argtypes = [i64, i64, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64, dp]
            lib.oracle_residual_dropout.restype = i32
            lib.oracle_residual_dropout.argtypes = [i64, i64, ctypes.c_double, dp, dp, dp, dp]
            lib.oracle_dropout_backward.restype = i32
            lib.oracle_dropout_backward.argtypes = [i64, i64, ctypes.c_double, dp, dp, dp]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_silu_grad.restype = ctypes.c_double
            lib.oracle_silu_grad.argtypes = [ctypes.c_double]
            lib.oracle_swiglu_forward.restype = i32
            lib.oracle_swiglu_forward.argtypes = [i64, i64, i64] + [dp] * 8
            lib.oracle_swiglu_backward.restype = i32
            lib.oracle_swiglu_backward.argtypes = [i64, i64, i64] + [dp] * 12
            lib.oracle_swiglu_sampled_bf16.restype = i32
            lib.oracle_swiglu_sampled_bf16.argtypes = [i64, i64, i64] + [dp] * 5 + [i64, dp, i64, dp] + [dp] * 5
            lib.oracle_attn_forward.restype = i32
            lib.oracle_attn_forward.argtypes = [i64] * 5 + [i32] + [dp] * 12
            lib.oracle_attn_backward.restype = i32
            lib.oracle_attn_backward.argtypes = [i64] * 5 + [dp] * 16
            lib.oracle_attn_sharded.restype = i32
            lib.oracle_attn_sharded.argtypes = [i64] * 6 + [i32] + [dp] * 14
            lib.oracle_attn_sampled_bf16.restype = i32
            lib.oracle_attn_sampled_bf16.argtypes = ([i64] * 5 + [i32] + [ctypes.c_void_p] * 5 + [i64, ctypes.c_void_p, i64]
                                                     + [dp] * 2)
            lib.oracle_swiglu_sharded.restype = i32
            lib.oracle_swiglu_sharded.argtypes = [i64, i64, i64, i64] + [dp] * 12
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _bits(x) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU torch bf16 tensor, as a contiguous uint16 array."""
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def act(x, kind: str = "gelu_tanh") -> np.ndarray:
    lib = _load()
    xs = _f64(x)
    return np.array([lib.oracle_act(ACTS[kind], float(v)) for v in xs.ravel()]).reshape(xs.shape)


def act_grad(x, kind: str = "gelu_tanh") -> np.ndarray:
    lib = _load()
    xs = _f64(x)
    return np.array([lib.oracle_act_grad(ACTS[kind], float(v)) for v in xs.ravel()]).reshape(xs.shape)


def forward(X, A, a, B, b, act: str = "gelu_tanh"):
    """(H, G, Y) of the unsharded block."""
    lib = _load()
    X, A, a, B, b = map(_f64, (X, A, a, B, b))
    T, h = X.shape
    f = A.shape[1]
    assert A.shape == (h, f) and a.shape == (f,) and B.shape == (f, h) and b.shape == (h,)
    H = np.empty((T, f)); G = np.empty((T, f)); Y = np.empty((T, h))
    rc = lib.oracle_mlp_forward(T, h, f, ACTS[act], _p(X), _p(A), _p(a), _p(B), _p(b),
                                _p(H), _p(G), _p(Y))
    assert rc == 0, rc
    return H, G, Y


def backward(X, A, B, H, G, dY, act: str = "gelu_tanh") -> dict:
    """dX, dA, da, dB, db (and dH) of the unsharded block, from the forward's H and G."""
    lib = _load()
    X, A, B, H, G, dY = map(_f64, (X, A, B, H, G, dY))
    T, h = X.shape
    f = A.shape[1]
    out = {"dX": np.empty((T, h)), "dA": np.empty((h, f)), "da": np.empty(f),
           "dB": np.empty((f, h)), "db": np.empty(h), "dH": np.empty((T, f))}
    rc = lib.oracle_mlp_backward(T, h, f, ACTS[act], _p(X), _p(A), _p(B), _p(H), _p(G), _p(dY),
                                 _p(out["dX"]), _p(out["dA"]), _p(out["da"]), _p(out["dB"]),
                                 _p(out["db"]), _p(out["dH"]))
    assert rc == 0, rc
    return out


def fwd_bwd(inp: dict, act: str = "gelu_tanh") -> dict:
    """Every output of one forward + backward: Y, H, G, dX, dA, da, dB, db, dH."""
    H, G, Y = forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], act)
    out = backward(inp["X"], inp["A"], inp["B"], H, G, inp["dY"], act)
    out.update(H=H, G=G, Y=Y)
    return out


def sharded(inp: dict, t: int, act: str = "gelu_tanh", parts: bool = False) -> dict:
    """The block computed shard by shard with explicit sums over the t shards."""
    lib = _load()
    X, A, a, B, b, dY = (_f64(inp[k]) for k in ("X", "A", "a", "B", "b", "dY"))
    T, h = X.shape
    f = A.shape[1]
    out = {"Y": np.empty((T, h)), "dX": np.empty((T, h)), "dA": np.empty((h, f)),
           "da": np.empty(f), "dB": np.empty((f, h)), "db": np.empty(h)}
    Yp = np.empty((t, T, h)) if parts else None
    dXp = np.empty((t, T, h)) if parts else None
    rc = lib.oracle_mlp_sharded(T, h, f, t, ACTS[act], _p(X), _p(A), _p(a), _p(B), _p(b), _p(dY),
                                _p(out["Y"]), _p(out["dX"]), _p(out["dA"]), _p(out["da"]),
                                _p(out["dB"]), _p(out["db"]),
                                _p(Yp) if parts else None, _p(dXp) if parts else None)
    if rc != 0:
        raise ValueError(f"oracle_mlp_sharded rejected T={T} h={h} f={f} t={t} (rc={rc})")
    if parts:
        out["Y_part"] = Yp
        out["dX_part"] = dXp
    return out


def sampled_bf16(inp: dict, rows, cols, act: str = "gelu_tanh") -> dict:
    """Sampled entries of the block over bf16 inputs (torch bf16 CPU tensors).

    Returns Y_rows [nR,h], dX_rows [nR,h], dA_cols [h,nC], dB_rows [nC,h], da [nC], db [h].
    """
    lib = _load()
    X, A, a, B, b, dY = (_bits(inp[k]) for k in ("X", "A", "a", "B", "b", "dY"))
    T, h = X.shape
    f = A.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    nR, nC = len(rows), len(cols)
    Yr = np.empty((nR, h)); dXr = np.empty((nR, h)); dAc = np.empty((nC, h))
    dBc = np.empty((nC, h)); dac = np.empty(nC); db = np.empty(h)
    rc = lib.oracle_mlp_sampled_bf16(T, h, f, ACTS[act], _p(X), _p(A), _p(a), _p(B), _p(b), _p(dY),
                                     nR, _p(rows), nC, _p(cols), _p(Yr), _p(dXr), _p(dAc), _p(dBc),
                                     _p(dac), _p(db))
    assert rc == 0, rc
    return {"Y_rows": Yr, "dX_rows": dXr, "dA_cols": dAc.T.copy(), "dB_rows": dBc, "da": dac,
            "db": db}


# ---- bias + dropout + residual add on the block output ----------------------------------

def philox4x32_10(counter, key) -> tuple:
    """Philox4x32-10 of one 128-bit counter (4 uint32) under a 64-bit key (2 uint32)."""
    lib = _load()
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return tuple(int(v) for v in out)


def dropout_keep(T: int, h: int, p: float, seed: int, offset: int = 0) -> np.ndarray:
    """Keep mask (uint8 0/1, [T,h]) of dropout with probability p."""
    lib = _load()
    keep = np.empty((T, h), dtype=np.uint8)
    rc = lib.oracle_dropout_keep(T, h, float(p), int(seed), int(offset), _p(keep))
    if rc != 0:
        raise ValueError(f"bad dropout arguments p={p}")
    return keep


def residual_dropout(Y, R, keep, p: float) -> np.ndarray:
    """Z = R + keep * Y / (1 - p)."""
    lib = _load()
    Y, R = _f64(Y), _f64(R)
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    T, h = Y.shape
    Z = np.empty((T, h))
    rc = lib.oracle_residual_dropout(T, h, float(p), _p(Y), _p(R), _p(keep), _p(Z))
    assert rc == 0, rc
    return Z


def dropout_backward(dZ, keep, p: float) -> np.ndarray:
    """dL/dY = dL/dZ * keep / (1 - p)."""
    lib = _load()
    dZ = _f64(dZ)
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    T, h = dZ.shape
    dY = np.empty((T, h))
    rc = lib.oracle_dropout_backward(T, h, float(p), _p(dZ), _p(keep), _p(dY))
    assert rc == 0, rc
    return dY


def fwd_bwd_residual_dropout(inp: dict, R, dZ, p: float, seed: int, offset: int = 0,
                             act: str = "gelu_tanh") -> dict:
    """The block followed by bias + dropout + residual add: Z, and every gradient given dZ."""
    T, h = _f64(inp["X"]).shape
    keep = dropout_keep(T, h, p, seed, offset)
    H, G, Y = forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], act)
    Z = residual_dropout(Y, R, keep, p)
    dY = dropout_backward(dZ, keep, p)
    out = backward(inp["X"], inp["A"], inp["B"], H, G, dY, act)
    out.update(H=H, G=G, Y=Y, Z=Z, keep=keep, dY=dY, dR=_f64(dZ))
    return out


# ---- SwiGLU variant: Y = (SiLU(X A) * X Wg) B ---------------------------------------------

def silu(x) -> np.ndarray:
    lib = _load()
    xs = _f64(x)
    return np.array([lib.oracle_silu(float(v)) for v in xs.ravel()]).reshape(xs.shape)


def silu_grad(x) -> np.ndarray:
    lib = _load()
    xs = _f64(x)
    return np.array([lib.oracle_silu_grad(float(v)) for v in xs.ravel()]).reshape(xs.shape)


def swiglu_fwd_bwd(inp: dict) -> dict:
    """Ha, Hg, U, Y and dX, dA, dWg, dB of the SwiGLU block (inputs X, A, Wg, B, dY)."""
    lib = _load()
    X, A, Wg, B, dY = (_f64(inp[k]) for k in ("X", "A", "Wg", "B", "dY"))
    T, h = X.shape
    f = A.shape[1]
    o = {k: np.empty((T, f)) for k in ("Ha", "Hg", "U")}
    o["Y"] = np.empty((T, h))
    rc = lib.oracle_swiglu_forward(T, h, f, _p(X), _p(A), _p(Wg), _p(B), _p(o["Ha"]), _p(o["Hg"]), _p(o["U"]),
                                   _p(o["Y"]))
    assert rc == 0, rc
    o.update(dX=np.empty((T, h)), dA=np.empty((h, f)), dWg=np.empty((h, f)), dB=np.empty((f, h)))
    rc = lib.oracle_swiglu_backward(T, h, f, _p(X), _p(A), _p(Wg), _p(B), _p(o["Ha"]), _p(o["Hg"]), _p(o["U"]),
                                    _p(dY), _p(o["dX"]), _p(o["dA"]), _p(o["dWg"]), _p(o["dB"]))
    assert rc == 0, rc
    return o


def swiglu_sharded(inp: dict, t: int, parts: bool = False) -> dict:
    lib = _load()
    X, A, Wg, B, dY = (_f64(inp[k]) for k in ("X", "A", "Wg", "B", "dY"))
    T, h = X.shape
    f = A.shape[1]
    o = {"Y": np.empty((T, h)), "dX": np.empty((T, h)), "dA": np.empty((h, f)), "dWg": np.empty((h, f)),
         "dB": np.empty((f, h))}
    Yp = np.empty((t, T, h)) if parts else None
    dXp = np.empty((t, T, h)) if parts else None
    rc = lib.oracle_swiglu_sharded(T, h, f, t, _p(X), _p(A), _p(Wg), _p(B), _p(dY), _p(o["Y"]), _p(o["dX"]),
                                   _p(o["dA"]), _p(o["dWg"]), _p(o["dB"]), _p(Yp) if parts else None,
                                   _p(dXp) if parts else None)
    if rc != 0:
        raise ValueError(f"oracle_swiglu_sharded rejected f={f} t={t}")
    if parts:
        o["Y_part"], o["dX_part"] = Yp, dXp
    return o


def swiglu_sampled_bf16(inp: dict, rows, cols) -> dict:
    """Sampled entries of the SwiGLU block over bf16 inputs: Y_rows, dX_rows [nR,h];
    dA_cols, dWg_cols [h,nC]; dB_rows [nC,h]."""
    lib = _load()
    X, A, Wg, B, dY = (_bits(inp[k]) for k in ("X", "A", "Wg", "B", "dY"))
    T, h = X.shape
    f = A.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    nR, nC = len(rows), len(cols)
    Yr = np.empty((nR, h)); dXr = np.empty((nR, h)); dAc = np.empty((nC, h)); dWc = np.empty((nC, h))
    dBc = np.empty((nC, h))
    rc = lib.oracle_swiglu_sampled_bf16(T, h, f, _p(X), _p(A), _p(Wg), _p(B), _p(dY), nR, _p(rows), nC, _p(cols),
                                        _p(Yr), _p(dXr), _p(dAc), _p(dWc), _p(dBc))
    assert rc == 0, rc
    return {"Y_rows": Yr, "dX_rows": dXr, "dA_cols": dAc.T.copy(), "dWg_cols": dWc.T.copy(), "dB_rows": dBc}


# ---- head-parallel self-attention block ---------------------------------------------------

def attn_fwd_bwd(inp: dict, b: int, s: int, a: int, causal: bool = True) -> dict:
    """Q, K, V, P, C, Y and dX, dWq, dWk, dWv, dWo of the attention block.

    inp: X [b*s, h], Wq/Wk/Wv [h, a*d], Wo [a*d, h], dY [b*s, h]."""
    lib = _load()
    X, Wq, Wk, Wv, Wo, dY = (_f64(inp[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo", "dY"))
    T, h = X.shape
    hd = Wq.shape[1]
    assert T == b * s and hd % a == 0
    d = hd // a
    o = {k: np.empty((T, hd)) for k in ("Q", "K", "V", "C")}
    o["P"] = np.empty((b, a, s, s))
    o["Y"] = np.empty((T, h))
    o["L"] = np.empty((b * a, s))
    rc = lib.oracle_attn_forward(b, s, h, a, d, int(causal), _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(o["Q"]),
                                 _p(o["K"]), _p(o["V"]), _p(o["P"]), _p(o["C"]), _p(o["Y"]), _p(o["L"]))
    assert rc == 0, rc
    o.update(dX=np.empty((T, h)), dWq=np.empty((h, hd)), dWk=np.empty((h, hd)), dWv=np.empty((h, hd)),
             dWo=np.empty((hd, h)))
    rc = lib.oracle_attn_backward(b, s, h, a, d, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(o["Q"]), _p(o["K"]),
                                  _p(o["V"]), _p(o["P"]), _p(o["C"]), _p(dY), _p(o["dX"]), _p(o["dWq"]),
                                  _p(o["dWk"]), _p(o["dWv"]), _p(o["dWo"]))
    assert rc == 0, rc
    return o


def attn_sharded(inp: dict, b: int, s: int, a: int, t: int, causal: bool = True, parts: bool = False) -> dict:
    lib = _load()
    X, Wq, Wk, Wv, Wo, dY = (_f64(inp[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo", "dY"))
    T, h = X.shape
    hd = Wq.shape[1]
    d = hd // a
    o = {"Y": np.empty((T, h)), "dX": np.empty((T, h)), "dWq": np.empty((h, hd)), "dWk": np.empty((h, hd)),
         "dWv": np.empty((h, hd)), "dWo": np.empty((hd, h))}
    Yp = np.empty((t, T, h)) if parts else None
    dXp = np.empty((t, T, h)) if parts else None
    rc = lib.oracle_attn_sharded(b, s, h, a, d, t, int(causal), _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(dY),
                                 _p(o["Y"]), _p(o["dX"]), _p(o["dWq"]), _p(o["dWk"]), _p(o["dWv"]), _p(o["dWo"]),
                                 _p(Yp) if parts else None, _p(dXp) if parts else None)
    if rc != 0:
        raise ValueError(f"oracle_attn_sharded rejected a={a} t={t}")
    if parts:
        o["Y_part"], o["dX_part"] = Yp, dXp
    return o


def attn_sampled_bf16(inp: dict, b: int, s: int, a: int, rows, heads, causal: bool = True) -> dict:
    """C[rows, heads] ([n_rows, n_heads, d]) and L[rows, heads] from the bf16 inputs, without
    computing the whole block (sampled outputs at full size)."""
    lib = _load()
    X, Wq, Wk, Wv = (_bits(inp[k]) for k in ("X", "Wq", "Wk", "Wv"))
    T, h = X.shape
    hd = Wq.shape[1]
    d = hd // a
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    C = np.empty((len(rows), len(heads), d))
    L = np.empty((len(rows), len(heads)))
    rc = lib.oracle_attn_sampled_bf16(b, s, h, a, d, int(causal), _p(X), _p(Wq), _p(Wk), _p(Wv), _p(rows), len(rows),
                                      _p(heads), len(heads), _p(C), _p(L))
    assert rc == 0, rc
    return {"C": C, "L": L}
