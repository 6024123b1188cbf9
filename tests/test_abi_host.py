"""Host-side checks of the C ABI: the library builds for sm_103a, loads without a GPU,
exports every function the header declares, and rejects bad arguments before it touches
the GPU (these calls fail in argument checking, so they never reach CUDA)."""

import pytest

from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300 import _lib


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return _lib.lib()


def test_header_symbols_exported(L):
    names = _lib.header_functions()
    assert {"mlp_tp_forward", "mlp_tp_backward", "mlp_tp_workspace_bytes",
            "mlp_tp_query_device_status", "mlp_tp_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/mlp_tp.h but not exported"


def test_status_strings(L):
    for code in range(8):
        s = _lib.mlp_tp_status_string(code)
        assert s.startswith(_lib._STATUS[code])
    assert "unknown" in _lib.mlp_tp_status_string(99)


def test_workspace_bytes():
    assert _lib.mlp_tp_workspace_bytes(128, 64, 256, 2) >= 128 * 256 * 2
    assert _lib.mlp_tp_workspace_bytes(128, 64, 256, 3) == 0      # f % t
    assert _lib.mlp_tp_workspace_bytes(128, 60, 256, 2) == 0      # h % 8
    assert _lib.mlp_tp_workspace_bytes(-1, 64, 256, 2) == 0
    assert _lib.mlp_tp_workspace_bytes(0, 64, 256, 2) > 0         # partials only


def test_forward_workspace_bytes():
    fw = _lib.mlp_tp_forward_workspace_bytes()
    assert fw == 40 * 1024 * 1024  # one 256 KB part per SM of up to 160 SMs
    # every backward workspace holds the split-tail region after its own intermediates
    assert _lib.mlp_tp_workspace_bytes(128, 64, 256, 2) >= 128 * 256 * 2 + fw
    assert _lib.mlp_tp_recompute_workspace_bytes(128, 64, 256, 2) == _lib.mlp_tp_workspace_bytes(128, 64, 256, 2)
    assert _lib.mlp_tp_swiglu_workspace_bytes(128, 64, 256, 2) >= 2 * 128 * 256 * 2 + fw


def test_rejected_calls_launch_nothing(L):
    n0 = _lib.mlp_tp_launch_count()
    assert n0 >= 0
    L.mlp_tp_forward(*([FAKE] * 5), 128, 64, 256, 3, FAKE, FAKE, FAKE, None, 0, None)
    L.mlp_tp_attn_forward(FAKE, FAKE, FAKE, 2, 64, 256, 2, 64, 1, 1, FAKE, FAKE, FAKE, FAKE, None, 0, None)
    assert _lib.mlp_tp_launch_count() == n0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails its checks


@pytest.mark.parametrize("T,h,f,t,code", [
    (128, 64, 256, 3, "MLP_ESHAPE"),   # f % t != 0
    (128, 60, 256, 2, "MLP_ESHAPE"),   # h % 8 != 0
    (128, 64, 256, 64, "MLP_ESHAPE"),  # f/t = 4, not a multiple of 8
    (128, 64, 256, 0, "MLP_EINVAL"),
    (-1, 64, 256, 2, "MLP_EINVAL"),
    (128, 0, 256, 2, "MLP_EINVAL"),
])
def test_forward_rejects_bad_shapes(L, T, h, f, t, code):
    st = L.mlp_tp_forward(*([FAKE] * 5), T, h, f, t, FAKE, FAKE, FAKE, None, 0, None)
    assert st == _lib.STATUS_CODES[code]


def test_forward_rejects_null_and_misaligned(L):
    assert L.mlp_tp_forward(None, *([FAKE] * 4), 128, 64, 256, 2, FAKE, FAKE, FAKE, None, 0, None) == 1
    assert L.mlp_tp_forward(FAKE + 8, *([FAKE] * 4), 128, 64, 256, 2, FAKE, FAKE, FAKE, None, 0, None) == 3
    # the optional split-tail workspace must be 256-byte aligned when given
    assert L.mlp_tp_forward(*([FAKE] * 5), 128, 64, 256, 2, FAKE, FAKE, FAKE, FAKE + 16, 1 << 20, None) == 3


def test_backward_rejects_bad_arguments(L):
    args = [FAKE] * 6 + [128, 64, 256, 2] + [FAKE] * 5
    ws = _lib.mlp_tp_workspace_bytes(128, 64, 256, 2)
    assert L.mlp_tp_backward(*args, FAKE, ws - 256, None) == _lib.STATUS_CODES["MLP_EWORKSPACE"]
    assert L.mlp_tp_backward(*args, FAKE + 16, ws, None) == _lib.STATUS_CODES["MLP_EALIGN"]
    assert L.mlp_tp_backward(*args, None, ws, None) == _lib.STATUS_CODES["MLP_EINVAL"]
    bad = [FAKE] * 6 + [128, 64, 256, 3] + [FAKE] * 5
    assert L.mlp_tp_backward(*bad, FAKE, ws, None) == _lib.STATUS_CODES["MLP_ESHAPE"]


def test_binding_raises_named_error(L):
    with pytest.raises(_lib.MlpError) as ei:
        _lib.mlp_tp_forward(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 64, 256, 3, FAKE, FAKE, FAKE, None, 0, stream=0)
    assert ei.value.name == "MLP_ESHAPE"


def test_attention_workspace_and_shape_rules():
    b, s, h, a, d = 2, 200, 256, 2, 128
    ws = _lib.mlp_tp_attn_workspace_bytes(b, s, h, a, d, 2)
    T, hd = b * s, a * d
    assert ws >= T * hd * 2 + b * a * s * 4 + T * 3 * hd * 2  # dC | D | dQKV
    assert _lib.mlp_tp_attn_workspace_bytes(b, s, h, a, 64, 1) == 0    # d != 128
    assert _lib.mlp_tp_attn_workspace_bytes(b, s, h, 3, d, 2) == 0     # a % t
    assert _lib.mlp_tp_attn_workspace_bytes(b, s, 250, a, d, 1) == 0   # h % 8
    assert _lib.mlp_tp_attn_workspace_bytes(b, 0, h, a, d, 1) == 0     # s < 1
    assert _lib.mlp_tp_attn_workspace_bytes(0, s, h, a, d, 1) == 0     # no tokens, nothing needed


@pytest.mark.parametrize("b,s,h,a,d,t,code", [
    (2, 64, 256, 2, 64, 1, "MLP_ESHAPE"),    # head width other than 128
    (2, 64, 256, 3, 128, 2, "MLP_ESHAPE"),   # a % t
    (2, 64, 250, 2, 128, 1, "MLP_ESHAPE"),   # h % 8
    (2, 0, 256, 2, 128, 1, "MLP_EINVAL"),    # s < 1
    (-1, 64, 256, 2, 128, 1, "MLP_EINVAL"),
    (2, 64, 256, 2, 128, 0, "MLP_EINVAL"),
])
def test_attention_rejects_bad_shapes(L, b, s, h, a, d, t, code):
    st = L.mlp_tp_attn_forward(FAKE, FAKE, FAKE, b, s, h, a, d, t, 1, FAKE, FAKE, FAKE, FAKE, None, 0, None)
    assert st == _lib.STATUS_CODES[code]
    st = L.mlp_tp_attn_backward(*([FAKE] * 7), b, s, h, a, d, t, 1, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == _lib.STATUS_CODES[code]


def test_attention_rejects_null_misaligned_and_short_workspace(L):
    shp = (2, 64, 256, 2, 128, 1, 1)
    assert L.mlp_tp_attn_forward(None, FAKE, FAKE, *shp, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 1
    assert L.mlp_tp_attn_forward(FAKE, FAKE, FAKE, *shp, FAKE + 8, FAKE, FAKE, FAKE, None, 0, None) == 3
    assert L.mlp_tp_attn_forward(FAKE, FAKE, FAKE, *shp, FAKE, FAKE, FAKE, FAKE, FAKE + 16, 1 << 20, None) == 3
    ws = _lib.mlp_tp_attn_workspace_bytes(2, 64, 256, 2, 128, 1)
    args = [FAKE] * 7 + list(shp) + [FAKE] * 3
    assert L.mlp_tp_attn_backward(*args, FAKE, ws - 256, None) == _lib.STATUS_CODES["MLP_EWORKSPACE"]
    assert L.mlp_tp_attn_backward(*args, FAKE + 16, ws, None) == _lib.STATUS_CODES["MLP_EALIGN"]


def test_recompute_backward_workspace_and_checks(L):
    need = _lib.mlp_tp_recompute_workspace_bytes(128, 64, 256, 2)
    assert need == _lib.mlp_tp_workspace_bytes(128, 64, 256, 2)  # G is never stored, not even here
    assert _lib.mlp_tp_recompute_workspace_bytes(128, 64, 256, 3) == 0
    args = [FAKE] * 5 + [128, 64, 256, 2] + [FAKE] * 5
    assert L.mlp_tp_backward_recompute(*args, FAKE, need - 256, None) == _lib.STATUS_CODES["MLP_EWORKSPACE"]
    bad = [FAKE] * 5 + [128, 64, 256, 3] + [FAKE] * 5
    assert L.mlp_tp_backward_recompute(*bad, FAKE, need, None) == _lib.STATUS_CODES["MLP_ESHAPE"]


def test_recompute_forward_checks(L):
    """The forward that keeps H alone: argument checks before any launch (no G argument)."""
    n0 = _lib.mlp_tp_launch_count()
    ok = [FAKE] * 5 + [128, 64, 256, 2] + [FAKE] * 2
    assert L.mlp_tp_forward_recompute(*([FAKE] * 5), 128, 64, 256, 3, FAKE, FAKE, None, 0, None) == \
        _lib.STATUS_CODES["MLP_ESHAPE"]
    assert L.mlp_tp_forward_recompute(*([FAKE] * 5), 128, 64, 256, 2, None, FAKE, None, 0, None) == \
        _lib.STATUS_CODES["MLP_EINVAL"]
    assert L.mlp_tp_forward_recompute(*ok, FAKE + 8, 1 << 20, None) == _lib.STATUS_CODES["MLP_EALIGN"]
    assert L.mlp_tp_forward_recompute(*([FAKE] * 4), FAKE + 2, 128, 64, 256, 2, FAKE, FAKE, None, 0, None) == \
        _lib.STATUS_CODES["MLP_EALIGN"]
    # mlp_tp_forward still needs its G
    assert L.mlp_tp_forward(*([FAKE] * 5), 128, 64, 256, 2, FAKE, None, FAKE, None, 0, None) == \
        _lib.STATUS_CODES["MLP_EINVAL"]
    assert _lib.mlp_tp_launch_count() == n0

