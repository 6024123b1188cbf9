"""CPU tests of the GEMM launch planner (csrc/gemm_plan.h, the host arithmetic every GEMM launch
goes through): tile widths, two-pair clusters, split tails and grids, against the kernel's
work decomposition (whole tiles in tile order, then each split tile as K ranges) restated here."""
import ctypes
import itertools
import os
import subprocess

import pytest

from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod

HERE = os.path.dirname(os.path.abspath(__file__))
KEYS = ("bn", "cg", "cluster_pairs", "tm", "units", "tiles", "split_tiles", "split_k", "grid", "n_fastest",
        "raster_group")
WS = 40 * 1024 * 1024  # the library's split workspace


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("plan") / "gemm_plan.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-I", build_mod.CSRC,
                    os.path.join(HERE, "gemm_plan_shim.cpp"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.gemm_plan.argtypes = [ctypes.c_int] * 8 + [ctypes.c_ulonglong, ctypes.POINTER(ctypes.c_longlong)]

    def f(M, N, K, bn=256, math=False, splittable=True, sms=152, quads=36, ws=WS):
        out = (ctypes.c_longlong * len(KEYS))()
        lib.gemm_plan(M, N, K, bn, int(math), int(splittable), sms, quads, ws, out)
        return dict(zip(KEYS, out))
    return f


def _work_units(p, K):
    """(tile, kb_lo, kb_hi) of every work unit, as the kernel's work_unit() decodes them."""
    nkb = -(-K // 64)
    n_whole = p["tiles"] - p["split_tiles"]
    units = [(t, 0, nkb) for t in range(n_whole)]
    for r in range(p["split_tiles"]):
        for s in range(p["split_k"]):
            units.append((n_whole + r, s * nkb // p["split_k"], (s + 1) * nkb // p["split_k"]))
    return units


def test_gpt3_175b_plans(plan):
    # forward down-projection and dX: 512 x 512 tiles on 36 clusters, 192 tiles, the last 12 in 3 parts
    p = plan(4096, 12288, 49152)
    assert (p["bn"], p["cg"], p["cluster_pairs"], p["tm"], p["units"], p["tiles"]) == (512, 2, 2, 512, 36, 192)
    assert (p["split_tiles"], p["split_k"], p["grid"]) == (12, 3, 144)
    # up-projection (bias + GELU, K = 12288): wide enough for the math epilogue too
    p = plan(4096, 49152, 12288, math=True)
    assert (p["bn"], p["cluster_pairs"], p["tiles"], p["split_tiles"], p["split_k"]) == (512, 2, 768, 12, 3)
    # dA = X^T dH: 2304 tiles fill 64 rounds exactly, no split
    p = plan(12288, 49152, 4096)
    assert (p["tiles"], p["split_tiles"], p["grid"]) == (2304, 0, 144)


def test_width_and_cluster_rules(plan):
    # K below the thresholds keeps 256-wide pair tiles (2048 plain, 4096 with math)
    assert plan(4096, 12288, 1984)["bn"] == 256
    assert plan(4096, 12288, 2048)["bn"] == 512
    assert plan(4096, 12288, 2304, math=True)["bn"] == 256
    assert plan(4096, 12288, 4096, math=True)["bn"] == 512
    # the SwiGLU derivative (two saved activations in, two outputs) never, at any K: the 175B
    # SwiGLU dU GEMM runs 16 x 128 tiles of 256 x 256 on CTA pairs
    p = plan(4096, 32768, 12288, math=2, splittable=False)
    assert (p["bn"], p["cg"], p["cluster_pairs"], p["tm"], p["tiles"]) == (256, 2, 1, 256, 16 * 128)
    assert all(plan(M, N, K, math=2)["bn"] == 256 for M, N, K in itertools.product((512, 4096), (512, 32768),
                                                                                    (2048, 65536)))
    # N not a multiple of 512, or at most 128 rows: no 512-wide tiles
    assert plan(4096, 2304, 9216)["bn"] == 256
    assert (plan(128, 12288, 49152)["cg"], plan(128, 12288, 49152)["bn"]) == (1, 256)
    # an odd number of 256-row blocks, or clusters of four covering < 90% of the SMs: pairs
    assert plan(2304, 12288, 49152)["cluster_pairs"] == 1
    assert plan(4096, 12288, 49152, quads=34)["cluster_pairs"] == 1
    assert plan(4096, 12288, 49152, quads=35)["cluster_pairs"] == 2
    assert plan(4096, 12288, 49152, quads=0)["cluster_pairs"] == 1
    # the tile order sweeps the smaller operand's dimension fastest
    assert plan(4096, 12288, 4096)["n_fastest"] == 0 and plan(12288, 4096, 4096)["n_fastest"] == 1


def test_no_split_without_room_or_fixup(plan):
    assert plan(4096, 12288, 49152, ws=0)["split_tiles"] == 0
    assert plan(4096, 12288, 49152, splittable=False)["split_tiles"] == 0
    # each part must keep >= 16 k blocks: K = 1024 gives 16 blocks, so no split
    assert plan(512, 1024, 1024)["split_tiles"] == 0
    # too little workspace for two parts of every short-round tile
    assert plan(4096, 12288, 49152, ws=12 * 512 * 512 * 4)["split_tiles"] == 0


SHAPES = list(itertools.product([1, 128, 300, 512, 2048, 4096, 16384], [8, 200, 1024, 2304, 12288],
                                [64, 800, 2048, 4096, 24576]))


@pytest.mark.parametrize("sms,quads", [(152, 36), (148, 37), (132, 0)])
def test_plans_cover_every_tile_and_k_block_once(plan, sms, quads):
    for (M, N, K), math, bn in itertools.product(SHAPES, (0, 1, 2), (128, 256)):
        if bn == 256 and N % 256:
            continue
        p = plan(M, N, K, bn=bn, math=math, sms=sms, quads=quads)
        tiles_m, tiles_n = -(-M // p["tm"]), -(-N // p["bn"])
        assert p["tiles"] == tiles_m * tiles_n
        assert p["cg"] * p["cluster_pairs"] * p["units"] <= sms
        work = _work_units(p, K)
        assert p["grid"] == p["cg"] * p["cluster_pairs"] * min(len(work), p["units"])
        if p["split_tiles"]:
            # the parts of the short last round fit in one round of units and in the workspace
            assert p["split_tiles"] == p["tiles"] % p["units"] or p["tiles"] < p["units"]
            assert p["split_tiles"] * p["split_k"] <= p["units"] and p["split_k"] >= 2
            assert p["split_tiles"] * p["split_k"] * p["tm"] * p["bn"] * 4 <= WS
        covered = {}
        for t, lo, hi in work:
            assert hi - lo >= (16 if p["split_tiles"] and t >= p["tiles"] - p["split_tiles"] else 1)
            covered.setdefault(t, []).append((lo, hi))
        assert sorted(covered) == list(range(p["tiles"]))
        nkb = -(-K // 64)
        for ranges in covered.values():  # each tile's K ranges tile [0, nkb) exactly
            ranges.sort()
            assert ranges[0][0] == 0 and ranges[-1][1] == nkb
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        if p["cluster_pairs"] == 2:
            assert p["bn"] == 512 and -(-M // 256) % 2 == 0 and 40 * p["units"] >= 9 * sms
