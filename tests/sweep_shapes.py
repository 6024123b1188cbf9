"""Seeded shape sweeps shared by the GPU parity and guard-band tests.

mlp_sweep_shapes(): (T, h, f, t) reaching every branch of the GEMM launch planner on a GB300
(152 SMs): 128-, 256- and 512-wide tiles; one CTA per tile, CTA pairs and clusters of two
pairs; whole rounds and split tails; ragged edges in every GEMM dimension.
attn_sweep_shapes(): (b, s, h, a, t, causal) with sequence lengths off the 128-query and
64-key blocks, one to three sequences and heads per shard, either mask."""
import numpy as np


def mlp_sweep_shapes():
    rng = np.random.default_rng(20240611)
    out = []
    while len(out) < 8:  # ragged: small enough that the oracle takes well under a second
        t = int(rng.integers(1, 9))
        T = int(rng.integers(1, 1200))
        h = 8 * int(rng.integers(1, 200))
        f = t * 8 * int(rng.integers(1, 120))
        if T * h * f <= 3e8:
            out.append((T, h, f, t))

    def ragged_rows(blocks):  # blocks 256-row blocks, the last one partly filled
        return 256 * blocks - 8 * int(rng.integers(1, 32))

    for blocks in (2, 3, 4):  # wide down-projection and dX: N = h, K = f >= 2048; clusters or pairs
        t = int(rng.choice([1, 2, 4]))
        out.append((ragged_rows(blocks), 512 * int(rng.integers(1, 3)), 512 * int(rng.integers(4, 7)), t))
    # 39 whole 512-wide tiles on 76 CTA pairs: more than half a round, so no split
    out.append((ragged_rows(3), 512 * 13, 2048, 2))
    for blocks in (3, 4):  # wide up-projection and dH: N = f, K = h >= 4096
        t = int(rng.choice([1, 2]))
        out.append((ragged_rows(blocks), 4096 + 8 * int(rng.integers(0, 64)), 512 * int(rng.integers(1, 3)), t))
    # wide dA and dB (K = T >= 2048): h of two 256-row blocks (clusters) and of three (pairs)
    out.append((2048 + 8 * int(rng.integers(1, 32)), 512, 1024, 2))
    out.append((2048 + 8 * int(rng.integers(1, 32)), 768, 1536, 3))
    for _ in range(2):  # short: few tokens, long K
        t = int(rng.choice([2, 4]))
        T = int(rng.integers(1, 257))
        h = 1024 * int(rng.integers(1, 3))
        f = 2048 * int(rng.integers(2, 4))
        out.append((T, h, f, t))
    # at most 128 tokens, 256-wide tiles, K too short to split
    out.append((int(rng.integers(1, 129)), 256, 512, 2))
    return out



def attn_sweep_shapes():
    """(b, s, h, a, t, causal): any sequence length (ragged query and key blocks, shorter than
    a block), one to three sequences, one to three heads per shard, either mask."""
    rng = np.random.default_rng(20240612)
    out = []
    for i in range(6):
        t = int(rng.integers(1, 4))
        a = t * int(rng.integers(1, 4))
        out.append((int(rng.integers(1, 4)), int(rng.integers(1, 1600)), 8 * int(rng.integers(16, 80)), a, t,
                    bool(i % 3 != 2)))
    return out
