"""Tensor-parallel Transformer MLP block (Megatron partitioning) on one GB300 (sm_103a).

Y = GELU(X*A + a)*B + b forward and backward, with A split by columns and B by rows into
t shards that all live on one GPU; the shard sums run inside tcgen05 tensor-core
accumulators. The compute lives in libmlp_tp.so (C ABI in include/mlp_tp.h); ``_lib`` is
its ctypes binding, ``block`` allocates buffers through PyTorch, ``inputs`` draws the
seeded synthetic workloads.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
