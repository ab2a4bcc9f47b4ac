"""Tensor-parallel sharding of the attention heads.

The engine runs tensor-parallel workers (nano-vllm-sansho README, "Key
Features": tensor parallelism; "How lunaryes/nano-vllm works", Connections:
the model runner dispatches work to tensor-parallel workers). For attention the
natural shard is by KV head: a rank owns a contiguous range of KV heads, the
query heads that read them (consecutive GQA groups), and those heads' slices of
q, the caches and the outputs. Each rank runs the unchanged kernels on its own
shard; nothing is exchanged inside the attention (the all-reduce after the
output projection lies outside it). This module only computes the ranges and
makes the per-rank contiguous copies.
"""
import numpy as np


def head_shard(rank: int, world_size: int, num_q_heads: int, num_kv_heads: int):
    """(query-head slice, KV-head slice) owned by `rank` of `world_size`."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError(f"rank {rank} outside a world of {world_size}")
    if num_kv_heads <= 0 or num_q_heads % num_kv_heads != 0:
        raise ValueError("num_q_heads must be a positive multiple of num_kv_heads")
    if num_kv_heads % world_size != 0:
        raise ValueError(f"{num_kv_heads} KV heads do not split over {world_size} ranks")
    kv = num_kv_heads // world_size
    g = num_q_heads // num_kv_heads
    return slice(rank * kv * g, (rank + 1) * kv * g), slice(rank * kv, (rank + 1) * kv)


def take_heads(a, heads: slice, dim: int):
    """Contiguous copy of array or tensor `a` restricted to `heads` along `dim`."""
    index = (slice(None),) * dim + (heads,)
    part = a[index]
    if isinstance(part, np.ndarray):
        return np.ascontiguousarray(part)
    return part.contiguous()
