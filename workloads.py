"""Seeded synthetic workloads shaped like Qwen3-0.6B attention layers.

This module is the only thing that the CUDA library's tests and benchmark share
with the fp64 oracle: it draws inputs and holds none of the attention
arithmetic. It plays the part of the engine's KV block manager ("How
lunaryes/nano-vllm works", Components: KV Block Manager, which "allocates cached
blocks" for the scheduler): it picks physical block ids for every sequence
(a seeded permutation of a fixed pool), lists the cache slot it handed out for
every token it wants stored, and fills the pool with a NaN poison so that any
read of a slot that was never written shows up in the results.

Values are drawn as float32 N(0, 1) with a CPU ``torch.Generator`` seeded per
case and rounded to bf16 (round to nearest even); bf16 arrays are returned as
``numpy.uint16`` bit patterns, indices as ``int32``.

Shapes follow one Qwen3-0.6B attention layer: 16 query heads, 8 KV heads,
head_dim 128. The five named workloads are:

* ``tiny``        block size 16, 64-block pool, 4 sequences; decode contexts
                  {17, 64, 100, 128}; prefill prompts {9, 33, 64, 64}.
* ``chain256``    block size 256, 32-block pool; prefill of 16 x 256 tokens,
                  then one decode step at context 257 over the same cache.
* ``ragged256``   block size 256, 64-block pool; prefill lengths U[256, 512],
                  decode contexts U[512, 1024]; 5 % of K rows scaled by 8.
* ``sweep64``     decode at c=64, context 640, block size 256, one distinct
                  seeded cache per layer for 28 layers.
* ``prefix8k``    8 sequences of 8192 tokens whose first 4096 tokens share the
                  same 16 cached blocks; prefill of the last 4096 tokens, then
                  one decode step at context 8193.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

H_Q = 16
H_KV = 8
HEAD_DIM = 128
NUM_LAYERS = 28
POISON_BF16 = 0x7FC0  # a quiet NaN in bf16
SCALE = float(np.float32(1.0 / np.sqrt(HEAD_DIM)))


@dataclass
class Store:
    """New K/V token rows and the cache slot of each (-1: not stored)."""
    k: np.ndarray            # uint16 [T, H_kv, D]
    v: np.ndarray            # uint16 [T, H_kv, D]
    slots: np.ndarray        # int32 [T]
    seq_ids: np.ndarray      # int32 [T]  sequence of each token
    positions: np.ndarray    # int32 [T]  logical position of each token

    @property
    def num_tokens(self) -> int:
        return int(self.slots.shape[0])


@dataclass
class DecodeStep:
    q: np.ndarray            # uint16 [S, H_q, D]
    context_lens: np.ndarray # int32 [S]
    new: Store               # the query tokens' own K/V, stored before attention

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max())


@dataclass
class PrefillStep:
    q: np.ndarray            # uint16 [T_q, H_q, D]
    cu_seqlens_q: np.ndarray # int32 [S + 1]
    cu_seqlens_k: np.ndarray # int32 [S + 1]
    new: Store               # the prompt tokens' K/V, stored before attention

    @property
    def max_seqlen_q(self) -> int:
        return int(np.diff(self.cu_seqlens_q).max(initial=0))

    @property
    def max_seqlen_k(self) -> int:
        return int(np.diff(self.cu_seqlens_k).max(initial=0))


@dataclass
class Case:
    name: str
    block_size: int
    num_blocks: int
    block_tables: np.ndarray           # int32 [S, max_blocks], -1 padded
    history: Optional[Store]           # stored before the step
    step: object                       # DecodeStep | PrefillStep
    H_q: int = H_Q
    H_kv: int = H_KV
    D: int = HEAD_DIM
    scale: float = SCALE
    notes: List[str] = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return int(self.block_tables.shape[0])

    def poisoned_pool(self) -> np.ndarray:
        """A fresh cache array [NB, bs, H_kv, D] filled with the NaN poison."""
        return np.full((self.num_blocks, self.block_size, self.H_kv, self.D),
                       POISON_BF16, np.uint16)


class _Rng:
    def __init__(self, seed: int):
        self.g = torch.Generator().manual_seed(int(seed))

    def normal_bf16(self, *shape) -> np.ndarray:
        x = torch.randn(*shape, generator=self.g, dtype=torch.float32)
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    def normal_f32(self, *shape) -> torch.Tensor:
        return torch.randn(*shape, generator=self.g, dtype=torch.float32)

    def perm(self, n: int) -> np.ndarray:
        return torch.randperm(n, generator=self.g).numpy().astype(np.int32)

    def randint(self, lo: int, hi: int, n: int) -> np.ndarray:
        """n integers uniform in [lo, hi] (inclusive)."""
        return torch.randint(lo, hi + 1, (n,), generator=self.g).numpy().astype(np.int32)


def _to_bf16(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _slots(tables: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray,
           block_size: int) -> np.ndarray:
    """The slot the block manager handed out for each token."""
    blocks = tables[seq_ids, positions // block_size]
    return np.where(blocks < 0, -1, blocks * block_size + positions % block_size).astype(np.int32)


def _store(k: np.ndarray, v: np.ndarray, tables, seq_ids, positions, block_size) -> Store:
    seq_ids = np.asarray(seq_ids, np.int32)
    positions = np.asarray(positions, np.int32)
    return Store(k=k, v=v, slots=_slots(tables, seq_ids, positions, block_size),
                 seq_ids=seq_ids, positions=positions)


def _token_list(ranges):
    """Concatenate (seq, start, stop) ranges into seq_ids, positions arrays."""
    seqs, pos = [], []
    for s, a, b in ranges:
        seqs.append(np.full(b - a, s, np.int32))
        pos.append(np.arange(a, b, dtype=np.int32))
    if not seqs:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    return np.concatenate(seqs), np.concatenate(pos)


def _draw_kv(rng: _Rng, n_tokens: int, H_kv: int, D: int, outlier_frac: float = 0.0):
    """K, V rows for n_tokens tokens; optionally scale round(frac*n) K rows by 8."""
    k = rng.normal_f32(n_tokens, H_kv, D)
    v = rng.normal_f32(n_tokens, H_kv, D)
    if outlier_frac > 0.0 and n_tokens > 0:
        n_out = int(round(outlier_frac * n_tokens))
        rows = torch.from_numpy(rng.perm(n_tokens)[:n_out].astype(np.int64))
        k[rows] *= 8.0
    return _to_bf16(k), _to_bf16(v)


def pad_tables(tables: np.ndarray, used_blocks: np.ndarray) -> np.ndarray:
    """Set entries at index >= used_blocks[s] to -1 (never read)."""
    t = tables.copy()
    for s, n in enumerate(used_blocks):
        t[s, int(n):] = -1
    return t


def decode_case(name: str, seed: int, context_lens, block_size: int, num_blocks: int,
                blocks_per_seq: int, H_q: int = H_Q, H_kv: int = H_KV, D: int = HEAD_DIM,
                outlier_frac: float = 0.0, pad: bool = True) -> Case:
    """Decode step: positions [0, ctx-1) are history, position ctx-1 is the new token."""
    rng = _Rng(seed)
    ctx = np.asarray(context_lens, np.int32)
    S = ctx.shape[0]
    if S * blocks_per_seq > num_blocks:
        raise ValueError("pool too small")
    perm = rng.perm(num_blocks)
    tables = perm[: S * blocks_per_seq].reshape(S, blocks_per_seq).astype(np.int32)
    if pad:
        tables = pad_tables(tables, -(-ctx // block_size))
    hs, hp = _token_list([(s, 0, int(ctx[s]) - 1) for s in range(S)])
    ns, npos = _token_list([(s, int(ctx[s]) - 1, int(ctx[s])) for s in range(S)])
    k, v = _draw_kv(rng, hs.shape[0] + S, H_kv, D, outlier_frac)
    nh = hs.shape[0]
    history = _store(k[:nh], v[:nh], tables, hs, hp, block_size)
    new = _store(k[nh:], v[nh:], tables, ns, npos, block_size)
    q = rng.normal_bf16(S, H_q, D)
    return Case(name=name, block_size=block_size, num_blocks=num_blocks, block_tables=tables,
                history=history, step=DecodeStep(q=q, context_lens=ctx, new=new),
                H_q=H_q, H_kv=H_kv, D=D)


def prefill_case(name: str, seed: int, q_lens, k_lens, block_size: int, num_blocks: int,
                 blocks_per_seq: int, H_q: int = H_Q, H_kv: int = H_KV, D: int = HEAD_DIM,
                 outlier_frac: float = 0.0, pad: bool = True) -> Case:
    """Prefill step: positions [0, Lk-Lq) are a cached prefix (history), the last Lq
    positions are the prompt's new tokens. Every sequence has private blocks."""
    rng = _Rng(seed)
    lq = np.asarray(q_lens, np.int32)
    lk = np.asarray(k_lens, np.int32)
    S = lq.shape[0]
    if np.any(lk < lq):
        raise ValueError("Lk must be >= Lq")
    perm = rng.perm(num_blocks)
    tables = perm[: S * blocks_per_seq].reshape(S, blocks_per_seq).astype(np.int32)
    if pad:
        tables = pad_tables(tables, -(-lk // block_size))
    hs, hp = _token_list([(s, 0, int(lk[s] - lq[s])) for s in range(S)])
    ns, npos = _token_list([(s, int(lk[s] - lq[s]), int(lk[s])) for s in range(S)])
    k, v = _draw_kv(rng, hs.shape[0] + ns.shape[0], H_kv, D, outlier_frac)
    nh = hs.shape[0]
    history = _store(k[:nh], v[:nh], tables, hs, hp, block_size) if nh else None
    new = _store(k[nh:], v[nh:], tables, ns, npos, block_size)
    q = rng.normal_bf16(int(lq.sum()), H_q, D)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return Case(name=name, block_size=block_size, num_blocks=num_blocks, block_tables=tables,
                history=history, step=PrefillStep(q=q, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                                                   new=new),
                H_q=H_q, H_kv=H_kv, D=D)


# --------------------------------------------------------------------------
# The five named workloads.
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 101) -> Case:
    return decode_case("tiny/decode", seed, [17, 64, 100, 128], block_size=16,
                       num_blocks=64, blocks_per_seq=8)


def tiny_prefill(seed: int = 102) -> Case:
    lens = [9, 33, 64, 64]
    return prefill_case("tiny/prefill", seed, lens, lens, block_size=16, num_blocks=64,
                        blocks_per_seq=8)


def chain256(seed: int = 201):
    """Prefill of 16 x 256 tokens, then a decode step at context 257 over the same
    cache: returns (prefill_case, decode_case); the decode case's history is the
    prefill's tokens."""
    rng = _Rng(seed)
    S, bs, NB = 16, 256, 32
    tables = rng.perm(NB).reshape(S, 2).astype(np.int32)
    ps, pp = _token_list([(s, 0, 256) for s in range(S)])
    k, v = _draw_kv(rng, ps.shape[0] + S, H_KV, HEAD_DIM)
    n = ps.shape[0]
    prompt = _store(k[:n], v[:n], tables, ps, pp, bs)
    q_pre = rng.normal_bf16(n, H_Q, HEAD_DIM)
    cu = (np.arange(S + 1) * 256).astype(np.int32)
    pre = Case(name="chain256/prefill", block_size=bs, num_blocks=NB, block_tables=tables,
               history=None, step=PrefillStep(q=q_pre, cu_seqlens_q=cu, cu_seqlens_k=cu,
                                              new=prompt))
    ds, dp = _token_list([(s, 256, 257) for s in range(S)])
    new = _store(k[n:], v[n:], tables, ds, dp, bs)
    q_dec = rng.normal_bf16(S, H_Q, HEAD_DIM)
    dec = Case(name="chain256/decode", block_size=bs, num_blocks=NB, block_tables=tables,
               history=prompt, step=DecodeStep(q=q_dec, context_lens=np.full(S, 257, np.int32),
                                               new=new))
    return pre, dec


def ragged256_prefill(seed: int = 301) -> Case:
    lens = _Rng(seed + 1000).randint(256, 512, 16)
    return prefill_case("ragged256/prefill", seed, lens, lens, block_size=256, num_blocks=64,
                        blocks_per_seq=4, outlier_frac=0.05)


def ragged256_decode(seed: int = 302) -> Case:
    ctx = _Rng(seed + 1000).randint(512, 1024, 16)
    return decode_case("ragged256/decode", seed, ctx, block_size=256, num_blocks=64,
                       blocks_per_seq=4, outlier_frac=0.05)


def sweep64_layer(layer: int, base_seed: int = 4000) -> Case:
    """One layer of the c=64 decode sweep: 64 sequences at context 640 (512 prompt +
    128 generated), 192-block pool of block size 256, seeded per layer."""
    return decode_case(f"sweep64/layer{layer}", base_seed + layer, np.full(64, 640, np.int32),
                       block_size=256, num_blocks=192, blocks_per_seq=3)


def prefix8k(seed: int = 501):
    """8 sequences of 8192 tokens sharing a 4096-token cached prefix (16 blocks with
    the same ids in every table), then one decode step at context 8193.
    Returns (prefill_case, decode_case). The prefill case's history is the shared
    prefix, stored once; the decode case's history is the prefix plus every
    sequence's 4096 prompt tokens."""
    rng = _Rng(seed)
    S, bs, prefix, total = 8, 256, 4096, 8192
    n_shared = prefix // bs                      # 16
    n_private = (total + 1 + bs - 1) // bs - n_shared  # 17: positions 4096..8192
    NB = n_shared + S * n_private                # 152
    perm = rng.perm(NB)
    shared = perm[:n_shared]
    tables = np.stack([np.concatenate([shared, perm[n_shared + s * n_private:
                                                     n_shared + (s + 1) * n_private]])
                       for s in range(S)]).astype(np.int32)
    # the shared prefix is stored once, through sequence 0's table
    hs, hp = _token_list([(0, 0, prefix)])
    ps, pp = _token_list([(s, prefix, total) for s in range(S)])
    ds, dp = _token_list([(s, total, total + 1) for s in range(S)])
    k, v = _draw_kv(rng, hs.shape[0] + ps.shape[0] + S, H_KV, HEAD_DIM)
    a, b = hs.shape[0], hs.shape[0] + ps.shape[0]
    prefix_store = _store(k[:a], v[:a], tables, hs, hp, bs)
    prompt = _store(k[a:b], v[a:b], tables, ps, pp, bs)
    new = _store(k[b:], v[b:], tables, ds, dp, bs)
    q_pre = rng.normal_bf16(ps.shape[0], H_Q, HEAD_DIM)
    cu_q = (np.arange(S + 1) * (total - prefix)).astype(np.int32)
    cu_k = (np.arange(S + 1) * total).astype(np.int32)
    pre = Case(name="prefix8k/prefill", block_size=bs, num_blocks=NB, block_tables=tables,
               history=prefix_store, step=PrefillStep(q=q_pre, cu_seqlens_q=cu_q,
                                                      cu_seqlens_k=cu_k, new=prompt))
    both = Store(k=np.concatenate([prefix_store.k, prompt.k]),
                 v=np.concatenate([prefix_store.v, prompt.v]),
                 slots=np.concatenate([prefix_store.slots, prompt.slots]),
                 seq_ids=np.concatenate([prefix_store.seq_ids, prompt.seq_ids]),
                 positions=np.concatenate([prefix_store.positions, prompt.positions]))
    q_dec = rng.normal_bf16(S, H_Q, HEAD_DIM)
    dec = Case(name="prefix8k/decode", block_size=bs, num_blocks=NB, block_tables=tables,
               history=both, step=DecodeStep(q=q_dec, context_lens=np.full(S, total + 1, np.int32),
                                             new=new))
    return pre, dec


def all_small_cases():
    """The cases small enough for a full oracle comparison in seconds."""
    pre2, dec2 = chain256()
    return [tiny_decode(), tiny_prefill(), pre2, dec2, ragged256_prefill(), ragged256_decode()]
