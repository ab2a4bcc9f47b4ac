"""Head-sharded (tensor-parallel) attention: each rank runs the kernels on its
own KV heads and their query heads, with no exchange inside the attention.

CPU: two gloo ranks each run the fp64 oracle on their shard; gathering the
shards reproduces the unsharded oracle bit for bit (each head is computed
independently), which pins the shard ranges. GPU: the CUDA kernels on every
shard of 2, 4 and 8 ranks (run one after another on the one GPU, as replicas
would on separate GPUs) match the oracle's outputs for the same heads."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads as W
from paged_kv_attention_22_gb300.shard import head_shard, take_heads
from runners import oracle_cache as _oracle_cache


def test_head_shard_ranges():
    assert head_shard(0, 2, 16, 8) == (slice(0, 8), slice(0, 4))
    assert head_shard(1, 2, 16, 8) == (slice(8, 16), slice(4, 8))
    assert head_shard(7, 8, 16, 8) == (slice(14, 16), slice(7, 8))
    assert head_shard(0, 1, 16, 8) == (slice(0, 16), slice(0, 8))
    with pytest.raises(ValueError):
        head_shard(0, 3, 16, 8)
    with pytest.raises(ValueError):
        head_shard(2, 2, 16, 8)
    with pytest.raises(ValueError):
        head_shard(0, 2, 12, 8)


def _oracle_shard(case, kc, vc, qh, kvh):
    st = case.step
    q = take_heads(st.q, qh, 1)
    kcs, vcs = take_heads(kc, kvh, 2), take_heads(vc, kvh, 2)
    if isinstance(st, W.DecodeStep):
        return oracle.decode(q, kcs, vcs, case.block_tables, st.context_lens, case.scale)
    return oracle.prefill(q, kcs, vcs, st.cu_seqlens_q, st.cu_seqlens_k, case.block_tables,
                          case.scale)


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    results = {}
    for case in (W.tiny_decode(), W.tiny_prefill()):
        kc, vc = _oracle_cache(case)
        qh, kvh = head_shard(rank, world, case.H_q, case.H_kv)
        o, l = _oracle_shard(case, kc, vc, qh, kvh)
        parts_o = [torch.empty_like(torch.from_numpy(o)) for _ in range(world)]
        parts_l = [torch.empty_like(torch.from_numpy(l)) for _ in range(world)]
        torch.distributed.all_gather(parts_o, torch.from_numpy(o))
        torch.distributed.all_gather(parts_l, torch.from_numpy(l))
        results[case.name] = (torch.cat(parts_o, dim=1).numpy(), torch.cat(parts_l, dim=1).numpy())
    torch.distributed.destroy_process_group()
    out[rank] = results


def test_gathered_oracle_shards_equal_the_unsharded_oracle():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29700 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    for case in (W.tiny_decode(), W.tiny_prefill()):
        kc, vc = _oracle_cache(case)
        full_o, full_l = _oracle_shard(case, kc, vc, slice(None), slice(None))
        for r in range(2):
            o, l = out[r][case.name]
            assert np.array_equal(o, full_o) and np.array_equal(l, full_l)


@pytest.mark.gpu
@pytest.mark.parametrize("world", [2, 4, 8])
def test_kernels_on_every_head_shard_match_the_oracle(world):
    from runners import assert_close, dev_bf16, dev_i32
    import paged_kv_attention_22_gb300 as pkv

    for case in (W.ragged256_decode(), W.ragged256_prefill()):
        kc, vc = _oracle_cache(case)
        full_o, full_l = _oracle_shard(case, kc, vc, slice(None), slice(None))
        st = case.step
        for rank in range(world):
            qh, kvh = head_shard(rank, world, case.H_q, case.H_kv)
            q = dev_bf16(take_heads(st.q, qh, 1))
            kcs, vcs = dev_bf16(take_heads(kc, kvh, 2)), dev_bf16(take_heads(vc, kvh, 2))
            bt = dev_i32(case.block_tables)
            if isinstance(st, W.DecodeStep):
                o, l = pkv.paged_decode_attn(q, kcs, vcs, bt, dev_i32(st.context_lens),
                                             st.max_context_len, case.scale)
            else:
                o, l = pkv.paged_prefill_attn(q, kcs, vcs, dev_i32(st.cu_seqlens_q),
                                              dev_i32(st.cu_seqlens_k), bt, st.max_seqlen_q,
                                              st.max_seqlen_k, case.scale)
            assert pkv.check_device_errors() == 0
            assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), full_o[:, qh],
                         full_l[:, qh], what=f"{case.name} rank {rank}/{world}")
