"""The host block manager (pkv_blocks.h): slots follow the slot formula (the
oracle's slot_mapping), prefix sharing, reuse of freed blocks, atomic failure,
invariants over a seeded random workload; and, on the GPU, the kernels driven
end to end by the manager's block tables and slots against the oracle."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_22_gb300 as pkv
import workloads as W
from paged_kv_attention_22_gb300 import build as pkv_build


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv_build.build()


def _tokens(rng, n):
    return rng.integers(0, 50000, n).astype(np.int32)


def _formula_slots(bm, seq_id):
    n = bm.num_tokens(seq_id)
    table = bm.block_table(seq_id)[None, :]
    return oracle.slot_mapping(table, np.zeros(n, np.int32), np.arange(n, dtype=np.int32),
                               bm.block_size)


def test_slots_follow_the_slot_formula():
    rng = np.random.default_rng(1)
    bm = pkv.BlockManager(64, 16)
    for sid, n in enumerate([1, 15, 16, 17, 100]):
        assert bm.add_sequence(sid, _tokens(rng, n)) == 0
        assert np.array_equal(bm.slots(sid, 0, n), _formula_slots(bm, sid))
        assert len(bm.block_table(sid)) == -(-n // 16)


def test_shared_prefix_blocks_are_reused_and_counted():
    rng = np.random.default_rng(2)
    bm = pkv.BlockManager(32, 8)
    base = _tokens(rng, 30)
    assert bm.add_sequence(0, base) == 0
    other = np.concatenate([base[:20], _tokens(rng, 5)])
    assert bm.add_sequence(1, other) == 16            # two full blocks of 8 in common
    t0, t1 = bm.block_table(0), bm.block_table(1)
    assert np.array_equal(t0[:2], t1[:2]) and t1[2] not in t0
    assert [bm.ref_count(b) for b in t0[:2]] == [2, 2]
    assert bm.num_free_blocks == 32 - 4 - 2
    # a different first block shares nothing, even with equal later blocks
    diff = base.copy()
    diff[0] += 1
    assert bm.add_sequence(2, diff) == 0


def test_a_fully_cached_prompt_still_computes_its_last_block():
    rng = np.random.default_rng(3)
    bm = pkv.BlockManager(16, 4)
    p = _tokens(rng, 12)
    bm.add_sequence(0, p)
    assert bm.add_sequence(1, p) == 8                 # not 12: one token must be computed
    assert bm.block_table(1)[2] != bm.block_table(0)[2]


def test_freed_blocks_stay_findable_until_handed_out():
    rng = np.random.default_rng(4)
    bm = pkv.BlockManager(6, 4)
    p = _tokens(rng, 9)                               # 3 blocks, 2 full
    bm.add_sequence(0, p)
    held = bm.block_table(0)
    bm.free_sequence(0)
    assert bm.num_free_blocks == 6
    assert bm.add_sequence(1, p) == 8                 # both full blocks found again
    assert np.array_equal(bm.block_table(1)[:2], held[:2])
    bm.free_sequence(1)
    # the oldest-freed blocks go first: fill the pool with other tokens
    bm.add_sequence(2, _tokens(rng, 24))
    bm.free_sequence(2)
    assert bm.add_sequence(3, p) == 0                 # the old content was overwritten


def test_out_of_blocks_changes_nothing():
    rng = np.random.default_rng(5)
    bm = pkv.BlockManager(4, 4)
    bm.add_sequence(0, _tokens(rng, 10))              # 3 blocks
    before = (bm.num_free_blocks, [bm.ref_count(b) for b in range(4)])
    with pytest.raises(pkv.PkvError) as e:
        bm.add_sequence(1, _tokens(rng, 5))           # needs 2
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert (bm.num_free_blocks, [bm.ref_count(b) for b in range(4)]) == before
    with pytest.raises(pkv.PkvError):
        bm.num_tokens(1)
    bm.add_sequence(2, _tokens(rng, 2))               # the one free block fits
    bm.append_token(2, 7)
    bm.append_token(2, 7)
    with pytest.raises(pkv.PkvError) as e:
        bm.append_token(2, 7)                         # block full, none free
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert bm.num_tokens(2) == 4


def test_appended_tokens_fill_blocks_that_new_prompts_share():
    rng = np.random.default_rng(6)
    bm = pkv.BlockManager(16, 4)
    p = _tokens(rng, 3)
    bm.add_sequence(0, p)
    gen = _tokens(rng, 6)
    for t in gen:
        bm.append_token(0, int(t))
    assert bm.num_tokens(0) == 9 and len(bm.block_table(0)) == 3
    assert np.array_equal(bm.slots(0, 0, 9), _formula_slots(bm, 0))
    full = np.concatenate([p, gen])
    assert bm.add_sequence(1, np.concatenate([full[:8], _tokens(rng, 3)])) == 8


def test_argument_errors():
    bm = pkv.BlockManager(8, 4)
    bm.add_sequence(0, [1, 2, 3])
    for call in (lambda: bm.add_sequence(0, [1]), lambda: bm.add_sequence(1, []),
                 lambda: bm.free_sequence(9), lambda: bm.append_token(9, 1),
                 lambda: bm.slots(0, 2, 2), lambda: bm.slots(0, -1, 1),
                 lambda: bm.block_table(0, max_blocks=0)):
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(0, 16)
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(1 << 20, 1 << 12)            # slots would not fit in int32


def test_invariants_over_a_random_workload():
    """Reference counts equal the number of sequences holding each block; free
    blocks are exactly those with none; a sequence never holds a block twice;
    two sequences share a block only where their token prefixes agree; slots
    always follow the formula."""
    rng = np.random.default_rng(7)
    bs, nb = 4, 40
    bm = pkv.BlockManager(nb, bs)
    vocab = 3                                         # small: many shared prefixes
    live = {}
    next_id = 0
    for step in range(600):
        op = rng.integers(0, 3)
        try:
            if op == 0 or not live:
                toks = rng.integers(0, vocab, int(rng.integers(1, 14))).astype(np.int32)
                bm.add_sequence(next_id, toks)
                live[next_id] = list(toks)
                next_id += 1
            elif op == 1:
                sid = list(live)[rng.integers(0, len(live))]
                t = int(rng.integers(0, vocab))
                bm.append_token(sid, t)
                live[sid].append(t)
            else:
                sid = list(live)[rng.integers(0, len(live))]
                bm.free_sequence(sid)
                del live[sid]
        except pkv.PkvError as e:
            assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
        refs = np.zeros(nb, np.int64)
        tables = {}
        for sid, toks in live.items():
            t = bm.block_table(sid)
            assert len(t) == -(-len(toks) // bs) and len(set(t.tolist())) == len(t)
            assert bm.num_tokens(sid) == len(toks)
            assert np.array_equal(bm.slots(sid, 0, len(toks)), _formula_slots(bm, sid))
            refs[t] += 1
            tables[sid] = t
        assert [bm.ref_count(b) for b in range(nb)] == refs.tolist()
        assert bm.num_free_blocks == int((refs == 0).sum())
        seen = {}
        for sid, t in tables.items():
            for i, b in enumerate(t.tolist()):
                if b in seen:
                    osid, oi = seen[b]
                    assert oi == i
                    n = min((i + 1) * bs, len(live[sid]), len(live[osid]))
                    assert live[sid][:n] == live[osid][:n]
                else:
                    seen[b] = (sid, i)


@pytest.mark.gpu
def test_kernels_driven_by_the_block_manager_match_the_oracle():
    """Two prompts sharing 512 tokens admitted through the manager: the store
    uses its slots (the shared blocks are stored once), prefill and a decode
    step use its tables; all against the oracle on the same cache."""
    import torch
    from runners import assert_cache_equal, assert_close, dev_bf16, dev_i32

    bs, nb, H_kv, D, H_q = 256, 12, W.H_KV, W.HEAD_DIM, W.H_Q
    rng = np.random.default_rng(8)
    trng = torch.Generator().manual_seed(8)
    bm = pkv.BlockManager(nb, bs)
    p0 = _tokens(rng, 600)
    p1 = np.concatenate([p0[:512], _tokens(rng, 100)])
    assert bm.add_sequence(0, p0) == 0
    assert bm.add_sequence(1, p1) == 512
    max_blocks = 4

    def rows(n):
        return (torch.randn(n, H_kv, D, generator=trng).to(torch.bfloat16)
                .view(torch.int16).numpy().view(np.uint16))

    # the step's tokens: all of prompt 0, the last 100 of prompt 1
    k = np.concatenate([rows(600), rows(100)])
    v = np.concatenate([rows(600), rows(100)])
    slots = np.concatenate([bm.slots(0, 0, 600), bm.slots(1, 512, 100)])
    q = (torch.randn(700, H_q, D, generator=trng).to(torch.bfloat16)
         .view(torch.int16).numpy().view(np.uint16))
    tables = bm.block_tables([0, 1], max_blocks)
    cu_q = np.array([0, 600, 700], np.int32)
    cu_k = np.array([0, 600, 1212], np.int32)
    scale = float(np.float32(1.0 / np.sqrt(D)))

    pool = np.full((nb, bs, H_kv, D), W.POISON_BF16, np.uint16)
    kc_ref, vc_ref = pool.copy(), pool.copy()
    oracle.kv_store(k, v, kc_ref, vc_ref, slots)
    ref_o, ref_l = oracle.prefill(q, kc_ref, vc_ref, cu_q, cu_k, tables, scale)

    kc, vc = dev_bf16(pool), dev_bf16(pool)
    pkv.kv_store(dev_bf16(k), dev_bf16(v), kc, vc, dev_i32(slots))
    o, l = pkv.paged_prefill_attn(dev_bf16(q), kc, vc, dev_i32(cu_q), dev_i32(cu_k),
                                  dev_i32(tables), 600, 612, scale)
    assert pkv.check_device_errors() == 0
    assert_cache_equal(kc, vc, kc_ref, vc_ref)
    assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), ref_o, ref_l,
                 what="prefill via the block manager")

    # one decode step: each sequence appends a token
    for sid in (0, 1):
        bm.append_token(sid, int(rng.integers(0, 50000)))
    lens = np.array([bm.num_tokens(0), bm.num_tokens(1)], np.int32)
    dslots = np.array([bm.slots(0, lens[0] - 1, 1)[0], bm.slots(1, lens[1] - 1, 1)[0]], np.int32)
    dk, dv = rows(2), rows(2)
    dq = (torch.randn(2, H_q, D, generator=trng).to(torch.bfloat16)
          .view(torch.int16).numpy().view(np.uint16))
    dtables = bm.block_tables([0, 1], max_blocks)
    oracle.kv_store(dk, dv, kc_ref, vc_ref, dslots)
    ref_o, ref_l = oracle.decode(dq, kc_ref, vc_ref, dtables, lens, scale)
    o, l = pkv.paged_decode_attn_store(dev_bf16(dk), dev_bf16(dv), dev_i32(dslots), dev_bf16(dq),
                                       kc, vc, dev_i32(dtables), dev_i32(lens), int(lens.max()),
                                       scale)
    assert pkv.check_device_errors() == 0
    assert_cache_equal(kc, vc, kc_ref, vc_ref)
    assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), ref_o, ref_l,
                 what="decode via the block manager")
