"""GPU parity: the CUDA library against the fp64 oracle on the same seeded
inputs. Cache bytes must be bit-exact over the whole (NaN-poisoned) pool;
attention outputs within max-abs 2e-2 and mean-abs 2e-3, lse within 1e-3."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_22_gb300 as pkv
import workloads as W
from runners import (assert_cache_equal, assert_close, dev_bf16, dev_i32, gpu_attend, gpu_pool,
                     gpu_run, gpu_store, host_u16, oracle_cache, oracle_run,
                     sampled_rows_reference)

pytestmark = pytest.mark.gpu

SMALL = {c.name: c for c in W.all_small_cases()}


@pytest.fixture(autouse=True)
def _reset_knobs():
    pkv.decode_set_config(0, 0)
    yield
    pkv.decode_set_config(0, 0)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_match_oracle(name):
    case = SMALL[name]
    got = gpu_run(case)
    ref = oracle_run(case)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], ref["kc"], ref["vc"])
    assert_close(got["out"], got["lse"], ref["out"], ref["lse"], name)


def test_chain256_prefill_then_decode_on_one_cache():
    pre, dec = W.chain256()
    g1 = gpu_run(pre)
    # decode reuses the prefill's cache: only the new token is stored
    g2 = gpu_run(dec, g1["kc"], g1["vc"], store_history=False)
    r1 = oracle_run(pre)
    r2 = oracle_run(dec)
    assert g1["flags"] == 0 and g2["flags"] == 0
    assert_close(g1["out"], g1["lse"], r1["out"], r1["lse"], "chain prefill")
    assert_close(g2["out"], g2["lse"], r2["out"], r2["lse"], "chain decode")
    assert_cache_equal(g2["kc"], g2["vc"], r2["kc"], r2["vc"])


def test_prefix8k_decode_full():
    _, dec = W.prefix8k()
    got = gpu_run(dec)
    ref = oracle_run(dec)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], ref["kc"], ref["vc"])
    assert_close(got["out"], got["lse"], ref["out"], ref["lse"], "prefix8k decode")


def test_prefix8k_prefill_full():
    # the prefix-cached prefill at full size (8 x 4096 new query rows over a
    # shared 4096-token cached prefix, 16 heads): every output element and
    # every lse against the fp64 oracle, cache bytes over the whole pool
    pre, _ = W.prefix8k()
    got = gpu_run(pre)
    ref = oracle_run(pre)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], ref["kc"], ref["vc"])
    assert got["out"].shape == ref["out"].shape == (32768, pre.H_q, pre.D)
    assert_close(got["out"], got["lse"], ref["out"], ref["lse"], "prefix8k prefill (every row)")


def test_prefix8k_prefill_sampled_rows():
    pre, _ = W.prefix8k()
    got = gpu_run(pre)
    kc, vc = oracle_cache(pre)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], kc, vc)
    assert np.all(np.isfinite(got["out"])) and np.all(np.isfinite(got["lse"]))
    rng = np.random.default_rng(0)
    st = pre.step
    rows = []
    for s in range(pre.num_seqs):
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        for r in [a, a + 1, a + 127, a + 128, b - 129, b - 1] + list(rng.integers(a, b, 6)):
            rows.append((int(r), int(rng.integers(0, pre.H_q))))
    ref_out, ref_lse = sampled_rows_reference(pre, kc, vc, rows)
    idx_r = [r for r, _ in rows]
    idx_h = [h for _, h in rows]
    assert_close(got["out"][idx_r, idx_h], got["lse"][idx_r, idx_h], ref_out, ref_lse,
                 "prefix8k prefill (sampled)")


def test_sweep64_layer_full():
    case = W.sweep64_layer(0)
    got = gpu_run(case)
    ref = oracle_run(case)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], ref["kc"], ref["vc"])
    assert_close(got["out"], got["lse"], ref["out"], ref["lse"], "sweep64 layer 0")


@pytest.mark.parametrize("ctas,variant", [(1, 0), (2, 0), (7, 0), (1000, 0), (0, 1), (3, 1),
                                          (0, 2), (5, 2)])
def test_decode_launch_shape_does_not_change_results(ctas, variant):
    # the grid decides how pairs are cut between CTAs (1 CTA: whole pairs per
    # CTA; 1000 CTAs: more CTAs than units); the variant decides the stages
    for case in (SMALL["ragged256/decode"], SMALL["tiny/decode"]):
        ref = oracle_run(case)
        pkv.decode_set_config(ctas, variant)
        got = gpu_run(case)
        assert got["flags"] == 0
        assert_close(got["out"], got["lse"], ref["out"], ref["lse"], f"{case.name} {ctas}/{variant}")


def test_decode_repeated_calls_reuse_the_workspace():
    case = SMALL["ragged256/decode"]
    ref = oracle_run(case)
    kc, vc = gpu_pool(case)
    gpu_store(case.history, kc, vc)
    gpu_store(case.step.new, kc, vc)
    st = case.step
    q, bt, ctx = dev_bf16(st.q), dev_i32(case.block_tables), dev_i32(st.context_lens)
    ws = pkv.new_decode_workspace(case.num_seqs, case.H_q, case.H_kv, case.D, st.max_context_len)
    ws.fill_(255)  # stale contents must not matter
    for ctas in (0, 5, 0):  # different cuts between CTAs reuse the same workspace
        pkv.decode_set_config(ctas, 0)
        out, lse = pkv.paged_decode_attn(q, kc, vc, bt, ctx, st.max_context_len, case.scale,
                                         workspace=ws)
        assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref["out"],
                     ref["lse"], f"repeat ctas={ctas}")
    assert pkv.check_device_errors() == 0


def _fused_run(case, kc=None, vc=None):
    if kc is None:
        kc, vc = gpu_pool(case)
        gpu_store(case.history, kc, vc)
    st = case.step
    out, lse = pkv.paged_decode_attn_store(
        dev_bf16(st.new.k), dev_bf16(st.new.v), dev_i32(st.new.slots), dev_bf16(st.q), kc, vc,
        dev_i32(case.block_tables), dev_i32(st.context_lens), st.max_context_len, case.scale)
    flags = pkv.check_device_errors()
    return kc, vc, out.double().cpu().numpy(), lse.double().cpu().numpy(), flags


@pytest.mark.parametrize("name", ["tiny/decode", "ragged256/decode", "chain256/decode"])
def test_fused_store_decode_matches_oracle(name):
    case = SMALL[name]
    kc, vc, out, lse, flags = _fused_run(case)
    ref = oracle_run(case)
    assert flags == 0
    assert_cache_equal(kc, vc, ref["kc"], ref["vc"])
    assert_close(out, lse, ref["out"], ref["lse"], "fused " + name)


def test_fused_store_decode_sweep_layer_and_long_context():
    for case in (W.sweep64_layer(3), W.prefix8k()[1],
                 W.decode_case("flong", 41, [20000, 1, 17, 333], block_size=16, num_blocks=5200,
                               blocks_per_seq=1300)):
        kc, vc, out, lse, flags = _fused_run(case)
        ref = oracle_run(case)
        assert flags == 0
        assert_cache_equal(kc, vc, ref["kc"], ref["vc"])
        assert_close(out, lse, ref["out"], ref["lse"], "fused " + case.name)


def test_fused_store_ignores_stale_cache_row():
    # the cache row of the new token holds garbage before the call: the
    # attention must use the new rows, and the row must end up written
    case = SMALL["ragged256/decode"]
    kc, vc = gpu_pool(case)
    gpu_store(case.history, kc, vc)
    junk = np.full_like(case.step.new.k, 0x4200)  # 32.0 in bf16
    gpu_store(W.Store(k=junk, v=junk, slots=case.step.new.slots, seq_ids=case.step.new.seq_ids,
                      positions=case.step.new.positions), kc, vc)
    kc, vc, out, lse, flags = _fused_run(case, kc, vc)
    ref = oracle_run(case)
    assert flags == 0
    assert_cache_equal(kc, vc, ref["kc"], ref["vc"])
    assert_close(out, lse, ref["out"], ref["lse"], "fused over stale row")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_block_relabelling_is_bit_identical(kind):
    case = SMALL["tiny/decode" if kind == "decode" else "tiny/prefill"]
    got = gpu_run(case)
    kc = host_u16(got["kc"])
    vc = host_u16(got["vc"])
    relabel = np.random.default_rng(1).permutation(case.num_blocks).astype(np.int32)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[relabel] = kc
    vc2[relabel] = vc
    bt2 = np.where(case.block_tables >= 0, relabel[np.maximum(case.block_tables, 0)], -1)
    case2 = dataclasses.replace(case, block_tables=bt2.astype(np.int32))
    out2, lse2 = gpu_attend(case2, dev_bf16(kc2), dev_bf16(vc2))
    assert np.array_equal(out2.double().cpu().numpy(), got["out"])
    assert np.array_equal(lse2.double().cpu().numpy(), got["lse"])


def test_decode_matches_last_prefill_row():
    n = 300
    pre = W.prefill_case("p300", 21, [n], [n], block_size=16, num_blocks=20, blocks_per_seq=20)
    got = gpu_run(pre)
    for t in (0, 127, 128, 255, n - 1):
        out_d, lse_d = pkv.paged_decode_attn(
            dev_bf16(pre.step.q[t:t + 1]), got["kc"], got["vc"], dev_i32(pre.block_tables),
            dev_i32(np.array([t + 1], np.int32)), t + 1, pre.scale)
        assert np.abs(out_d.double().cpu().numpy()[0] - got["out"][t]).max() <= 2 * 2e-2
        assert np.abs(lse_d.double().cpu().numpy()[0] - got["lse"][t]).max() <= 2e-3


# ---------------------------------------------------------------- edge cases

def _check_case(case):
    got = gpu_run(case)
    ref = oracle_run(case)
    assert got["flags"] == 0
    assert_cache_equal(got["kc"], got["vc"], ref["kc"], ref["vc"])
    return assert_close(got["out"], got["lse"], ref["out"], ref["lse"], case.name)


def test_decode_single_key_and_block_edges():
    # contexts 1, 15, 16, 17, 31, 32, 33 with block size 16
    _check_case(W.decode_case("edges", 31, [1, 15, 16, 17, 31, 32, 33], block_size=16,
                              num_blocks=40, blocks_per_seq=3))


def test_decode_long_context_mixed():
    _check_case(W.decode_case("long", 32, [32768, 5, 4097, 1000], block_size=256,
                              num_blocks=4 * 128, blocks_per_seq=128))


@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (32, 8), (4, 2)])
def test_decode_other_gqa_groups(h_q, h_kv):
    _check_case(W.decode_case(f"gqa{h_q}x{h_kv}", 33, [77, 300, 1], block_size=32, num_blocks=30,
                              blocks_per_seq=10, H_q=h_q, H_kv=h_kv))


@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (32, 8)])
def test_prefill_other_gqa_groups(h_q, h_kv):
    _check_case(W.prefill_case(f"pgqa{h_q}x{h_kv}", 34, [130, 7], [200, 7], block_size=64,
                               num_blocks=8, blocks_per_seq=4, H_q=h_q, H_kv=h_kv))


def test_prefill_ragged_prefix_empty_and_single_rows():
    # empty segment, single-token prompt over a prefix, unaligned prefix, block size 16
    _check_case(W.prefill_case("ragged", 35, q_lens=[1, 0, 129, 255, 40],
                               k_lens=[1, 30, 129 + 19, 300, 40 + 200], block_size=16,
                               num_blocks=5 * 20, blocks_per_seq=20))


def test_prefill_block_sizes():
    for bs in (32, 48, 128):
        _check_case(W.prefill_case(f"bs{bs}", 36 + bs, [70, 260], [90, 260], block_size=bs,
                                   num_blocks=2 * (300 // bs + 1), blocks_per_seq=300 // bs + 1))


def test_kv_store_minus_one_and_empty():
    case = SMALL["tiny/decode"]
    kc, vc = gpu_pool(case)
    st = case.step.new
    slots = st.slots.copy()
    slots[1] = -1
    pkv.kv_store(dev_bf16(st.k), dev_bf16(st.v), kc, vc, dev_i32(slots))
    empty = np.zeros((0, case.H_kv, case.D), np.uint16)
    pkv.kv_store(dev_bf16(empty), dev_bf16(empty), kc, vc, dev_i32(np.zeros(0, np.int32)))
    assert pkv.check_device_errors() == 0
    rk, rv = case.poisoned_pool(), case.poisoned_pool()
    oracle.kv_store(st.k, st.v, rk, rv, slots)
    assert_cache_equal(kc, vc, rk, rv)


# ---------------------------------------------------------------- device-side checks

def test_out_of_range_slot_is_skipped_and_flagged():
    case = SMALL["tiny/decode"]
    kc, vc = gpu_pool(case)
    st = case.step.new
    slots = st.slots.copy()
    slots[2] = case.num_blocks * case.block_size  # one past the pool
    pkv.kv_store(dev_bf16(st.k), dev_bf16(st.v), kc, vc, dev_i32(slots))
    assert pkv.check_device_errors() & pkv.DEVERR_SLOT
    rk, rv = case.poisoned_pool(), case.poisoned_pool()
    ok = slots.copy()
    ok[2] = -1
    oracle.kv_store(st.k, st.v, rk, rv, ok)
    assert_cache_equal(kc, vc, rk, rv)
    assert pkv.check_device_errors() == 0  # reading clears the word


def test_bad_block_entry_and_context_are_flagged():
    case = SMALL["tiny/decode"]
    got = gpu_run(case)
    bt = case.block_tables.copy()
    bt[2, 0] = case.num_blocks  # outside the pool
    pkv.paged_decode_attn(dev_bf16(case.step.q), got["kc"], got["vc"], dev_i32(bt),
                          dev_i32(case.step.context_lens), case.step.max_context_len, case.scale)
    assert pkv.check_device_errors() & pkv.DEVERR_BLOCK
    ctx = case.step.context_lens.copy()
    ctx[0] = 0
    pkv.paged_decode_attn(dev_bf16(case.step.q), got["kc"], got["vc"],
                          dev_i32(case.block_tables), dev_i32(ctx), case.step.max_context_len,
                          case.scale)
    assert pkv.check_device_errors() & pkv.DEVERR_CONTEXT


def test_prefill_bad_seqlens_are_flagged():
    case = SMALL["tiny/prefill"]
    got = gpu_run(case)
    st = case.step
    # claim a smaller maximum than the real prompt lengths
    pkv.paged_prefill_attn(dev_bf16(st.q), got["kc"], got["vc"], dev_i32(st.cu_seqlens_q),
                           dev_i32(st.cu_seqlens_k), dev_i32(case.block_tables), 32, 64,
                           case.scale)
    assert pkv.check_device_errors() & pkv.DEVERR_SEQLENS


def test_classic_launch_gives_the_same_results():
    # programmatic dependent launch only changes when kernels may start
    case = SMALL["ragged256/decode"]
    pre = SMALL["ragged256/prefill"]
    a = gpu_run(case), gpu_run(pre)
    pkv.set_programmatic_launch(False)
    try:
        b = gpu_run(case), gpu_run(pre)
    finally:
        pkv.set_programmatic_launch(True)
    for x, y in zip(a, b):
        assert np.array_equal(x["out"], y["out"]) and np.array_equal(x["lse"], y["lse"])


def test_fused_store_with_stable_inputs_over_a_chain_of_layers():
    """The decode step as the engine runs it: one fused call per layer back to
    back on one stream, each allowed to read its caches, tables and lengths
    while the previous call finishes (PKV_DECODE_STABLE_INPUTS). Every layer
    matches the oracle and every cache byte is as stored."""
    layers = [W.sweep64_layer(i) for i in range(6)]
    dev = []
    for case in layers:
        kc, vc = gpu_pool(case)
        gpu_store(case.history, kc, vc)
        dev.append((kc, vc))
    torch.cuda.synchronize()
    ws = pkv.new_decode_workspace(64, 16, 8, 128, 640)  # one workspace shared by every layer
    outs = []
    for case, (kc, vc) in zip(layers, dev):
        st = case.step
        outs.append(pkv.paged_decode_attn_store(
            dev_bf16(st.new.k), dev_bf16(st.new.v), dev_i32(st.new.slots), dev_bf16(st.q), kc, vc,
            dev_i32(case.block_tables), dev_i32(st.context_lens), st.max_context_len, case.scale,
            workspace=ws, stable_inputs=True))
    assert pkv.check_device_errors() == 0
    for case, (kc, vc), (o, l) in zip(layers, dev, outs):
        ref = oracle_run(case)
        assert_cache_equal(kc, vc, ref["kc"], ref["vc"])
        assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), ref["out"], ref["lse"],
                     what=case.name + " (stable inputs)")


def test_fused_store_rejects_unknown_flags():
    import ctypes
    case = W.tiny_decode()
    st = case.step
    kc, vc = gpu_pool(case)
    q = dev_bf16(st.q)
    out = torch.empty_like(q)
    ws = pkv.new_decode_workspace(st.q.shape[0], 16, 8, 128, st.max_context_len)
    k, v, slots = dev_bf16(st.new.k), dev_bf16(st.new.v), dev_i32(st.new.slots)
    bt, ctx = dev_i32(case.block_tables), dev_i32(st.context_lens)
    P = ctypes.c_void_p
    rc = pkv.lib().pkv_paged_decode_attn_store(
        P(k.data_ptr()), P(v.data_ptr()), P(slots.data_ptr()), P(q.data_ptr()), P(kc.data_ptr()),
        P(vc.data_ptr()), P(bt.data_ptr()), bt.shape[1], P(ctx.data_ptr()), st.max_context_len,
        q.shape[0], 16, 8, 128, case.block_size, case.num_blocks, ctypes.c_float(case.scale), 0,
        P(out.data_ptr()), None, P(ws.data_ptr()), ws.numel(), 0x2, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG


def test_decode_workspace_reused_across_cut_structures():
    """One workspace, never cleared, through calls whose CTA ranges cut
    different pairs into different numbers of pieces, with one CTA per SM and
    with one unit per CTA (every pair cut into as many pieces as it has
    units)."""
    for ctas in (0, 1000):
        pkv.decode_set_config(ctas, 0)
        try:
            ws = pkv.new_decode_workspace(6, 16, 8, 128, 4096)
            ws.fill_(255)
            for i, ctx in enumerate([[77, 300, 1], [4096, 3, 640, 17, 900, 2], [16, 32],
                                     [300, 301, 302], [1, 1, 1, 1, 1, 1], [2000, 640]]):
                case = W.decode_case(f"reuse{i}", 60 + i, ctx, block_size=64,
                                     num_blocks=6 * 65, blocks_per_seq=65)
                st = case.step
                kc, vc = gpu_pool(case)
                gpu_store(case.history, kc, vc)
                gpu_store(st.new, kc, vc)
                q = dev_bf16(st.q)
                out = torch.full_like(q, float("nan"))  # a row not written fails below
                out, lse = pkv.paged_decode_attn(q, kc, vc, dev_i32(case.block_tables),
                                                 dev_i32(st.context_lens), st.max_context_len,
                                                 case.scale, out=out, workspace=ws)
                assert pkv.check_device_errors() == 0
                ref = oracle_run(case)
                assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(),
                             ref["out"], ref["lse"], f"{case.name} ctas {ctas}")
        finally:
            pkv.decode_set_config(0, 0)

