"""Pins for the fp64 oracle, checked against things other than itself:
torch's fp64 scaled_dot_product_attention and logsumexp on keys assembled in
logical order from the generator's token lists (not through slots or tables),
closed forms, and invariants of the definition. CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bf16_bits_to_f64, logical_kv, sdpa_rows


def _filled_cache(case, extra_stores=()):
    kc, vc = case.poisoned_pool(), case.poisoned_pool()
    for st in ([case.history] if case.history is not None else []) + list(extra_stores):
        oracle.kv_store(st.k, st.v, kc, vc, st.slots)
    return kc, vc


def _run_decode(case):
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    return oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale)


def _run_prefill(case):
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    return oracle.prefill(st.q, kc, vc, st.cu_seqlens_q, st.cu_seqlens_k,
                          case.block_tables, case.scale)


def _stores(case):
    return ([case.history] if case.history is not None else []) + [case.step.new]


# ---------------------------------------------------------------- slot mapping

def test_slot_mapping_closed_form():
    # table row [5, 2, -1], block size 16: position p -> table[p // 16] * 16 + p % 16
    bt = np.array([[5, 2, -1]], np.int32)
    pos = np.array([0, 15, 16, 31, 32], np.int32)
    got = oracle.slot_mapping(bt, np.zeros(5, np.int32), pos, 16)
    assert got.tolist() == [80, 95, 32, 47, -1]


@pytest.mark.parametrize("make", [W.tiny_decode, W.tiny_prefill, W.ragged256_decode])
def test_generator_slots_match_oracle(make):
    case = make()
    for st in _stores(case):
        want = oracle.slot_mapping(case.block_tables, st.seq_ids, st.positions, case.block_size)
        np.testing.assert_array_equal(st.slots, want)
        # the block manager never hands out one slot twice
        valid = st.slots[st.slots >= 0]
        assert np.unique(valid).size == valid.size


# ---------------------------------------------------------------- KV store

def test_kv_store_places_rows_and_leaves_the_rest():
    case = W.tiny_decode()
    kc, vc = _filled_cache(case, [case.step.new])
    rows_k = kc.reshape(-1, case.H_kv, case.D)
    rows_v = vc.reshape(-1, case.H_kv, case.D)
    written = np.zeros(rows_k.shape[0], bool)
    for st in _stores(case):
        np.testing.assert_array_equal(rows_k[st.slots], st.k)
        np.testing.assert_array_equal(rows_v[st.slots], st.v)
        written[st.slots] = True
    assert np.all(rows_k[~written] == W.POISON_BF16)
    assert np.all(rows_v[~written] == W.POISON_BF16)


def test_kv_store_skips_minus_one_and_rejects_out_of_range():
    kc = np.full((2, 4, 1, 8), W.POISON_BF16, np.uint16)
    vc = kc.copy()
    k = np.arange(16, dtype=np.uint16).reshape(2, 1, 8)
    v = k + 100
    oracle.kv_store(k, v, kc, vc, np.array([-1, 5], np.int32))
    flat = kc.reshape(8, 8)
    assert np.all(flat[5] == k[1, 0]) and np.all(flat[[0, 1, 2, 3, 4, 6, 7]] == W.POISON_BF16)
    before = kc.copy()
    with pytest.raises(oracle.OracleError):
        oracle.kv_store(k, v, kc, vc, np.array([3, 8], np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.kv_store(k, v, kc, vc, np.array([-2, 1], np.int32))
    np.testing.assert_array_equal(kc, before)  # nothing written on rejection


# ---------------------------------------------------------------- attention vs library SDPA

@pytest.mark.parametrize("make", [W.tiny_decode, W.ragged256_decode])
def test_decode_matches_library_attention(make):
    case = make()
    out, lse = _run_decode(case)
    st = case.step
    for s in range(case.num_seqs):
        ctx = int(st.context_lens[s])
        k, v = logical_kv(_stores(case), s, ctx)
        ref_out, ref_lse = sdpa_rows(st.q[s:s + 1], k, v, case.scale, [ctx])
        np.testing.assert_allclose(out[s], ref_out[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[s], ref_lse[0], rtol=0, atol=1e-12)


def _prefill_vs_sdpa(case):
    out, lse = _run_prefill(case)
    st = case.step
    for s in range(case.num_seqs):
        q0, q1 = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        Lq, Lk = q1 - q0, int(st.cu_seqlens_k[s + 1] - st.cu_seqlens_k[s])
        if Lq == 0:
            continue
        k, v = logical_kv(_stores(case), s, Lk)
        limits = [Lk - Lq + i + 1 for i in range(Lq)]  # bottom-right causal
        ref_out, ref_lse = sdpa_rows(st.q[q0:q1], k, v, case.scale, limits)
        np.testing.assert_allclose(out[q0:q1], ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[q0:q1], ref_lse, rtol=0, atol=1e-12)


def test_prefill_matches_library_attention_no_prefix():
    _prefill_vs_sdpa(W.tiny_prefill())


def test_prefill_matches_library_attention_with_cached_prefix():
    # three sequences with 0, 20 and 45 cached prefix tokens, block size 16,
    # plus an empty segment (Lq = 0) in the middle
    case = W.prefill_case("prefix-small", 7, q_lens=[12, 0, 30, 19], k_lens=[12, 5, 50, 64],
                          block_size=16, num_blocks=40, blocks_per_seq=6)
    _prefill_vs_sdpa(case)


# ---------------------------------------------------------------- invariants and closed forms

def test_block_relabelling_is_bit_identical():
    case = W.tiny_decode()
    out, lse = _run_decode(case)
    kc, vc = _filled_cache(case, [case.step.new])
    relabel = np.random.default_rng(0).permutation(case.num_blocks).astype(np.int32)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[relabel] = kc
    vc2[relabel] = vc
    bt2 = np.where(case.block_tables >= 0, relabel[np.maximum(case.block_tables, 0)], -1)
    out2, lse2 = oracle.decode(case.step.q, kc2, vc2, bt2.astype(np.int32),
                               case.step.context_lens, case.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_single_key_returns_its_value():
    case = W.decode_case("one-key", 3, [1, 1], block_size=16, num_blocks=4, blocks_per_seq=1)
    out, lse = _run_decode(case)
    new = case.step.new
    for s in range(2):
        for h in range(case.H_q):
            g = h // (case.H_q // case.H_kv)
            np.testing.assert_array_equal(out[s, h], bf16_bits_to_f64(new.v[s, g]).numpy())
            z = case.scale * float(np.dot(bf16_bits_to_f64(case.step.q[s, h]).numpy(),
                                          bf16_bits_to_f64(new.k[s, g]).numpy()))
            assert abs(lse[s, h] - z) <= 1e-12 * max(1.0, abs(z))


def test_constant_values_give_that_value():
    case = W.tiny_decode()
    c = np.uint16(0x3FC0)  # 1.5 in bf16
    for st in _stores(case):
        st.v[...] = c
    out, _ = _run_decode(case)
    # summation rounding: at most a few ulps per key over <= 128 keys
    np.testing.assert_allclose(out, 1.5, rtol=0, atol=1e-13)


def test_equal_keys_give_mean_value_and_log_count():
    case = W.decode_case("equal-keys", 5, [37, 9], block_size=16, num_blocks=8, blocks_per_seq=3)
    for st in _stores(case):
        st.k[...] = case.step.new.k[0:1]
    out, lse = _run_decode(case)
    for s in range(case.num_seqs):
        ctx = int(case.step.context_lens[s])
        k, v = logical_kv(_stores(case), s, ctx)
        vf = bf16_bits_to_f64(v).numpy()
        for h in range(case.H_q):
            g = h // 2
            np.testing.assert_allclose(out[s, h], vf[:, g].mean(axis=0), rtol=0, atol=1e-14)
            z = case.scale * float(np.dot(bf16_bits_to_f64(case.step.q[s, h]).numpy(),
                                          bf16_bits_to_f64(k[0, g]).numpy()))
            assert abs(lse[s, h] - (z + math.log(ctx))) <= 1e-12


def test_two_key_closed_form():
    """q = e0, k0 = 0, k1 = 2 e0, scale 1/2: logits (0, 1), so the weights are
    sigmoid(-1) and sigmoid(1) and lse = 1 + ln(1 + e^-1)."""
    D = 4
    bf = lambda x: np.array(x, np.float32).astype(np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)
    q = bf([[[1, 0, 0, 0]]])
    kc = np.full((1, 16, 1, D), W.POISON_BF16, np.uint16)
    vc = kc.copy()
    kc[0, 0, 0] = bf([0, 0, 0, 0]); kc[0, 1, 0] = bf([2, 0, 0, 0])
    vc[0, 0, 0] = bf([1, 0, 0, 0]); vc[0, 1, 0] = bf([0, 1, 0, 0])
    out, lse = oracle.decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([2], np.int32), 0.5)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    np.testing.assert_allclose(out[0, 0], [sig(-1), sig(1), 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - (1.0 + math.log1p(math.exp(-1.0)))) < 1e-15


def test_causal_row_ignores_later_keys():
    case = W.prefill_case("causal", 11, q_lens=[40], k_lens=[40], block_size=16,
                          num_blocks=3, blocks_per_seq=3)
    out, lse = _run_prefill(case)
    i = 17
    # perturb every key/value after position i
    sel = case.step.new.positions > i
    case.step.new.k[sel] ^= np.uint16(0x1234)
    case.step.new.v[sel] ^= np.uint16(0x0F0F)
    out2, lse2 = _run_prefill(case)
    assert np.array_equal(out[: i + 1], out2[: i + 1]) and np.array_equal(lse[: i + 1], lse2[: i + 1])
    assert not np.array_equal(out[i + 1:], out2[i + 1:])


def test_decode_equals_last_prefill_row():
    n = 45
    pre = W.prefill_case("p", 13, [n], [n], block_size=16, num_blocks=4, blocks_per_seq=3)
    kc, vc = _filled_cache(pre, [pre.step.new])
    out_p, lse_p = oracle.prefill(pre.step.q, kc, vc, pre.step.cu_seqlens_q,
                                  pre.step.cu_seqlens_k, pre.block_tables, pre.scale)
    out_d, lse_d = oracle.decode(pre.step.q[n - 1:n], kc, vc, pre.block_tables,
                                 np.array([n], np.int32), pre.scale)
    assert np.array_equal(out_d[0], out_p[n - 1]) and np.array_equal(lse_d[0], lse_p[n - 1])


# ---------------------------------------------------------------- sliding window
# (the SWA-256 serving target of the nano-vllm-sansho README, "Sansho Fork";
# reading: a query at position i sees keys i - window < p <= i)

@pytest.mark.parametrize("window", [1, 37, 256, 700])
def test_windowed_decode_matches_banded_library_attention(window):
    case = W.ragged256_decode()
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    out, lse = oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale,
                             window=window)
    for s in range(case.num_seqs):
        n = int(st.context_lens[s])
        k, v = logical_kv(_stores(case), s, n)
        ref_out, ref_lse = sdpa_rows(st.q[s:s + 1], k, v, case.scale, [n], [max(0, n - window)])
        np.testing.assert_allclose(out[s], ref_out[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[s], ref_lse[0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [1, 16, 100])
def test_windowed_prefill_matches_banded_library_attention(window):
    case = W.prefill_case("prefix-window", 7, q_lens=[12, 0, 30, 19], k_lens=[12, 5, 50, 64],
                          block_size=16, num_blocks=40, blocks_per_seq=6)
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    out, lse = oracle.prefill(st.q, kc, vc, st.cu_seqlens_q, st.cu_seqlens_k, case.block_tables,
                              case.scale, window=window)
    for s in range(case.num_seqs):
        q0, q1 = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        Lq, Lk = q1 - q0, int(st.cu_seqlens_k[s + 1] - st.cu_seqlens_k[s])
        if Lq == 0:
            continue
        k, v = logical_kv(_stores(case), s, Lk)
        hi = [Lk - Lq + i + 1 for i in range(Lq)]
        lo = [max(0, n - window) for n in hi]
        ref_out, ref_lse = sdpa_rows(st.q[q0:q1], k, v, case.scale, hi, lo)
        np.testing.assert_allclose(out[q0:q1], ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[q0:q1], ref_lse, rtol=0, atol=1e-12)


def test_window_covering_every_key_changes_nothing():
    case = W.ragged256_decode()
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    full = oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale)
    wide = oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale,
                         window=int(st.context_lens.max()))
    assert np.array_equal(full[0], wide[0]) and np.array_equal(full[1], wide[1])
    pre = W.ragged256_prefill()
    kc, vc = _filled_cache(pre, [pre.step.new])
    ps = pre.step
    a = oracle.prefill(ps.q, kc, vc, ps.cu_seqlens_q, ps.cu_seqlens_k, pre.block_tables, pre.scale)
    b = oracle.prefill(ps.q, kc, vc, ps.cu_seqlens_q, ps.cu_seqlens_k, pre.block_tables, pre.scale,
                       window=ps.max_seqlen_k)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_window_of_one_returns_the_own_value_and_logit():
    case = W.tiny_decode()
    kc, vc = _filled_cache(case, [case.step.new])
    st = case.step
    out, lse = oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale, window=1)
    G = case.H_q // case.H_kv
    for s in range(case.num_seqs):
        n = int(st.context_lens[s])
        k, v = logical_kv(_stores(case), s, n)
        for h in range(case.H_q):
            kk = bf16_bits_to_f64(k[n - 1, h // G]).numpy()
            vv = bf16_bits_to_f64(v[n - 1, h // G]).numpy()
            qq = bf16_bits_to_f64(st.q[s, h]).numpy()
            assert np.array_equal(out[s, h], vv)
            assert lse[s, h] == pytest.approx(case.scale * float(np.dot(qq, kk)), abs=1e-12)


def test_windowed_row_ignores_keys_before_its_window():
    window, n = 20, 45
    case = W.prefill_case("win-causal", 11, q_lens=[n], k_lens=[n], block_size=16,
                          num_blocks=3, blocks_per_seq=3)
    run = lambda c: oracle.prefill(c.step.q, *_filled_cache(c, [c.step.new]),
                                   c.step.cu_seqlens_q, c.step.cu_seqlens_k, c.block_tables,
                                   c.scale, window=window)
    out, lse = run(case)
    # perturb every key/value before position 10: rows i >= 29 see keys >= 10 only
    sel = case.step.new.positions < 10
    case.step.new.k[sel] ^= np.uint16(0x1234)
    case.step.new.v[sel] ^= np.uint16(0x0F0F)
    out2, lse2 = run(case)
    assert np.array_equal(out[29:], out2[29:]) and np.array_equal(lse[29:], lse2[29:])
    assert not np.array_equal(out[:29], out2[:29])


def test_windowed_decode_equals_last_windowed_prefill_row():
    n, window = 45, 19
    pre = W.prefill_case("pw", 13, [n], [n], block_size=16, num_blocks=4, blocks_per_seq=3)
    kc, vc = _filled_cache(pre, [pre.step.new])
    out_p, lse_p = oracle.prefill(pre.step.q, kc, vc, pre.step.cu_seqlens_q,
                                  pre.step.cu_seqlens_k, pre.block_tables, pre.scale,
                                  window=window)
    out_d, lse_d = oracle.decode(pre.step.q[n - 1:n], kc, vc, pre.block_tables,
                                 np.array([n], np.int32), pre.scale, window=window)
    assert np.array_equal(out_d[0], out_p[n - 1]) and np.array_equal(lse_d[0], lse_p[n - 1])


def test_attend_rows_matches_full_decode():
    case = W.tiny_decode()
    out, lse = _run_decode(case)
    kc, vc = _filled_cache(case, [case.step.new])
    seqs = np.array([0, 2, 3, 1], np.int32)
    heads = np.array([0, 5, 15, 8], np.int32)
    nk = case.step.context_lens[seqs].astype(np.int64)
    o, l = oracle.attend_rows(case.step.q[seqs, heads], seqs, heads, nk, kc, vc,
                              case.block_tables, case.H_q, case.scale)
    assert np.array_equal(o, out[seqs, heads]) and np.array_equal(l, lse[seqs, heads])


def test_decode_rejects_bad_block_and_empty_context():
    case = W.tiny_decode()
    kc, vc = _filled_cache(case, [case.step.new])
    bt = case.block_tables.copy()
    bt[0, 0] = case.num_blocks  # outside the pool
    with pytest.raises(oracle.OracleError):
        oracle.decode(case.step.q, kc, vc, bt, case.step.context_lens, case.scale)
    ctx = case.step.context_lens.copy()
    ctx[1] = 0
    with pytest.raises(oracle.OracleError):
        oracle.decode(case.step.q, kc, vc, case.block_tables, ctx, case.scale)


def test_generator_is_deterministic():
    a, b = W.ragged256_decode(), W.ragged256_decode()
    assert np.array_equal(a.step.q, b.step.q) and np.array_equal(a.history.k, b.history.k)
    assert np.array_equal(a.block_tables, b.block_tables)
    c = W.ragged256_decode(seed=999)
    assert not np.array_equal(a.step.q, c.step.q)


def test_outlier_rows_are_scaled_by_eight():
    case = W.ragged256_decode()
    k = np.concatenate([case.history.k, case.step.new.k])
    kf = bf16_bits_to_f64(k).abs().amax(dim=(1, 2)).numpy()
    n_out = int(round(0.05 * k.shape[0]))
    # N(0,1) rows of 1024 values rarely exceed |x| = 5.5; scaled rows nearly always do
    assert abs(int((kf > 9.0).sum()) - n_out) <= max(3, n_out // 50)
