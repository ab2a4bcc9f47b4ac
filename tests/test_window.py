"""Sliding-window attention on the GPU against the windowed fp64 oracle (a
query at position i sees keys i - W < p <= i; W = 0: no window), through the
C ABI: decode (plain, fused store, other launch shapes, no-workspace), prefill
(with a cached prefix, empty segments, both CTA layouts) and the full-size
prefix workload."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_22_gb300 as pkv
import workloads as W
from runners import (assert_cache_equal, assert_close, dev_bf16, dev_i32, gpu_pool, gpu_store,
                     oracle_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_knobs():
    pkv.decode_set_config(0, 0)
    yield
    pkv.decode_set_config(0, 0)


def _filled(case):
    kc, vc = gpu_pool(case)
    if case.history is not None:
        gpu_store(case.history, kc, vc)
    gpu_store(case.step.new, kc, vc)
    return kc, vc


def _host(o, l):
    return o.double().cpu().numpy(), l.double().cpu().numpy()


def _check_decode(case, window, what=""):
    st = case.step
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.decode(st.q, ref_kc, ref_vc, case.block_tables, st.context_lens, case.scale,
                        window=window)
    kc, vc = _filled(case)
    o, l = pkv.paged_decode_attn(dev_bf16(st.q), kc, vc, dev_i32(case.block_tables),
                                 dev_i32(st.context_lens), st.max_context_len, case.scale,
                                 sliding_window=window)
    assert pkv.check_device_errors() == 0
    assert_close(*_host(o, l), *ref, what=f"{case.name} window {window} {what}")


def _check_prefill(case, window):
    st = case.step
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.prefill(st.q, ref_kc, ref_vc, st.cu_seqlens_q, st.cu_seqlens_k,
                         case.block_tables, case.scale, window=window)
    kc, vc = _filled(case)
    o, l = pkv.paged_prefill_attn(dev_bf16(st.q), kc, vc, dev_i32(st.cu_seqlens_q),
                                  dev_i32(st.cu_seqlens_k), dev_i32(case.block_tables),
                                  st.max_seqlen_q, st.max_seqlen_k, case.scale,
                                  sliding_window=window)
    assert pkv.check_device_errors() == 0
    o, l = _host(o, l)
    rows = np.zeros(st.q.shape[0], bool)   # rows of empty segments are not written
    for s in range(len(st.cu_seqlens_q) - 1):
        rows[st.cu_seqlens_q[s]:st.cu_seqlens_q[s + 1]] = True
    assert_close(o[rows], l[rows], ref[0][rows], ref[1][rows],
                 what=f"{case.name} window {window}")


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 256, 1023, 2000])
def test_windowed_decode(window):
    _check_decode(W.ragged256_decode(), window)


def test_windowed_decode_tiny_and_small_blocks():
    for window in (1, 5, 16, 40):
        _check_decode(W.tiny_decode(), window)


@pytest.mark.parametrize("ctas,variant", [(1, 0), (7, 0), (1000, 0), (0, 1), (0, 2), (5, 2)])
def test_windowed_decode_launch_shapes(ctas, variant):
    pkv.decode_set_config(ctas, variant)
    _check_decode(W.ragged256_decode(), 100, what=f"ctas {ctas} variant {variant}")


def test_windowed_fused_store_decode():
    case = W.ragged256_decode()
    st = case.step
    window = 37
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.decode(st.q, ref_kc, ref_vc, case.block_tables, st.context_lens, case.scale,
                        window=window)
    kc, vc = gpu_pool(case)
    gpu_store(case.history, kc, vc)
    o, l = pkv.paged_decode_attn_store(dev_bf16(st.new.k), dev_bf16(st.new.v),
                                       dev_i32(st.new.slots), dev_bf16(st.q), kc, vc,
                                       dev_i32(case.block_tables), dev_i32(st.context_lens),
                                       st.max_context_len, case.scale, sliding_window=window)
    assert pkv.check_device_errors() == 0
    assert_cache_equal(kc, vc, ref_kc, ref_vc)
    assert_close(*_host(o, l), *ref, what="fused store, window 37")


def test_windowed_noalloc_decode():
    case = W.ragged256_decode()
    st = case.step
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.decode(st.q, ref_kc, ref_vc, case.block_tables, st.context_lens, case.scale,
                        window=64)
    kc, vc = _filled(case)
    q = dev_bf16(st.q)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    pkv.paged_decode_attn_noalloc(q, kc, vc, dev_i32(case.block_tables), dev_i32(st.context_lens),
                                  st.max_context_len, case.scale, out, lse, sliding_window=64)
    assert pkv.check_device_errors() == 0
    assert_close(*_host(out, lse), *ref, what="no-workspace decode, window 64")


@pytest.mark.parametrize("window", [1, 64, 100, 128, 129, 256, 600])
def test_windowed_prefill(window):
    _check_prefill(W.ragged256_prefill(), window)


def test_windowed_prefill_with_prefix_and_empty_segment():
    case = W.prefill_case("prefix-window", 7, q_lens=[12, 0, 30, 19], k_lens=[12, 5, 50, 64],
                          block_size=16, num_blocks=40, blocks_per_seq=6)
    for window in (1, 16, 100):
        _check_prefill(case, window)


def test_windowed_prefill_one_query_head_per_kv_head():
    # without grouping a CTA holds two different row tiles, with different windows
    case = W.prefill_case("pwin-g1", 34, [300, 7], [420, 7], block_size=64, num_blocks=16,
                          blocks_per_seq=8, H_q=8, H_kv=8)
    for window in (50, 200):
        _check_prefill(case, window)


def test_windowed_prefill_four_query_heads_per_kv_head():
    # a KV head serving four query heads: an item holds two of them, and the
    # other two of the same KV head form another item over the same rows
    case = W.prefill_case("pwin-g4", 37, [300, 7, 130], [420, 7, 130], block_size=64,
                          num_blocks=24, blocks_per_seq=8, H_q=32, H_kv=8)
    for window in (1, 64, 200):
        _check_prefill(case, window)


def test_windowed_decode_four_query_heads_per_kv_head():
    case = W.decode_case("dwin-g4", 38, [77, 300, 1, 160], block_size=32, num_blocks=40,
                         blocks_per_seq=10, H_q=32, H_kv=8)
    for window in (1, 40, 200):
        _check_decode(case, window, what="4 query heads per KV head")


def test_windowed_prefix8k_prefill_full():
    # the full-size prefix workload with the SWA-256 window: every output
    # element and every lse against the windowed fp64 oracle
    pre, _ = W.prefix8k()
    _check_prefill(pre, 256)


def test_windowed_prefix8k_decode_and_sampled_prefill_rows():
    pre, dec = W.prefix8k()
    window = 256
    _check_decode(dec, window, what="prefix8k")
    st = pre.step
    kc, vc = _filled(pre)
    o, l = pkv.paged_prefill_attn(dev_bf16(st.q), kc, vc, dev_i32(st.cu_seqlens_q),
                                  dev_i32(st.cu_seqlens_k), dev_i32(pre.block_tables),
                                  st.max_seqlen_q, st.max_seqlen_k, pre.scale,
                                  sliding_window=window)
    assert pkv.check_device_errors() == 0
    o, l = _host(o, l)
    rng = np.random.default_rng(9)
    rows = np.concatenate([rng.integers(0, st.q.shape[0], 200), [0, 4095, 4096, st.q.shape[0] - 1]])
    heads = rng.integers(0, pre.H_q, rows.shape[0])
    seqs = np.searchsorted(st.cu_seqlens_q, rows, side="right") - 1
    Lq = np.diff(st.cu_seqlens_q)[seqs]
    Lk = np.diff(st.cu_seqlens_k)[seqs]
    n_keys = (Lk - Lq + (rows - st.cu_seqlens_q[seqs]) + 1).astype(np.int64)
    ref_kc, ref_vc = oracle_cache(pre)
    ro, rl = oracle.attend_rows(st.q[rows, heads], seqs.astype(np.int32), heads.astype(np.int32),
                                n_keys, ref_kc, ref_vc, pre.block_tables, pre.H_q, pre.scale,
                                window=window)
    assert_close(o[rows, heads], l[rows, heads], ro, rl, what="prefix8k prefill, window 256")
