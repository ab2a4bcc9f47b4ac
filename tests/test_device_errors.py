"""Device error words: the non-blocking readout and the skip that a timeout
starts, tested with a host-side injection of the timeout bit (no kernel is made
to wait or fault).

After PKV_DEVERR_TIMEOUT every decode and prefill call returns PKV_OK but does
nothing until pkv_check_device_errors clears the words; a caller that never
synchronises learns of it through pkv_read_device_errors_async."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_22_gb300 as pkv
import workloads as W
from paged_kv_attention_22_gb300 import build as pkv_build
from runners import (assert_cache_equal, assert_close, dev_bf16, dev_i32, gpu_pool, gpu_store,
                     host_u16, oracle_run)


@pytest.fixture(scope="module")
def L():
    pkv_build.build()
    return pkv.lib()


def test_readout_and_raise_reject_bad_arguments(L):
    # checked before any device access, so this holds with or without a GPU
    assert L.pkv_read_device_errors_async(None, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_raise_device_errors(0x100, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_raise_device_errors(pkv.DEVERR_TIMEOUT | 0x40, None) == pkv.PKV_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_raise_without_gpu_reports_cuda_error(L):
    assert L.pkv_raise_device_errors(pkv.DEVERR_TIMEOUT, None) == pkv.PKV_ERR_CUDA


def _readout(stream=None):
    word = torch.zeros(1, dtype=torch.int32).pin_memory()
    pkv.read_device_errors_async(word, stream)
    torch.cuda.current_stream().synchronize()
    return int(word[0])


@pytest.mark.gpu
def test_readout_needs_page_locked_memory(L):
    pageable = (ctypes.c_uint32 * 4)()
    assert L.pkv_read_device_errors_async(ctypes.cast(pageable, ctypes.c_void_p), None) == \
        pkv.PKV_ERR_INVALID_ARG
    # the argument error leaves no runtime error behind: a valid readout works
    assert pkv.check_device_errors() == 0
    assert _readout() == 0


@pytest.mark.gpu
def test_timeout_makes_later_calls_skip_until_cleared(L):
    pkv.decode_set_config(0, 0)
    assert pkv.check_device_errors() == 0
    dec = W.tiny_decode()
    pre = W.tiny_prefill()
    ref_dec, ref_pre = oracle_run(dec), oracle_run(pre)

    # decode case: history in the cache, the new token left to the fused call
    kc, vc = gpu_pool(dec)
    gpu_store(dec.history, kc, vc)
    st = dec.step
    q, bt, ctx = dev_bf16(st.q), dev_i32(dec.block_tables), dev_i32(st.context_lens)
    kn, vn, slots = dev_bf16(st.new.k), dev_bf16(st.new.v), dev_i32(st.new.slots)
    # prefill case: its prompt already in the cache
    pkc, pvc = gpu_pool(pre)
    gpu_store(pre.step.new, pkc, pvc)
    ps = pre.step
    pq, cq, ck, pbt = dev_bf16(ps.q), dev_i32(ps.cu_seqlens_q), dev_i32(ps.cu_seqlens_k), \
        dev_i32(pre.block_tables)
    torch.cuda.synchronize()
    cache_before = (host_u16(kc), host_u16(vc))

    pkv.raise_device_errors(pkv.DEVERR_TIMEOUT)
    nan = float("nan")
    o1 = torch.full_like(q, nan)
    l1 = torch.full((q.shape[0], q.shape[1]), nan, device="cuda")
    o2, l2 = torch.full_like(q, nan), torch.full_like(l1, nan)
    o3 = torch.full_like(pq, nan)
    l3 = torch.full((pq.shape[0], pq.shape[1]), nan, device="cuda")
    ws = pkv.new_decode_workspace(q.shape[0], dec.H_q, dec.H_kv, dec.D, st.max_context_len)
    pkv.paged_decode_attn_store(kn, vn, slots, q, kc, vc, bt, ctx, st.max_context_len, dec.scale,
                                out=o1, lse=l1, workspace=ws)
    pkv.paged_decode_attn(q, kc, vc, bt, ctx, st.max_context_len, dec.scale, out=o2, lse=l2,
                          workspace=ws)
    pkv.paged_prefill_attn(pq, pkc, pvc, cq, ck, pbt, ps.max_seqlen_q, ps.max_seqlen_k, pre.scale,
                           out=o3, lse=l3)
    # the caller learns of the timeout without a blocking call of the library
    assert _readout() & pkv.DEVERR_TIMEOUT
    for t in (o1, l1, o2, l2, o3, l3):
        assert torch.isnan(t.float()).all(), "a call wrote output after the timeout"
    assert np.array_equal(host_u16(kc), cache_before[0]) and \
        np.array_equal(host_u16(vc), cache_before[1]), "the fused store ran after the timeout"
    # the words stay set until cleared: the readout clears nothing
    assert _readout() & pkv.DEVERR_TIMEOUT
    assert pkv.check_device_errors() & pkv.DEVERR_TIMEOUT
    assert _readout() == 0

    # cleared: the same calls compute again
    out, lse = pkv.paged_decode_attn_store(kn, vn, slots, q, kc, vc, bt, ctx, st.max_context_len,
                                           dec.scale, workspace=ws)
    pout, plse = pkv.paged_prefill_attn(pq, pkc, pvc, cq, ck, pbt, ps.max_seqlen_q,
                                        ps.max_seqlen_k, pre.scale)
    assert pkv.check_device_errors() == 0
    assert_cache_equal(kc, vc, ref_dec["kc"], ref_dec["vc"])
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_dec["out"],
                 ref_dec["lse"], "decode after clearing")
    assert_close(pout.double().cpu().numpy(), plse.double().cpu().numpy(), ref_pre["out"],
                 ref_pre["lse"], "prefill after clearing")


@pytest.mark.gpu
def test_readout_reports_a_device_side_error(L):
    # an out-of-pool slot is a device-side error the kernel itself raises
    case = W.tiny_decode()
    kc, vc = gpu_pool(case)
    k, v = dev_bf16(case.step.new.k), dev_bf16(case.step.new.v)
    bad = torch.full((k.shape[0],), case.num_blocks * case.block_size, dtype=torch.int32,
                     device="cuda")
    pkv.kv_store(k, v, kc, vc, bad)
    assert _readout() == pkv.DEVERR_SLOT
    assert pkv.check_device_errors() == pkv.DEVERR_SLOT
    assert _readout() == 0
