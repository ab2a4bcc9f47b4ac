"""Every cache block size the kernels take (a multiple of 16), against the fp64
oracle, through the C ABI: prefill with cached prefixes and ragged tails (its
K/V boxes are 16, 32, 64 or 128 rows tall depending on the block size) and a
decode step over the same range of block sizes."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_22_gb300 as pkv
import workloads as W
from runners import assert_close, dev_bf16, dev_i32, gpu_pool, gpu_store, oracle_cache

pytestmark = pytest.mark.gpu

BLOCK_SIZES = [16, 32, 48, 64, 96, 128, 256, 512]


def _filled(case):
    kc, vc = gpu_pool(case)
    if case.history is not None:
        gpu_store(case.history, kc, vc)
    gpu_store(case.step.new, kc, vc)
    return kc, vc


def _pool(block_size, k_lens):
    per_seq = -(-max(k_lens) // block_size) + 1
    return per_seq, per_seq * len(k_lens) + 3


@pytest.mark.parametrize("block_size", BLOCK_SIZES)
@pytest.mark.parametrize("grouped", [True, False])
def test_prefill_block_size(block_size, grouped):
    q_lens, k_lens = [200, 37, 300, 129], [330, 37, 429, 640]
    per_seq, nb = _pool(block_size, k_lens)
    heads = {} if grouped else {"H_q": 8, "H_kv": 8}
    case = W.prefill_case(f"prefill-bs{block_size}", 700 + block_size, q_lens, k_lens,
                          block_size=block_size, num_blocks=nb, blocks_per_seq=per_seq, **heads)
    st = case.step
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.prefill(st.q, ref_kc, ref_vc, st.cu_seqlens_q, st.cu_seqlens_k,
                         case.block_tables, case.scale)
    kc, vc = _filled(case)
    o, l = pkv.paged_prefill_attn(dev_bf16(st.q), kc, vc, dev_i32(st.cu_seqlens_q),
                                  dev_i32(st.cu_seqlens_k), dev_i32(case.block_tables),
                                  st.max_seqlen_q, st.max_seqlen_k, case.scale)
    assert pkv.check_device_errors() == 0
    assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), *ref,
                 what=f"prefill, block size {block_size}, grouped {grouped}")


@pytest.mark.parametrize("block_size", BLOCK_SIZES)
def test_decode_block_size(block_size):
    ctx = [1, 130, 257, 500, 640]
    per_seq, nb = _pool(block_size, ctx)
    case = W.decode_case(f"decode-bs{block_size}", 800 + block_size, ctx, block_size=block_size,
                         num_blocks=nb, blocks_per_seq=per_seq)
    st = case.step
    ref_kc, ref_vc = oracle_cache(case)
    ref = oracle.decode(st.q, ref_kc, ref_vc, case.block_tables, st.context_lens, case.scale)
    kc, vc = _filled(case)
    o, l = pkv.paged_decode_attn(dev_bf16(st.q), kc, vc, dev_i32(case.block_tables),
                                 dev_i32(st.context_lens), st.max_context_len, case.scale)
    assert pkv.check_device_errors() == 0
    assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), *ref,
                 what=f"decode, block size {block_size}")
