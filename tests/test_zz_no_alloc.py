"""The allocation-free decode entry point, through the C ABI.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device
memory (a plugin inside a framework that owns the device pool, a deployment
that forbids allocation after start-up, a latency-critical loop): its scratch
is a static device array inside libpkv.so instead of a caller workspace. It
must give the same result as pkv_paged_decode_attn, also on a second call right
after a first one of a different size, since every call shares that array.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_22_gb300 as pkv
import workloads as W
from paged_kv_attention_22_gb300 import build as pkv_build
from runners import OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS, dev_bf16, dev_i32, gpu_pool, gpu_store

pytestmark = pytest.mark.gpu


def _noalloc(L, case, q, kc, vc, bt, ctx, out, lse):
    P = ctypes.c_void_p
    st = case.step
    return L.pkv_paged_decode_attn_noalloc(
        P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), P(bt.data_ptr()), bt.shape[1],
        P(ctx.data_ptr()), st.max_context_len, q.shape[0], case.H_q, case.H_kv, case.D,
        case.block_size, case.num_blocks, ctypes.c_float(case.scale), 0, P(out.data_ptr()),
        P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    pkv_build.build()
    L = pkv.lib()
    pkv.decode_set_config(0, 0)
    # two calls in a row with different sizes: the second reuses the scratch
    for case in (W.ragged256_decode(), W.tiny_decode()):
        kc, vc = gpu_pool(case)
        gpu_store(case.history, kc, vc)
        gpu_store(case.step.new, kc, vc)
        q, bt, ctx = dev_bf16(case.step.q), dev_i32(case.block_tables), dev_i32(case.step.context_lens)
        ref_out, ref_lse = pkv.paged_decode_attn(q, kc, vc, bt, ctx, case.step.max_context_len,
                                                 case.scale)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(L, case, q, kc, vc, bt, ctx, out, lse) == pkv.PKV_OK
        assert pkv.check_device_errors() == 0
        a, b = out.double().cpu().numpy(), ref_out.double().cpu().numpy()
        err = np.abs(a - b)
        assert np.all(np.isfinite(a))
        assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, case.name
        assert np.abs(lse.double().cpu().numpy() - ref_lse.double().cpu().numpy()).max() <= LSE_MAX_ABS


def test_noalloc_rejects_sizes_beyond_its_scratch():
    pkv_build.build()
    L = pkv.lib()
    case = W.tiny_decode()
    kc, vc = gpu_pool(case)
    q, bt, ctx = dev_bf16(case.step.q), dev_i32(case.block_tables), dev_i32(case.step.context_lens)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    # a 4000-CTA grid needs more partial-result slots than the static scratch holds
    pkv.decode_set_config(4000, 0)
    try:
        assert pkv.decode_workspace_size(q.shape[0], case.H_q, case.H_kv, case.D,
                                         case.step.max_context_len) > \
            pkv.DECODE_NOALLOC_SCRATCH_BYTES
        rc = _noalloc(L, case, q, kc, vc, bt, ctx, out, lse)
    finally:
        pkv.decode_set_config(0, 0)
    assert rc == pkv.PKV_ERR_WORKSPACE_TOO_SMALL
