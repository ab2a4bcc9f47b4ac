"""The allocation-free decode entry point, through the C ABI.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device
memory (a plugin inside a framework that owns the device pool, a deployment
that forbids allocation after start-up, a latency-critical loop): its scratch
is a static device array inside libpkv.so instead of a caller workspace. It
must give the same result as pkv_paged_decode_attn (and stay within the stated
tolerance of the fp64 oracle), also on a second call enqueued right behind a
first one of a different size, since every call shares that array, and it must
allocate no device memory.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_22_gb300 as pkv
import workloads as W
from paged_kv_attention_22_gb300 import build as pkv_build
from runners import (OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS, dev_bf16, dev_i32, gpu_pool, gpu_store,
                     oracle_run)

pytestmark = pytest.mark.gpu


def _noalloc(L, case, q, kc, vc, bt, ctx, out, lse):
    P = ctypes.c_void_p
    st = case.step
    return L.pkv_paged_decode_attn_noalloc(
        P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), P(bt.data_ptr()), bt.shape[1],
        P(ctx.data_ptr()), st.max_context_len, q.shape[0], case.H_q, case.H_kv, case.D,
        case.block_size, case.num_blocks, ctypes.c_float(case.scale), 0, P(out.data_ptr()),
        P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))


def _prepared(case):
    """Device inputs of a decode case, its cache filled (history and new token)."""
    kc, vc = gpu_pool(case)
    gpu_store(case.history, kc, vc)
    gpu_store(case.step.new, kc, vc)
    st = case.step
    return dict(q=dev_bf16(st.q), kc=kc, vc=vc, bt=dev_i32(case.block_tables),
                ctx=dev_i32(st.context_lens))


def _close(out, lse, ref_out, ref_lse, what):
    a, b = out.double().cpu().numpy(), np.asarray(ref_out, dtype=np.float64)
    err = np.abs(a - b)
    assert np.all(np.isfinite(a)), what
    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, what
    assert np.abs(lse.double().cpu().numpy() - np.asarray(ref_lse)).max() <= LSE_MAX_ABS, what


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    pkv_build.build()
    L = pkv.lib()
    pkv.decode_set_config(0, 0)
    pkv.set_programmatic_launch(True)
    cases = (W.ragged256_decode(), W.tiny_decode())
    dev = [_prepared(c) for c in cases]
    refs = []
    for case, d in zip(cases, dev):
        st = case.step
        refs.append(pkv.paged_decode_attn(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"],
                                          st.max_context_len, case.scale))
    outs = [(torch.full_like(d["q"], float("nan")),
             torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda"))
            for d in dev]
    # a first call sets up the scratch address and loads the kernels
    warm_out, warm_lse = torch.empty_like(dev[1]["q"]), torch.empty_like(outs[1][1])
    assert _noalloc(L, cases[1], dev[1]["q"], dev[1]["kc"], dev[1]["vc"], dev[1]["bt"],
                    dev[1]["ctx"], warm_out, warm_lse) == pkv.PKV_OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    allocated_before = torch.cuda.memory_allocated()
    # two calls of different sizes back to back on one stream, with no host
    # synchronisation between them: the second one's decode kernel may start
    # while the first one's merge still reads the shared scratch
    for case, d, (out, lse) in zip(cases, dev, outs):
        assert _noalloc(L, case, d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], out, lse) == \
            pkv.PKV_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == allocated_before
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory was allocated"
    assert pkv.check_device_errors() == 0
    for case, (out, lse), (ref_out, ref_lse) in zip(cases, outs, refs):
        # the same result as the workspace entry point, and within the stated
        # tolerance of the fp64 oracle
        _close(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
               case.name + " vs workspace entry point")
        ref = oracle_run(case)
        _close(out, lse, ref["out"], ref["lse"], case.name + " vs oracle")


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
