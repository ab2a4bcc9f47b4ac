"""Run a workload case through the CUDA library and through the fp64 oracle on
the same seeded inputs, and compare with the stated tolerances."""
import numpy as np
import torch

import oracle
import paged_kv_attention_22_gb300 as pkv
import workloads as W

# bf16 output against the fp64 oracle, per call; fp32 lse in natural-log units
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_pool(case):
    return dev_bf16(case.poisoned_pool()), dev_bf16(case.poisoned_pool())


def gpu_store(st: W.Store, kc, vc):
    pkv.kv_store(dev_bf16(st.k), dev_bf16(st.v), kc, vc, dev_i32(st.slots))


def gpu_attend(case, kc, vc):
    st = case.step
    bt = dev_i32(case.block_tables)
    if isinstance(st, W.DecodeStep):
        out, lse = pkv.paged_decode_attn(dev_bf16(st.q), kc, vc, bt, dev_i32(st.context_lens),
                                         st.max_context_len, case.scale)
    else:
        out, lse = pkv.paged_prefill_attn(dev_bf16(st.q), kc, vc, dev_i32(st.cu_seqlens_q),
                                          dev_i32(st.cu_seqlens_k), bt, st.max_seqlen_q,
                                          st.max_seqlen_k, case.scale)
    return out, lse


def gpu_run(case, kc=None, vc=None, store_history=True):
    """History store (unless the cache already holds it), the step's store, then
    attention. Returns dict with device caches and host float64 results."""
    if kc is None:
        kc, vc = gpu_pool(case)
    if store_history and case.history is not None:
        gpu_store(case.history, kc, vc)
    gpu_store(case.step.new, kc, vc)
    out, lse = gpu_attend(case, kc, vc)
    flags = pkv.check_device_errors()
    return dict(kc=kc, vc=vc, out=out.double().cpu().numpy(), lse=lse.double().cpu().numpy(),
                flags=flags)


def oracle_cache(case):
    kc, vc = case.poisoned_pool(), case.poisoned_pool()
    if case.history is not None:
        oracle.kv_store(case.history.k, case.history.v, kc, vc, case.history.slots)
    oracle.kv_store(case.step.new.k, case.step.new.v, kc, vc, case.step.new.slots)
    return kc, vc


def oracle_run(case, kc=None, vc=None):
    if kc is None:
        kc, vc = oracle_cache(case)
    st = case.step
    if isinstance(st, W.DecodeStep):
        out, lse = oracle.decode(st.q, kc, vc, case.block_tables, st.context_lens, case.scale)
    else:
        out, lse = oracle.prefill(st.q, kc, vc, st.cu_seqlens_q, st.cu_seqlens_k,
                                  case.block_tables, case.scale)
    return dict(kc=kc, vc=vc, out=out, lse=lse)


def assert_close(out, lse, ref_out, ref_lse, what=""):
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    max_abs, mean_abs = float(err.max()), float(err.mean())
    lse_err = float(np.abs(lse - ref_lse).max())
    assert max_abs <= OUT_MAX_ABS, f"{what}: max abs error {max_abs:.3e} > {OUT_MAX_ABS}"
    assert mean_abs <= OUT_MEAN_ABS, f"{what}: mean abs error {mean_abs:.3e} > {OUT_MEAN_ABS}"
    assert lse_err <= LSE_MAX_ABS, f"{what}: lse error {lse_err:.3e} > {LSE_MAX_ABS}"
    return max_abs, mean_abs, lse_err


def assert_cache_equal(gpu_kc, gpu_vc, ref_kc, ref_vc):
    assert np.array_equal(host_u16(gpu_kc), ref_kc), "k_cache bytes differ from the oracle"
    assert np.array_equal(host_u16(gpu_vc), ref_vc), "v_cache bytes differ from the oracle"


def sampled_rows_reference(case, kc, vc, rows):
    """Oracle attention for selected output rows of a case: rows is a list of
    (token_or_seq, head). For prefill, token is a global query row."""
    st = case.step
    seqs, heads, nk, qs = [], [], [], []
    for r, h in rows:
        if isinstance(st, W.DecodeStep):
            s, n = r, int(st.context_lens[r])
        else:
            s = int(np.searchsorted(st.cu_seqlens_q, r, side="right") - 1)
            Lq = int(st.cu_seqlens_q[s + 1] - st.cu_seqlens_q[s])
            Lk = int(st.cu_seqlens_k[s + 1] - st.cu_seqlens_k[s])
            n = Lk - Lq + (r - int(st.cu_seqlens_q[s])) + 1
        seqs.append(s)
        heads.append(h)
        nk.append(n)
        qs.append(st.q[r, h])
    return oracle.attend_rows(np.stack(qs), np.array(seqs, np.int32), np.array(heads, np.int32),
                              np.array(nk, np.int64), kc, vc, case.block_tables, case.H_q,
                              case.scale)
