"""fp64 CPU oracle for paged-KV-cache attention (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA library (``paged_kv_attention_22_gb300``) and never imports it.

Every function takes numpy arrays: bf16 data as ``uint16`` bit patterns,
indices as ``int32``. Results are float64. Each function follows the plain
definition written at the top of ``oracle.c`` (slot mapping, KV store, softmax
attention over keys gathered through block tables).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIBRARY) or (
            os.path.getmtime(_build.LIBRARY) < os.path.getmtime(_build.SOURCE)):
        _build.build()
    lib = ctypes.CDLL(_build.LIBRARY)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_slot_mapping.argtypes = [P, i32, i32, P, P, i64, i32, P]
    lib.oracle_kv_store.argtypes = [P, P, P, P, P, i64, i64, i64]
    lib.oracle_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                  i64, f64, i32, P, P]
    lib.oracle_prefill.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                   i32, i64, f64, i32, P, P]
    lib.oracle_attend_rows.argtypes = [P, P, P, P, i64, P, P, P, i32, i32, i32,
                                       i32, i32, i64, f64, i32, P, P]
    for name in ("oracle_slot_mapping", "oracle_kv_store", "oracle_decode",
                 "oracle_prefill", "oracle_attend_rows"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def slot_mapping(block_tables, seq_of_token, pos_of_token, block_size):
    """Cache slot of every (sequence, position) pair; -1 where the table has no block."""
    bt = _c(block_tables, np.int32)
    seq = _c(seq_of_token, np.int32)
    pos = _c(pos_of_token, np.int32)
    out = np.empty(seq.shape[0], np.int32)
    _check(_load().oracle_slot_mapping(_ptr(bt), bt.shape[1], bt.shape[0],
                                       _ptr(seq), _ptr(pos), seq.shape[0],
                                       int(block_size), _ptr(out)),
           "slot_mapping")
    return out


def kv_store(k, v, k_cache, v_cache, slot_mapping):
    """Write token rows k, v [T, H_kv, D] into the caches [NB, bs, H_kv, D] in place."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise TypeError("caches must be C-contiguous uint16 arrays")
    row = int(np.prod(k.shape[1:]))
    slots = k_cache.shape[0] * k_cache.shape[1]
    _check(_load().oracle_kv_store(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(sm), k.shape[0], row, slots), "kv_store")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, window=0):
    """Decode attention: q [S, H_q, D] -> (out [S, H_q, D], lse [S, H_q]) in float64.
    window > 0: each query sees only the last `window` keys up to itself."""
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    out = np.empty((S, H_q, D), np.float64)
    lse = np.empty((S, H_q), np.float64)
    _check(_load().oracle_decode(_ptr(q), _ptr(_c(k_cache, np.uint16)),
                                 _ptr(_c(v_cache, np.uint16)), _ptr(bt), bt.shape[1],
                                 _ptr(cl), S, H_q, H_kv, D, bs, NB, float(scale),
                                 int(window), _ptr(out), _ptr(lse)), "decode")
    return out, lse


def prefill(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale, window=0):
    """Varlen causal prefill: q [T_q, H_q, D] -> (out [T_q, H_q, D], lse [T_q, H_q]).
    window > 0: each query sees only the last `window` keys up to itself."""
    q = _c(q, np.uint16)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    bt = _c(block_tables, np.int32)
    T, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    out = np.zeros((T, H_q, D), np.float64)
    lse = np.zeros((T, H_q), np.float64)
    _check(_load().oracle_prefill(_ptr(q), _ptr(_c(k_cache, np.uint16)),
                                  _ptr(_c(v_cache, np.uint16)), _ptr(cq), _ptr(ck),
                                  _ptr(bt), bt.shape[1], cq.shape[0] - 1, H_q, H_kv,
                                  D, bs, NB, float(scale), int(window), _ptr(out),
                                  _ptr(lse)),
           "prefill")
    return out, lse


def attend_rows(q_rows, seq_ids, head_ids, n_keys, k_cache, v_cache, block_tables,
                num_q_heads, scale, window=0):
    """Attention of sampled rows: row r is query q_rows[r] (head head_ids[r] of
    sequence seq_ids[r]) over that sequence's first n_keys[r] cached keys (the
    last `window` of them if window > 0)."""
    q_rows = _c(q_rows, np.uint16)
    sid = _c(seq_ids, np.int32)
    hid = _c(head_ids, np.int32)
    nk = _c(n_keys, np.int64)
    bt = _c(block_tables, np.int32)
    R, D = q_rows.shape
    NB, bs, H_kv, _ = k_cache.shape
    out = np.empty((R, D), np.float64)
    lse = np.empty(R, np.float64)
    _check(_load().oracle_attend_rows(_ptr(q_rows), _ptr(sid), _ptr(hid), _ptr(nk), R,
                                      _ptr(_c(k_cache, np.uint16)),
                                      _ptr(_c(v_cache, np.uint16)), _ptr(bt),
                                      bt.shape[1], int(num_q_heads), H_kv, D, bs, NB,
                                      float(scale), int(window), _ptr(out), _ptr(lse)),
           "attend_rows")
    return out, lse
