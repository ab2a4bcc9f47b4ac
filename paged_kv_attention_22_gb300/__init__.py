"""Paged-KV-cache attention for GB300 (sm_103a): Python binding of libpkv.so.

The functions here have the names of the C entry points in ``include/pkv.h``
and do argument marshalling only: they check dtypes and shapes of torch
tensors, pass their device pointers and the current CUDA stream to the C ABI,
and allocate outputs the caller did not supply. Every step of the computation
runs in the library's CUDA kernels. There is no fallback: if libpkv.so has not
been built, or a call fails, an exception is raised.

Tensors (all CUDA, contiguous):
    k, v           bf16 [T, H_kv, 128]       new K/V rows
    k_cache,v_cache bf16 [num_blocks, block_size, H_kv, 128]
    slot_mapping   int32 [T]
    q              bf16 [S, H_q, 128] (decode) or [T_q, H_q, 128] (prefill)
    block_tables   int32 [S, max_blocks_per_seq], -1 padded
    context_lens   int32 [S]
    cu_seqlens_q/k int32 [S + 1]
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_WORKSPACE_TOO_SMALL = 3
PKV_ERR_CUDA = 4
PKV_ERR_OUT_OF_BLOCKS = 5

DECODE_STABLE_INPUTS = 0x1  # flag of paged_decode_attn_store (PKV_DECODE_STABLE_INPUTS)

DEVERR_SLOT = 0x1
DEVERR_BLOCK = 0x2
DEVERR_CONTEXT = 0x4
DEVERR_SEQLENS = 0x8
DEVERR_TIMEOUT = 0x10

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        name = status_string(status)
        detail = lib().pkv_last_cuda_error().decode() if status == PKV_ERR_CUDA else ""
        super().__init__(f"{what}: {name}" + (f" ({detail})" if detail else ""))


def lib():
    """The loaded libpkv.so (ctypes), with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY_PATH):
        raise ImportError(
            f"{LIBRARY_PATH} is missing: build it with "
            "`python -m paged_kv_attention_22_gb300.build` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIBRARY_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_last_cuda_error.argtypes = []
    L.pkv_last_cuda_error.restype = ctypes.c_char_p
    L.pkv_kv_store.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, P]
    L.pkv_kv_store.restype = ctypes.c_int
    L.pkv_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.pkv_decode_workspace_size.restype = sz
    L.pkv_paged_decode_attn.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64,
                                        f32, i32, P, P, P, sz, P]
    L.pkv_paged_decode_attn.restype = ctypes.c_int
    L.pkv_paged_decode_attn_store.argtypes = [P, P, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                              i32, i32, i64, f32, i32, P, P, P, sz,
                                              ctypes.c_uint32, P]
    L.pkv_paged_decode_attn_store.restype = ctypes.c_int
    L.pkv_paged_decode_attn_noalloc.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                i32, i64, f32, i32, P, P, P]
    L.pkv_paged_decode_attn_noalloc.restype = ctypes.c_int
    L.pkv_set_programmatic_launch.argtypes = [i32]
    L.pkv_set_programmatic_launch.restype = None
    L.pkv_decode_set_config.argtypes = [i32, i32]
    L.pkv_decode_set_config.restype = None
    L.pkv_prefill_workspace_size.argtypes = [i32, i32]
    L.pkv_prefill_workspace_size.restype = sz
    L.pkv_paged_prefill_attn.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                         i32, i32, i64, f32, i32, P, P, P, sz, P]
    L.pkv_paged_prefill_attn.restype = ctypes.c_int
    L.pkv_check_device_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    L.pkv_check_device_errors.restype = ctypes.c_int
    L.pkv_read_device_errors_async.argtypes = [P, P]
    L.pkv_read_device_errors_async.restype = ctypes.c_int
    L.pkv_raise_device_errors.argtypes = [ctypes.c_uint32, P]
    L.pkv_raise_device_errors.restype = ctypes.c_int
    pi32 = ctypes.POINTER(ctypes.c_int32)
    L.pkv_bm_create.argtypes = [i32, i32]
    L.pkv_bm_create.restype = P
    L.pkv_bm_destroy.argtypes = [P]
    L.pkv_bm_destroy.restype = None
    L.pkv_bm_num_free_blocks.argtypes = [P]
    L.pkv_bm_num_free_blocks.restype = i32
    L.pkv_bm_ref_count.argtypes = [P, i32]
    L.pkv_bm_ref_count.restype = i32
    L.pkv_bm_add_sequence.argtypes = [P, i64, P, i32, pi32]
    L.pkv_bm_add_sequence.restype = ctypes.c_int
    L.pkv_bm_append_token.argtypes = [P, i64, i32]
    L.pkv_bm_append_token.restype = ctypes.c_int
    L.pkv_bm_free_sequence.argtypes = [P, i64]
    L.pkv_bm_free_sequence.restype = ctypes.c_int
    L.pkv_bm_num_tokens.argtypes = [P, i64, pi32]
    L.pkv_bm_num_tokens.restype = ctypes.c_int
    L.pkv_bm_block_table.argtypes = [P, i64, P, i32, pi32]
    L.pkv_bm_block_table.restype = ctypes.c_int
    L.pkv_bm_slots.argtypes = [P, i64, i32, i32, P]
    L.pkv_bm_slots.restype = ctypes.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _check(status, what):
    if status != PKV_OK:
        raise PkvError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kv_store(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """Scatter k, v [T, H_kv, D] into the caches at slot_mapping (-1: skip)."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    NB, bs, H_kv, D = k_cache.shape
    if v_cache.shape != k_cache.shape or k.shape != v.shape or k.shape[1:] != (H_kv, D) \
            or slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("inconsistent shapes")
    _check(lib().pkv_kv_store(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                              k.shape[0], H_kv, D, bs, NB, _stream(stream)), "pkv_kv_store")


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len) -> int:
    """Workspace bytes of paged_decode_attn on the current device (0: invalid sizes)."""
    return int(lib().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               max_context_len))


DECODE_NUM_VARIANTS = 3


def new_decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                         device="cuda"):
    """A decode workspace for these sizes on the current device."""
    need = decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len)
    if need == 0:
        raise PkvError(PKV_ERR_CUDA, "pkv_decode_workspace_size")
    return torch.zeros(need, dtype=torch.uint8, device=device)


def set_programmatic_launch(enabled: bool) -> None:
    """Launch kernels with programmatic dependent launch (the default) or not."""
    lib().pkv_set_programmatic_launch(1 if enabled else 0)


def decode_set_config(ctas: int = 0, variant: int = 0) -> None:
    """Tuning knob of the decode launch: persistent CTAs (0 = one per SM) and
    launch-shape variant (0 = default). Process-wide."""
    lib().pkv_decode_set_config(int(ctas), int(variant))


def paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
                      out=None, lse=None, workspace=None, stream=None, with_lse=True,
                      sliding_window=0):
    """q=1 decode attention through block tables (sliding_window > 0: each query
    sees only the last sliding_window keys up to its own). Returns (out, lse)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    S, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and with_lse:
        lse = torch.empty((S, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        workspace = new_decode_workspace(S, H_q, H_kv, D, int(max_context_len), q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    _check(lib().pkv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), S, H_q, H_kv, D, bs, NB, float(scale),
        int(sliding_window), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream)), "pkv_paged_decode_attn")
    return out, lse


def paged_decode_attn_store(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                            context_lens, max_context_len, scale, out=None, lse=None,
                            workspace=None, stream=None, with_lse=True, sliding_window=0,
                            stable_inputs=False):
    """Fused decode step: store each sequence's new K/V row (position
    context_lens[s] - 1, slot slot_mapping[s]) and attend. Returns (out, lse).
    stable_inputs: the caches (but the new rows), block_tables and context_lens
    are not written by the kernels still in flight on the stream, so the call
    may read them before the previous kernel ends (PKV_DECODE_STABLE_INPUTS)."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    S, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    if k_new.shape != (S, H_kv, D) or v_new.shape != k_new.shape or slot_mapping.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and with_lse:
        lse = torch.empty((S, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        workspace = new_decode_workspace(S, H_q, H_kv, D, int(max_context_len), q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    _check(lib().pkv_paged_decode_attn_store(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), int(max_context_len), S,
        H_q, H_kv, D, bs, NB, float(scale), int(sliding_window), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), DECODE_STABLE_INPUTS if stable_inputs else 0,
        _stream(stream)), "pkv_paged_decode_attn_store")
    return out, lse


# Static scratch of paged_decode_attn_noalloc (PKV_DECODE_NOALLOC_SCRATCH_BYTES).
DECODE_NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_decode_attn_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                              scale, out, lse=None, stream=None, sliding_window=0):
    """Decode attention for callers that cannot allocate device memory: same
    result as paged_decode_attn, with the library's static scratch in place of a
    workspace. `out` (and `lse`, if wanted) must be supplied; nothing is
    allocated here either. Calls overlapping on one GPU race on the scratch."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    S, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    _check(lib().pkv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), S, H_q, H_kv, D, bs, NB, float(scale),
        int(sliding_window), _ptr(out), _ptr(lse), _stream(stream)),
        "pkv_paged_decode_attn_noalloc")
    return out, lse


def prefill_workspace_size(num_seqs, max_seqlen_q) -> int:
    return int(lib().pkv_prefill_workspace_size(num_seqs, max_seqlen_q))


def paged_prefill_attn(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables,
                       max_seqlen_q, max_seqlen_k, scale, out=None, lse=None, workspace=None,
                       stream=None, with_lse=True, sliding_window=0):
    """Varlen causal prefill over the paged cache (bottom-right aligned;
    sliding_window > 0: each query sees only the last sliding_window keys up to
    its own). Returns (out, lse)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    T, H_q, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and with_lse:
        lse = torch.empty((T, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    need = prefill_workspace_size(S, int(max_seqlen_q))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib().pkv_paged_prefill_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        _ptr(block_tables), block_tables.shape[1], S, T, int(max_seqlen_q), int(max_seqlen_k),
        H_q, H_kv, D, bs, NB, float(scale), int(sliding_window), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() if workspace is not None else 0, _stream(stream)),
        "pkv_paged_prefill_attn")
    return out, lse


def check_device_errors(stream=None) -> int:
    """Synchronise, then return and clear the OR of the kernels' device error words."""
    flags = ctypes.c_uint32(0)
    _check(lib().pkv_check_device_errors(_stream(stream), ctypes.byref(flags)),
           "pkv_check_device_errors")
    return int(flags.value)


def read_device_errors_async(host_flags, stream=None) -> None:
    """Enqueue a non-blocking readout of the OR of the kernels' device error
    words into host_flags, a pinned (page-locked) CPU int32/uint32 tensor of
    at least one element; its first element holds the value once the work
    enqueued before this call on the stream has completed. Nothing is cleared."""
    if not isinstance(host_flags, torch.Tensor) or host_flags.is_cuda \
            or host_flags.dtype not in (torch.int32,) or host_flags.numel() < 1:
        raise TypeError("host_flags must be a CPU int32 tensor")
    _check(lib().pkv_read_device_errors_async(_ptr(host_flags), _stream(stream)),
           "pkv_read_device_errors_async")


def raise_device_errors(flags: int, stream=None) -> None:
    """Raise bits of the device error words from the host, in stream order (for
    tests of error handling)."""
    _check(lib().pkv_raise_device_errors(int(flags), _stream(stream)), "pkv_raise_device_errors")


class BlockManager:
    """The host-side KV block manager of libpkv.so (pkv_blocks.h): reference-
    counted cache blocks with prefix sharing of full blocks; it emits block-table
    rows and the slots of the tokens to store."""

    def __init__(self, num_blocks: int, block_size: int):
        import numpy as np  # noqa: F401  (used by the methods)
        self._L = lib()
        self._h = self._L.pkv_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise PkvError(PKV_ERR_INVALID_ARG, "pkv_bm_create")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            self._L.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @property
    def num_free_blocks(self) -> int:
        return int(self._L.pkv_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._L.pkv_bm_ref_count(self._h, int(block)))

    def add_sequence(self, seq_id: int, token_ids) -> int:
        """Admit a prompt; returns how many leading tokens are already cached."""
        import numpy as np
        tok = np.ascontiguousarray(token_ids, dtype=np.int32)
        cached = ctypes.c_int32(0)
        _check(self._L.pkv_bm_add_sequence(self._h, int(seq_id), tok.ctypes.data, tok.shape[0],
                                           ctypes.byref(cached)), "pkv_bm_add_sequence")
        return int(cached.value)

    def append_token(self, seq_id: int, token_id: int) -> None:
        _check(self._L.pkv_bm_append_token(self._h, int(seq_id), int(token_id)),
               "pkv_bm_append_token")

    def free_sequence(self, seq_id: int) -> None:
        _check(self._L.pkv_bm_free_sequence(self._h, int(seq_id)), "pkv_bm_free_sequence")

    def num_tokens(self, seq_id: int) -> int:
        n = ctypes.c_int32(0)
        _check(self._L.pkv_bm_num_tokens(self._h, int(seq_id), ctypes.byref(n)),
               "pkv_bm_num_tokens")
        return int(n.value)

    def block_table(self, seq_id: int, max_blocks: int = None):
        """The sequence's block ids, padded with -1 to max_blocks (default: none)."""
        import numpy as np
        n = ctypes.c_int32(0)
        self._L.pkv_bm_block_table(self._h, int(seq_id), None, 0, ctypes.byref(n))
        width = int(n.value) if max_blocks is None else int(max_blocks)
        row = np.empty(width, np.int32)
        _check(self._L.pkv_bm_block_table(self._h, int(seq_id), row.ctypes.data, width,
                                          ctypes.byref(n)), "pkv_bm_block_table")
        return row

    def block_tables(self, seq_ids, max_blocks: int):
        """Block-table rows of several sequences [len(seq_ids), max_blocks]."""
        import numpy as np
        return np.stack([self.block_table(s, max_blocks) for s in seq_ids]).astype(np.int32)

    def slots(self, seq_id: int, first: int, count: int):
        """Cache slots of positions first .. first + count - 1."""
        import numpy as np
        out = np.empty(int(count), np.int32)
        _check(self._L.pkv_bm_slots(self._h, int(seq_id), int(first), int(count),
                                    out.ctypes.data), "pkv_bm_slots")
        return out
