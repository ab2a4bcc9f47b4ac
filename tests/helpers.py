"""Helpers shared by the tests: widening bf16 bit patterns with torch (a library
conversion, independent of the oracle's own), and assembling each sequence's
keys and values in logical order straight from the generator's token lists
(independent of slots, tables and the cache)."""
import numpy as np
import torch


def bf16_bits_to_f64(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def bf16_bits_to_torch(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def logical_kv(stores, seq: int, n_keys: int):
    """K, V [n_keys, H_kv, D] (uint16) of sequence `seq` at positions 0..n_keys-1,
    from the token rows of the given stores. Rows of a shared prefix stored through
    another sequence's table are found through their position alone when `seq`
    has none of its own at that position."""
    H_kv, D = stores[0].k.shape[1:]
    k = np.zeros((n_keys, H_kv, D), np.uint16)
    v = np.zeros((n_keys, H_kv, D), np.uint16)
    have = np.zeros(n_keys, bool)
    for st in stores:
        sel = (st.seq_ids == seq) & (st.positions < n_keys)
        k[st.positions[sel]] = st.k[sel]
        v[st.positions[sel]] = st.v[sel]
        have[st.positions[sel]] = True
    for st in stores:  # shared prefix rows
        sel = (~have[np.minimum(st.positions, n_keys - 1)]) & (st.positions < n_keys)
        k[st.positions[sel]] = st.k[sel]
        v[st.positions[sel]] = st.v[sel]
        have[st.positions[sel]] = True
    assert have.all(), "some key positions were never stored"
    return k, v


def sdpa_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, n_keys_per_row,
              first_key_per_row=None):
    """Library attention (torch SDPA, fp64) of query rows q_rows [R, H_q, D] over
    k, v [Lk, H_kv, D] where row r may see keys [first_key_per_row[r] (default 0),
    n_keys_per_row[r]). Returns (out [R, H_q, D], lse [R, H_q])."""
    q = bf16_bits_to_f64(q_rows).permute(1, 0, 2)            # [H_q, R, D]
    kk = bf16_bits_to_f64(k).permute(1, 0, 2)                # [H_kv, Lk, D]
    vv = bf16_bits_to_f64(v).permute(1, 0, 2)
    G = q.shape[0] // kk.shape[0]
    kk = kk.repeat_interleave(G, dim=0)
    vv = vv.repeat_interleave(G, dim=0)
    R, Lk = q.shape[1], kk.shape[1]
    lim = torch.as_tensor(np.asarray(n_keys_per_row), dtype=torch.int64)
    mask = torch.arange(Lk)[None, :] < lim[:, None]           # [R, Lk]
    if first_key_per_row is not None:
        lo = torch.as_tensor(np.asarray(first_key_per_row), dtype=torch.int64)
        mask &= torch.arange(Lk)[None, :] >= lo[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=scale)
    logits = torch.matmul(q, kk.transpose(1, 2)) * scale
    logits = logits.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(logits, dim=-1)                     # [H_q, R]
    return out.permute(1, 0, 2).numpy(), lse.T.numpy()
