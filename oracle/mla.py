"""MLA-absorb sparse attention over the combined-row paged cache.

Test infrastructure only (see oracle/__init__.py).

"KvQuantSparseFlashAttention" README, 参数说明 rows query / key / value /
sparse_indices / attention_mode / rope_head_dim / quant_scale_repo_mode /
sparse_mode, and the formula under 计算公式:

* query [T, Q_N, 576] = q_nope (512) || q_rope (64), TND with inclusive
  prefix sums ``cu_seqlens_q`` (actual_seq_lengths_query);
* the cache is PA_BSND [block_num, block_size, 1, 656]: per token 512 INT8
  nope codes, 64 bf16 rope values, 4 fp32 per-128-tile scales (combined
  storage, quant_scale_repo_mode = 1);
* attention_mode 2 (MLA-absorb): K and V are the same stored row; the key is
  the dequantised nope followed by the rope part (576 wide), the value is the
  dequantised nope (512 wide), so the output is [T, Q_N, 512];
* sparse_indices [T, 1, sparse_size] lists logical token positions of the
  request (mapped through block_table); valid entries come first, the first
  -1 ends the list; with sparse_block_size n > 1 (row sparse_block_size,
  block-wise sparsity) an entry names the n tokens [id*n, id*n + n) of the
  request, which share the decision, and the tokens at or past L_kv of the
  last block are not keys;
* sparse_mode 3 additionally drops ids outside the right-down causal region.
"""
import numpy as np

from . import cache
from .attention import NEG_INF, attend_rows, page_rows


def valid_ids(index_row, L_kv, block=1):
    """Token positions named by one sparse_indices row: its entries up to the
    first -1, each covering `block` tokens (clipped to the sequence)."""
    ids = []
    for x in np.asarray(index_row).tolist():
        if x < 0:
            break
        if x * block >= L_kv:
            raise ValueError(f"sparse index {x} outside the sequence (L = {L_kv})")
        for o in range(block):
            if x * block + o < L_kv:
                ids.append(int(x) * block + o)
    return np.asarray(ids, dtype=np.int64)


def mla_sparse_decode(q, kv_pool, sparse_indices, block_table, seqlens_kv,
                      cu_seqlens_q, scale, sparse_mode=0, tokens=None, sparse_block_size=1):
    """q f32 [T, QN, 576] (bf16 values); kv_pool u8 [P, bs, 1, 656];
    sparse_indices int32 [T, 1, S]; returns (O f64[T, QN, 512], lse f64[T, QN]).
    ``tokens``: optional subset of query tokens to compute.
    """
    q = np.asarray(q, dtype=np.float64)
    T, QN, _ = q.shape
    P, bs, _, W = kv_pool.shape
    flat = kv_pool.reshape(P * bs, W)
    begin, end = cache.seq_bounds(cu_seqlens_q)
    O = np.zeros((T, QN, cache.MLA_NOPE))
    lse = np.full((T, QN), NEG_INF)
    todo = set(range(T)) if tokens is None else set(int(t) for t in tokens)
    for b in range(len(begin)):
        Lq = int(end[b] - begin[b])
        Lk = int(seqlens_kv[b])
        for i in range(Lq):
            t = int(begin[b]) + i
            if t not in todo:
                continue
            ids = valid_ids(sparse_indices[t, 0], Lk, sparse_block_size)
            if sparse_mode == 3:
                ids = ids[ids <= i + (Lk - Lq)]
            if ids.size == 0:
                continue
            K, V = cache.mla_unpack_rows(flat[page_rows(block_table[b], bs, ids)])
            o, l = attend_rows(q[t], K, V, scale)
            O[t] = o
            lse[t] = l
    return O, lse
