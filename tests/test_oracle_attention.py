"""Pins for the oracle's attention paths (CPU only): brute force against torch
SDPA in float64, closed forms and invariants that a dropped term, a wrong
sign, a transposed operand or a wrong head/page index would break."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, cache, e4m3, mla, quant, rope
from quantized_paged_kv_varlen_gb300 import synth


def _sdpa(Q, K, V, scale, mask=None):
    """torch SDPA in float64 on the CPU (library routine)."""
    q = torch.from_numpy(np.ascontiguousarray(Q))[None, None]
    k = torch.from_numpy(np.ascontiguousarray(K))[None, None]
    v = torch.from_numpy(np.ascontiguousarray(V))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=m, scale=scale)[0, 0].numpy()


def _fp8_cache(wl):
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    z8 = np.zeros((P, ps, H, D), np.uint8)
    zs = np.zeros((P, ps, H), np.float32)
    kp, vp, ks, vs, _, _ = cache.write_fp8_token_head(
        k, v, wl.cu_seqlens, np.zeros(wl.B, np.int64), wl.block_table, ps, z8, z8, zs, zs)
    return kp, vp, ks, vs


def test_hand_worked_two_keys():
    # q = (1, 0); keys (1, 0), (0, 1); values (1, 2), (3, 4); scale 1:
    # logits (1, 0), O = ((e + 3)/(e + 1), (2e + 4)/(e + 1)), lse = ln(e + 1)
    e = math.e
    O, lse = attention.attend_rows(np.array([[1.0, 0.0]]), np.eye(2),
                                   np.array([[1.0, 2.0], [3.0, 4.0]]), 1.0)
    assert np.allclose(O[0], [(e + 3) / (e + 1), (2 * e + 4) / (e + 1)], rtol=1e-15)
    assert abs(lse[0] - math.log(e + 1)) < 1e-15


def test_paged_decode_matches_sdpa_bruteforce():
    wl = synth.tiny_decode(0)
    kp, vp, ks, vs = _fp8_cache(wl)
    O, lse = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table,
                                        wl.lengths, wl.scale)
    # dense dequantised copy built by walking the tokens in order
    k, v = wl.kv_all()
    kc, kscale = quant.quant_fp8_last_axis(k)
    vc, vscale = quant.quant_fp8_last_axis(v)
    Kd = e4m3.decode(kc) * kscale[..., None]
    Vd = e4m3.decode(vc) * vscale[..., None]
    off = 0
    for b, L in enumerate(wl.lengths):
        for h in range(wl.Hq):
            ref = _sdpa(wl.q[b, h:h + 1].astype(np.float64), Kd[off:off + L, 0],
                        Vd[off:off + L, 0], wl.scale)
            assert np.allclose(O[b, h], ref[0], rtol=1e-12, atol=1e-13)
            lg = wl.scale * Kd[off:off + L, 0] @ wl.q[b, h].astype(np.float64)
            assert abs(lse[b, h] - (lg.max() + np.log(np.exp(lg - lg.max()).sum()))) < 1e-12
        off += L


def test_single_visible_key_returns_its_value_row():
    rng = np.random.default_rng(0)
    K = rng.standard_normal((1, 8))
    V = rng.standard_normal((1, 5))
    q = rng.standard_normal((3, 8))
    O, lse = attention.attend_rows(q, K, V, 0.3)
    assert np.array_equal(O, np.repeat(V, 3, axis=0))
    assert np.allclose(lse, 0.3 * q @ K[0], rtol=1e-15)
    # causal, query 0 of a square problem sees key 0 only
    K = rng.standard_normal((6, 8))
    V = rng.standard_normal((6, 5))
    O, _ = attention.attend_rows(rng.standard_normal((6, 8)), K, V, 0.3,
                                 attention.causal_visible(6, 6))
    assert np.allclose(O[0], V[0], rtol=1e-15)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    K = np.repeat(rng.standard_normal((1, 8)), 7, axis=0)
    V = rng.standard_normal((7, 4))
    q = rng.standard_normal((2, 8))
    O, lse = attention.attend_rows(q, K, V, 0.5)
    assert np.allclose(O, V.mean(0)[None], rtol=1e-14, atol=1e-15)
    assert np.allclose(lse, 0.5 * q @ K[0] + np.log(7), rtol=1e-14)


def test_no_visible_key_gives_zero_and_neg_inf():
    O, lse = attention.attend_rows(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 1.0)
    assert np.all(O == 0) and np.all(np.isneginf(lse))
    vis = np.zeros((1, 3), dtype=bool)
    O, lse = attention.attend_rows(np.ones((1, 4)), np.ones((3, 4)), np.ones((3, 3)), 1.0, vis)
    assert np.all(O == 0) and np.all(np.isneginf(lse)) and not np.isnan(O).any()


def test_permuted_page_table_is_bitwise_invariant():
    wl = synth.tiny_decode(0)
    kp, vp, ks, vs = _fp8_cache(wl)
    O1, l1 = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table,
                                        wl.lengths, wl.scale)
    # contiguous storage: identity page table, pages moved accordingly
    P = wl.num_pages
    order = np.concatenate([wl.block_table[b, :(L + 15) // 16] for b, L in enumerate(wl.lengths)])
    ident = np.full_like(wl.block_table, -1)
    off = 0
    for b, L in enumerate(wl.lengths):
        n = (L + 15) // 16
        ident[b, :n] = np.arange(off, off + n)
        off += n
    O2, l2 = attention.paged_decode_fp8(wl.q, kp[order], vp[order], ks[order], vs[order],
                                        ident, wl.lengths, wl.scale)
    assert off == P
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_wrong_head_mapping_or_transposed_page_is_caught():
    """Planted mistakes (in copies here): interleaved GQA heads, or reading
    token offsets as page indices, change the result."""
    wl = synth.tiny_decode(0)
    kp, vp, ks, vs = _fp8_cache(wl)
    O, _ = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table,
                                      wl.lengths, wl.scale)
    # request 0 has 37 tokens: pages 0, 1 full, page 2 holds 5; swapping a
    # full page with the partial one reads 11 unwritten slots
    bad_bt = wl.block_table.copy()
    bad_bt[0, [0, 2]] = bad_bt[0, [2, 0]]
    O_bad, _ = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, bad_bt, wl.lengths, wl.scale)
    assert not np.allclose(O[0], O_bad[0])
    q_perm = wl.q[:, [0, 2, 1, 3]]
    O_perm, _ = attention.paged_decode_fp8(q_perm, kp, vp, ks, vs, wl.block_table,
                                           wl.lengths, wl.scale)
    assert np.allclose(O_perm[:, [0, 2, 1, 3]], O)        # one kv head: heads are independent


def test_shift_invariance():
    rng = np.random.default_rng(2)
    Q = rng.standard_normal((4, 16))
    K = rng.standard_normal((30, 16))
    V = rng.standard_normal((30, 8))
    c = rng.standard_normal(16)
    O1, l1 = attention.attend_rows(Q, K, V, 0.25)
    O2, l2 = attention.attend_rows(Q, K - c[None], V, 0.25)
    assert np.allclose(O1, O2, rtol=1e-12, atol=1e-13)
    assert np.allclose(l2, l1 - 0.25 * Q @ c, rtol=1e-12)


def test_split_and_lse_merge_equals_unsplit():
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((3, 16))
    K = rng.standard_normal((100, 16))
    V = rng.standard_normal((100, 8))
    O, lse = attention.attend_rows(Q, K, V, 0.25)
    cuts = [0, 13, 13, 64, 100]                              # includes an empty split
    parts = [attention.attend_rows(Q, K[a:b], V[a:b], 0.25) for a, b in zip(cuts[:-1], cuts[1:])]
    Om, lm = attention.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(Om, O, rtol=1e-12, atol=1e-13)
    assert np.allclose(lm, lse, rtol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    wl = synth.tiny_decode(1)
    kp, vp, ks, vs = _fp8_cache(wl)
    O, lse = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table,
                                        wl.lengths, wl.scale)
    G = wl.Hq
    rep = lambda a: np.repeat(a, G, axis=2)
    Om, lm = attention.paged_decode_fp8(wl.q, rep(kp), rep(vp), rep(ks), rep(vs),
                                        wl.block_table, wl.lengths, wl.scale)
    # same math, different BLAS row grouping: equal up to fp64 rounding
    assert np.allclose(O, Om, rtol=1e-13, atol=1e-14) and np.allclose(lse, lm, rtol=1e-14)


def test_causal_prefill_matches_sdpa_with_explicit_mask():
    rng = np.random.default_rng(4)
    wl = synth.varlen_prefill(0, lengths=[5, 131, 1], H=2, D=16, page_size=16)
    cos, sin = rope.cos_sin_table(256, wl.D, wl.theta)
    T = int(wl.lengths.sum())
    P = wl.num_pages
    k0 = np.zeros((P, 16, wl.H, wl.D), np.int8)
    v0 = np.zeros((P, 16, wl.H, wl.D), np.uint16)
    kp, vp, kscale, q8, qscale, _ = cache.write_int8_block128_rope(
        wl.q, wl.k, wl.v, wl.cu_seqlens, wl.block_table, 16, cos, sin, wl.num_blocks, k0, v0)
    O, lse = attention.paged_prefill_int8(q8, qscale, kp, kscale, vp, wl.block_table,
                                          wl.cu_seqlens, wl.lengths, wl.scale, causal=True)
    # dense reference from the oracle's own quantised values, mask built by loops
    off = 0
    for b, L in enumerate(wl.lengths):
        mask = np.array([[j <= i for j in range(L)] for i in range(L)])
        for h in range(wl.H):
            blk = np.arange(L) // 128
            Qd = q8[off:off + L, h].astype(np.float64) * qscale[b, blk, h][:, None]
            k_rot = rope.rotate(wl.k[off:off + L], np.arange(L), cos, sin)
            kc, ks = cache.block128_quant(k_rot, np.array([L]), wl.num_blocks)
            Kd = kc[:, h].astype(np.float64) * ks[0, blk, h][:, None]
            Vd = wl.v[off:off + L, h].astype(np.float64)
            ref = _sdpa(Qd, Kd, Vd, wl.scale, mask)
            assert np.allclose(O[off:off + L, h], ref, rtol=1e-11, atol=1e-12)
        off += L
    # right-down causal with L_q < L_kv: the last query sees every key
    Q = rng.standard_normal((2, 8))
    K = rng.standard_normal((5, 8))
    vis = attention.causal_visible(2, 5)
    assert vis[1].all() and vis[0].tolist() == [True, True, True, True, False]


def test_dense_fp8_matches_sdpa():
    rng = np.random.default_rng(5)
    B, S, H, D = 2, 9, 3, 16
    raw = [rng.standard_normal((B, S, H, D)).astype(np.float32) for _ in range(3)]
    codes, desc = [], []
    for x in raw:
        amax = np.abs(x).max(axis=(1, 3))                    # [B, H]
        s = (amax / np.float32(448)).astype(np.float32)
        codes.append(quant.quant_fp8(x, s[:, None, :, None]))
        desc.append(s)
    O, lse = attention.dense_fp8(*codes, *desc, 0.25, causal=True)
    for b in range(B):
        for h in range(H):
            Qd, Kd, Vd = (e4m3.decode(c[b, :, h]) * d[b, h] for c, d in zip(codes, desc))
            mask = np.tril(np.ones((S, S), dtype=bool))
            ref = _sdpa(Qd, Kd, Vd, 0.25, mask)
            assert np.allclose(O[b, :, h], ref, rtol=1e-12, atol=1e-13)
    rows = [(1, 4, 2), (0, 0, 0)]
    Os, _ = attention.dense_fp8(*codes, *desc, 0.25, causal=True, rows=rows)
    for b, s, h in rows:
        assert np.allclose(Os[b, s, h], O[b, s, h], rtol=1e-13, atol=1e-14)


def _mla_pool(wl):
    P, bs = wl.num_pages, wl.block_size
    pool = np.zeros((P, bs, 1, 656), np.uint8)
    for b in range(wl.B):
        kv = wl.kv(b)
        L = kv.shape[0]
        pool, _ = cache.write_mla_rows(kv, np.array([L]), np.array([0]),
                                       wl.block_table[b:b + 1], bs, pool)
    return pool


def test_mla_sparse_covering_equals_dense_and_is_order_free():
    wl = synth.mla_sparse(0, B=2, QN=4, lengths=[70, 130], block_size=64, topk=200,
                          sparse_size=160)
    pool = _mla_pool(wl)
    O, lse = mla.mla_sparse_decode(wl.q, pool, wl.sparse_indices, wl.block_table,
                                   wl.lengths, wl.cu_seqlens_q, wl.scale)
    for b in range(2):
        L = int(wl.lengths[b])
        n_valid = min(L, 160)
        ids = wl.sparse_indices[b, 0, :n_valid]
        assert sorted(ids.tolist()) == (list(range(L)) if L <= 160 else sorted(ids.tolist()))
        K, V = cache.mla_unpack_rows(cache.mla_pack_rows(wl.kv(b))[ids])
        ref, lref = attention.attend_rows(wl.q[b].astype(np.float64), K, V, wl.scale)
        assert np.allclose(O[b], ref, rtol=1e-12, atol=1e-13)
        if L <= 160:                                           # covering: dense over all L
            Kd, Vd = cache.mla_unpack_rows(cache.mla_pack_rows(wl.kv(b)))
            dense, _ = attention.attend_rows(wl.q[b].astype(np.float64), Kd, Vd, wl.scale)
            assert np.allclose(O[b], dense, rtol=1e-12, atol=1e-13)
    # permuting the listed ids does not change the result
    idx2 = wl.sparse_indices.copy()
    idx2[0, 0, :70] = idx2[0, 0, :70][::-1]
    O2, _ = mla.mla_sparse_decode(wl.q, pool, idx2, wl.block_table, wl.lengths,
                                  wl.cu_seqlens_q, wl.scale)
    assert np.allclose(O2, O, rtol=1e-12, atol=1e-13)


def test_mla_reduces_to_plain_attention_with_unit_scales_and_zero_rope():
    """Integer-valued nope with absmax 127 in every tile has scale exactly 1,
    so Dequant is the identity; a zero rope part drops out of the logits."""
    rng = np.random.default_rng(6)
    L, QN = 40, 3
    nope = rng.integers(-126, 127, (L, 512)).astype(np.float32)
    nope[:, ::128] = 127.0
    kv = np.concatenate([nope, np.zeros((L, 64), np.float32)], axis=1)
    rows = cache.mla_pack_rows(kv)
    assert np.all(rows[:, 640:].copy().view("<f4") == 1.0)
    q = synth.bf16_normal(rng, (1, QN, 576))
    pool = rows.reshape(1, L, 1, 656)
    idx = np.arange(L, dtype=np.int32).reshape(1, 1, L)
    O, _ = mla.mla_sparse_decode(q, pool, idx, np.zeros((1, 1), np.int32), np.array([L]),
                                 np.array([1]), 1.0 / 24)
    ref = _sdpa(q[0, :, :512].astype(np.float64), nope.astype(np.float64),
                nope.astype(np.float64), 1.0 / 24)
    assert np.allclose(O[0], ref, rtol=1e-12, atol=1e-10)


def test_mla_index_list_stops_at_first_negative_and_rejects_out_of_range():
    assert mla.valid_ids([3, 1, -1, 7], 10).tolist() == [3, 1]
    with pytest.raises(ValueError):
        mla.valid_ids([3, 10], 10)


def test_mla_block_sparse_covering_equals_dense():
    """Block-wise lists (sparse_block_size n): listing every n-token block of
    the sequence, in any order, is dense attention over all L tokens; a
    single block id sees exactly its (clipped) tokens; a block starting at or
    past L_kv is out of range."""
    rng = np.random.default_rng(21)
    L, QN, n, bs = 45, 3, 8, 16
    kv = synth.bf16_normal(rng, (L, 576))
    q = synth.bf16_normal(rng, (1, QN, 576))
    bt = rng.permutation(3).astype(np.int32)[None]
    pool = np.zeros((3, bs, 1, 656), np.uint8)
    pool, _ = cache.write_mla_rows(kv, np.array([L]), np.array([0]), bt, bs, pool)
    Kd, Vd = cache.mla_unpack_rows(cache.mla_pack_rows(kv))
    nblk = (L + n - 1) // n                                   # 6 blocks, the last holds 5 tokens
    idx = np.full((1, 1, 8), -1, np.int32)
    idx[0, 0, :nblk] = rng.permutation(nblk)
    O, lse = mla.mla_sparse_decode(q, pool, idx, bt, np.array([L]), np.array([1]), 0.05,
                                   sparse_block_size=n)
    dense, ldense = attention.attend_rows(q[0].astype(np.float64), Kd, Vd, 0.05)
    assert np.allclose(O[0], dense, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse[0], ldense, rtol=1e-13, atol=1e-13)
    idx1 = np.full((1, 1, 2), -1, np.int32)
    idx1[0, 0, 0] = 5                                         # tokens 40..44
    O1, _ = mla.mla_sparse_decode(q, pool, idx1, bt, np.array([L]), np.array([1]), 0.05,
                                  sparse_block_size=n)
    ref, _ = attention.attend_rows(q[0].astype(np.float64), Kd[40:45], Vd[40:45], 0.05)
    assert np.allclose(O1[0], ref, rtol=1e-12, atol=1e-13)
    assert mla.valid_ids([1, -1], 45, 8).tolist() == list(range(8, 16))
    with pytest.raises(ValueError):
        mla.valid_ids([6], 45, 8)                             # 6 * 8 = 48 >= 45


def test_hnd_layout_holds_the_same_tokens_and_decodes_the_same():
    """HND pools [P, H, page_size, D] hold token (page, offset o) of head h
    at [page, h, o]: the same codes as NHD's [page, o, h], with the scale
    pools unchanged, and decode over either layout gives identical results."""
    wl = synth.batched_decode(3, B=3, lo=20, hi=70, Hq=8, Hkv=2, D=64, page_size=16)
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    start = np.zeros(wl.B, np.int64)
    zs = np.zeros((P, ps, H), np.float32)
    nhd = cache.write_fp8_token_head(k, v, wl.cu_seqlens, start, wl.block_table, ps,
                                     np.zeros((P, ps, H, D), np.uint8),
                                     np.zeros((P, ps, H, D), np.uint8), zs, zs)
    hnd = cache.write_fp8_token_head(k, v, wl.cu_seqlens, start, wl.block_table, ps,
                                     np.zeros((P, H, ps, D), np.uint8),
                                     np.zeros((P, H, ps, D), np.uint8), zs, zs, layout="HND")
    b_of, p_of = cache.token_positions(wl.cu_seqlens, start)
    for t in range(0, len(b_of), 7):
        page = wl.block_table[b_of[t], p_of[t] // ps]
        o = p_of[t] % ps
        for h in range(H):
            assert np.array_equal(hnd[0][page, h, o], nhd[0][page, o, h])
            assert np.array_equal(hnd[1][page, h, o], nhd[1][page, o, h])
    assert np.array_equal(hnd[2], nhd[2]) and np.array_equal(hnd[3], nhd[3])
    O1, l1 = attention.paged_decode_fp8(wl.q, *nhd[:4], wl.block_table, wl.lengths, wl.scale)
    O2, l2 = attention.paged_decode_fp8(wl.q, *hnd[:4], wl.block_table, wl.lengths, wl.scale,
                                        layout="HND")
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)
