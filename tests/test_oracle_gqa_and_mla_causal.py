"""Pins for two readings the oracle shares with the kernels (CPU only):

* the GQA grouping: q head h reads kv head h // (Hq / Hkv), i.e. contiguous
  groups of Hq / Hkv query heads per kv head;
* the right-down causal rule of the MLA sparse decode (sparse_mode 3 of the
  "KvQuantSparseFlashAttention" README, 参数说明 row sparse_mode:
  rightDownCausal): query i of L_q sees key j iff j <= i + (L_kv - L_q).

Each expected value is built here by brute force (torch SDPA in float64 on
explicitly chosen heads, or an explicit loop over the listed ids), with more
than one kv head and ids on both sides of the diagonal, so that the
interleaved mapping h % Hkv, a strict '<' or a dropped L_kv - L_q offset
give a different answer; the tests check that they do.
"""
import numpy as np
import torch

from oracle import attention, cache, e4m3, mla, quant
from quantized_paged_kv_varlen_gb300 import synth

HQ, HKV = 8, 2
G = HQ // HKV


def _sdpa(Q, K, V, scale, mask=None):
    q = torch.from_numpy(np.ascontiguousarray(Q, dtype=np.float64))[None, None]
    k = torch.from_numpy(np.ascontiguousarray(K, dtype=np.float64))[None, None]
    v = torch.from_numpy(np.ascontiguousarray(V, dtype=np.float64))[None, None]
    m = None if mask is None else torch.from_numpy(np.ascontiguousarray(mask))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    return out[0, 0].numpy()


def _contiguous(h):
    return h // G


def _interleaved(h):
    return h % HKV


def _differs_somewhere(a, b):
    return not np.allclose(a, b, rtol=1e-6, atol=1e-6)


def test_gqa_grouping_paged_decode():
    wl = synth.batched_decode(11, B=2, lo=20, hi=60, Hq=HQ, Hkv=HKV, D=32, page_size=16)
    k, v = wl.kv_all()
    P, ps, D = wl.num_pages, wl.page_size, wl.D
    z8 = np.zeros((P, ps, HKV, D), np.uint8)
    zs = np.zeros((P, ps, HKV), np.float32)
    kp, vp, ks, vs, _, _ = cache.write_fp8_token_head(
        k, v, wl.cu_seqlens, np.zeros(wl.B, np.int64), wl.block_table, ps, z8, z8, zs, zs)
    O, _ = attention.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table, wl.lengths, wl.scale)
    # dense dequantised keys per kv head, from the quantiser applied to the draws
    kc, kscale = quant.quant_fp8_last_axis(k)
    vc, vscale = quant.quant_fp8_last_axis(v)
    Kd = e4m3.decode(kc) * kscale[..., None]
    Vd = e4m3.decode(vc) * vscale[..., None]
    off = 0
    wrong_seen = False
    for b, L in enumerate(wl.lengths):
        for h in range(HQ):
            q = wl.q[b, h:h + 1].astype(np.float64)
            want = _sdpa(q, Kd[off:off + L, _contiguous(h)], Vd[off:off + L, _contiguous(h)],
                         wl.scale)
            assert np.allclose(O[b, h], want[0], rtol=1e-12, atol=1e-13)
            bad = _sdpa(q, Kd[off:off + L, _interleaved(h)], Vd[off:off + L, _interleaved(h)],
                        wl.scale)
            if _interleaved(h) != _contiguous(h):
                assert _differs_somewhere(O[b, h], bad[0])
                wrong_seen = True
        off += L
    assert wrong_seen


def test_gqa_grouping_int8_prefill():
    rng = np.random.default_rng(12)
    L, D, ps = 40, 16, 16
    P = (L + ps - 1) // ps
    bt = rng.permutation(P).astype(np.int32)[None]
    q8 = rng.integers(-127, 128, (L, HQ, D)).astype(np.int8)
    k8 = rng.integers(-127, 128, (L, HKV, D)).astype(np.int8)
    vv = synth.bf16_normal(rng, (L, HKV, D))
    qs = (rng.random((1, 1, HQ)) * 0.02 + 0.005).astype(np.float32)
    ks = (rng.random((1, 1, HKV)) * 0.02 + 0.005).astype(np.float32)
    kp = np.zeros((P, ps, HKV, D), np.int8)
    vp = np.zeros((P, ps, HKV, D), np.uint16)
    for j in range(L):                                     # place token j by an explicit page walk
        kp[bt[0, j // ps], j % ps] = k8[j]
        vp[bt[0, j // ps], j % ps] = cache.bf16_bits(vv[j])
    scale = 0.25
    O, _ = attention.paged_prefill_int8(q8, qs, kp, ks, vp, bt, np.array([L]), np.array([L]),
                                        scale, causal=True)
    mask = np.array([[j <= i for j in range(L)] for i in range(L)])
    for h in range(HQ):
        Q = q8[:, h].astype(np.float64) * float(qs[0, 0, h])
        def kv_of(hk):
            return (k8[:, hk].astype(np.float64) * float(ks[0, 0, hk]),
                    vv[:, hk].astype(np.float64))
        want = _sdpa(Q, *kv_of(_contiguous(h)), scale, mask)
        assert np.allclose(O[:, h], want, rtol=1e-11, atol=1e-12)
        if _interleaved(h) != _contiguous(h):
            assert _differs_somewhere(O[:, h], _sdpa(Q, *kv_of(_interleaved(h)), scale, mask))


def test_gqa_grouping_dense_fp8():
    rng = np.random.default_rng(13)
    B, S, D = 1, 12, 16
    raw_q = rng.standard_normal((B, S, HQ, D)).astype(np.float32)
    raw_k = rng.standard_normal((B, S, HKV, D)).astype(np.float32)
    raw_v = rng.standard_normal((B, S, HKV, D)).astype(np.float32)
    codes, desc = [], []
    for x in (raw_q, raw_k, raw_v):
        s = (np.abs(x).max(axis=(1, 3)) / np.float32(448)).astype(np.float32)   # [B, H]
        codes.append(quant.quant_fp8(x, s[:, None, :, None]))
        desc.append(s)
    O, _ = attention.dense_fp8(*codes, *desc, 0.25, causal=True)
    mask = np.tril(np.ones((S, S), dtype=bool))
    deq = lambda i, hh: e4m3.decode(codes[i][0, :, hh]) * float(desc[i][0, hh])
    for h in range(HQ):
        Q = deq(0, h)
        want = _sdpa(Q, deq(1, _contiguous(h)), deq(2, _contiguous(h)), 0.25, mask)
        assert np.allclose(O[0, :, h], want, rtol=1e-12, atol=1e-13)
        if _interleaved(h) != _contiguous(h):
            bad = _sdpa(Q, deq(1, _interleaved(h)), deq(2, _interleaved(h)), 0.25, mask)
            assert _differs_somewhere(O[0, :, h], bad)


def _mla_case():
    """One request with L_q = 3 queries over L_kv = 10 keys: query i may see
    keys j <= i + 7.  The listed ids straddle that boundary for every query
    (ids 7, 8, 9 are each on the boundary of one query)."""
    rng = np.random.default_rng(14)
    Lq, Lk, QN, bs = 3, 10, 2, 4
    kv = synth.bf16_normal(rng, (Lk, 576))
    q = synth.bf16_normal(rng, (Lq, QN, 576))
    P = (Lk + bs - 1) // bs
    bt = rng.permutation(P).astype(np.int32)[None]
    pool = np.zeros((P, bs, 1, 656), np.uint8)
    pool, _ = cache.write_mla_rows(kv, np.array([Lk]), np.array([0]), bt, bs, pool)
    ids = np.array([9, 2, 7, 8, 0, 5, -1, -1], np.int32)
    idx = np.tile(ids, (Lq, 1))[:, None, :]
    K, V = cache.mla_unpack_rows(cache.mla_pack_rows(kv))
    return dict(q=q, pool=pool, idx=idx, bt=bt, Lq=Lq, Lk=Lk, K=K, V=V, ids=ids[:6])


def _expected(case, rule, scale):
    out = []
    for i in range(case["Lq"]):
        keep = [j for j in case["ids"].tolist() if rule(i, j)]
        if not keep:
            out.append(np.zeros((case["q"].shape[1], 512)))
            continue
        o, _ = attention.attend_rows(case["q"][i].astype(np.float64), case["K"][keep],
                                     case["V"][keep], scale)
        out.append(o)
    return np.stack(out)


def test_mla_sparse_mode3_right_down_causal():
    c = _mla_case()
    scale = 1.0 / 24
    O, _ = mla.mla_sparse_decode(c["q"], c["pool"], c["idx"], c["bt"], np.array([c["Lk"]]),
                                 np.array([c["Lq"]]), scale, sparse_mode=3)
    off = c["Lk"] - c["Lq"]
    want = _expected(c, lambda i, j: j <= i + off, scale)
    assert np.allclose(O, want, rtol=1e-12, atol=1e-13)
    # the boundary ids: query 0 keeps 7 but not 8 or 9; query 2 keeps all six
    for wrong in (lambda i, j: j < i + off,                  # strict comparison
                  lambda i, j: j <= i):                     # L_kv - L_q dropped
        assert _differs_somewhere(O, _expected(c, wrong, scale))
    # sparse_mode 0 ignores the diagonal: every listed id for every query
    O0, _ = mla.mla_sparse_decode(c["q"], c["pool"], c["idx"], c["bt"], np.array([c["Lk"]]),
                                  np.array([c["Lq"]]), scale, sparse_mode=0)
    assert np.allclose(O0, _expected(c, lambda i, j: True, scale), rtol=1e-12, atol=1e-13)
    assert _differs_somewhere(O0[0], O[0]) and np.allclose(O0[2], O[2], rtol=1e-13, atol=1e-14)


def test_mla_order_of_the_listed_ids_does_not_matter():
    """The keys of a token are a set: the oracle's output and lse are the same
    for any order of the ids before the first -1 (the kernel sorts each
    512-key group by pool row and relies on this).  The -1 that ends the list
    is part of the reading: moving it changes which ids count, and that does
    change the result."""
    rng = np.random.default_rng(23)
    L, bs, QN = 300, 16, 4
    bt, P = synth.page_tables(rng, np.array([L], np.int32), bs)
    kv = synth.bf16_normal(rng, (L, 576))
    q = synth.bf16_normal(rng, (1, QN, 576))
    pool = np.zeros((P, bs, 1, 656), np.uint8)
    pool, _ = cache.write_mla_rows(kv, np.array([L], np.int32), np.zeros(1, np.int64), bt, bs, pool)
    ids = rng.permutation(L)[:120].astype(np.int32)
    idx = np.full((1, 1, 160), -1, np.int32)
    idx[0, 0, :120] = ids
    lk, cu = np.array([L], np.int32), np.array([1], np.int32)
    o1, l1 = mla.mla_sparse_decode(q, pool, idx, bt, lk, cu, 1.0 / np.sqrt(576.0))
    idx2 = idx.copy()
    idx2[0, 0, :120] = ids[rng.permutation(120)]
    o2, l2 = mla.mla_sparse_decode(q, pool, idx2, bt, lk, cu, 1.0 / np.sqrt(576.0))
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)
    # the first -1 ends the list: ids after it are not keys
    idx3 = idx.copy()
    idx3[0, 0, 60] = -1
    o3, _ = mla.mla_sparse_decode(q, pool, idx3, bt, lk, cu, 1.0 / np.sqrt(576.0))
    assert _differs_somewhere(o1, o3)
