"""Attention over dequantised, page-gathered keys and values, in float64.

Test infrastructure only (see oracle/__init__.py).

The definition ("KvQuantSparseFlashAttention" README, 计算公式):

    Attention = softmax(scale * Q . Dequant(K~, S_K)^T) . Dequant(V~, S_V)

with ``scale`` the README's scale_value (1/sqrt(d_k) by default; the aiter
FP8 usage passes softmax_scale=None for the same default), K~ / V~ the keys
and values a request may see: its first L_kv tokens gathered through
block_table, optionally restricted to the ids listed in sparse_indices and
to the right-down causal region (参数说明 row sparse_mode: 3 =
rightDownCausal, the lower triangle whose boundary runs from the bottom-right
corner; 0 = everything).

Readings where the pages are silent: query i of a request with L_q queries and
L_kv keys sees key j iff j <= i + (L_kv - L_q) under sparse_mode 3; q head h
reads kv head h // (Hq / Hkv); lse = logsumexp of the scaled logits (natural
log); a row with no visible key gives O = 0 and lse = -inf.

Every softmax here is the plain formula over the full visible set: no
blocking, no running maximum.
"""
import numpy as np

from . import cache, e4m3, quant

NEG_INF = -np.inf


def attend_rows(Q, K, V, scale, visible=None):
    """Q f64[m, D], K f64[n, D], V f64[n, Dv], visible bool[m, n] or None.

    Returns (O f64[m, Dv], lse f64[m]).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m = Q.shape[0]
    O = np.zeros((m, V.shape[1]), dtype=np.float64)
    lse = np.full(m, NEG_INF, dtype=np.float64)
    if K.shape[0] == 0 or m == 0:
        return O, lse
    logits = float(scale) * (Q @ K.T)
    if visible is not None:
        logits = np.where(visible, logits, NEG_INF)
    mx = np.max(logits, axis=1)
    has = np.isfinite(mx)
    if not np.any(has):
        return O, lse
    p = np.exp(logits[has] - mx[has, None])
    denom = np.sum(p, axis=1)
    O[has] = (p @ V) / denom[:, None]
    lse[has] = mx[has] + np.log(denom)
    return O, lse


def causal_visible(Lq, Lk):
    """Right-down causal mask bool[Lq, Lk]: j <= i + (Lk - Lq)."""
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    return j <= i + (Lk - Lq)


def page_rows(block_table_row, page_size, positions):
    """Pool row (page * ps + offset) of logical token positions."""
    positions = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table_row, dtype=np.int64)
    return bt[positions // page_size] * page_size + positions % page_size


def lse_merge(O_parts, lse_parts):
    """Combine partial results over disjoint key sets.

    O_parts f64[S, ..., Dv], lse_parts f64[S, ...] -> (O, lse): the weights are
    exp(lse_s - M) with M the largest finite lse (flashinfer plan/run split,
    "Batch Decode/Prefill Attention Kernels").
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = np.max(lse_parts, axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - Ms[None]), 0.0)
    tot = np.sum(w, axis=0)
    safe = np.where(tot > 0, tot, 1.0)
    O = np.sum(w[..., None] * O_parts, axis=0) / safe[..., None]
    O = np.where((tot > 0)[..., None], O, 0.0)
    lse = np.where(tot > 0, Ms + np.log(safe), NEG_INF)
    return O, lse


# ---------------------------------------------------------------- decode (FP8)

def gather_fp8_token_head(k_pool, v_pool, k_scale_pool, v_scale_pool,
                          block_table_row, L, h, layout="NHD"):
    """Dequantised K, V f64[L, D] of kv head h of one request.

    layout "NHD": pools [P, page_size, H, D]; "HND" (flashinfer's
    kv_layout_code): pools [P, H, page_size, D].  Scale pools are
    [P, page_size, H] in both."""
    if layout == "HND":
        P, H, ps, D = k_pool.shape
    else:
        P, ps, H, D = k_pool.shape
    pos = np.arange(L)
    page = np.asarray(block_table_row, dtype=np.int64)[pos // ps]
    off = pos % ps
    if layout == "HND":
        kc, vc = k_pool[page, h, off], v_pool[page, h, off]
    else:
        kc, vc = k_pool[page, off, h], v_pool[page, off, h]
    K = quant.dequant_fp8(kc, k_scale_pool[page, off, h][:, None])
    V = quant.dequant_fp8(vc, v_scale_pool[page, off, h][:, None])
    return K, V


def paged_decode_fp8(q, k_pool, v_pool, k_scale_pool, v_scale_pool,
                     block_table, seqlens_kv, scale, requests=None, layout="NHD"):
    """One query token per request (L_q = 1) over an FP8 paged cache.

    q: f32/f64 [B, Hq, D] (bf16 values).  Returns (O f64[B, Hq, D],
    lse f64[B, Hq]); with ``requests`` given only those rows are filled.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1 if layout == "HND" else 2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), NEG_INF)
    for b in (range(B) if requests is None else requests):
        L = int(seqlens_kv[b])
        for h in range(Hkv):
            K, V = gather_fp8_token_head(k_pool, v_pool, k_scale_pool, v_scale_pool,
                                         block_table[b], L, h, layout)
            o, l = attend_rows(q[b, h * G:(h + 1) * G], K, V, scale)
            O[b, h * G:(h + 1) * G] = o
            lse[b, h * G:(h + 1) * G] = l
    return O, lse


# ------------------------------------------------- varlen prefill (INT8 Q/K)

def paged_prefill_int8(q8, q_scale, k_pool, k_scale, v_pool_bits, block_table,
                       cu_seqlens_q, seqlens_kv, scale, causal=True,
                       rows=None, v_scale=None):
    """Sage-style varlen prefill: INT8 Q and K with per-(sequence, 128-token
    block, head) scales, bf16 V, all K/V gathered through block_table.

    q8 int8 [T, H, D]; q_scale / k_scale f32 [B, NB, H]; k_pool int8
    [P, ps, Hkv, D]; v_pool_bits uint16 (bf16) [P, ps, Hkv, D].
    Query block of query i is i // 128, key block of key j is j // 128.
    ``rows``: optional list of (token, head) pairs to compute (else all).
    With ``v_scale`` (f32 [B, Hkv, D]) the V pool holds E4M3 codes and
    V = code * v_scale[b, head, channel].
    Returns (O f64[T, H, D], lse f64[T, H]).
    """
    T, H, D = q8.shape
    P, ps, Hkv, _ = k_pool.shape
    G = H // Hkv
    begin, end = cache.seq_bounds(cu_seqlens_q)
    O = np.zeros((T, H, D))
    lse = np.full((T, H), NEG_INF)
    want = None
    if rows is not None:
        want = {}
        for t, h in rows:
            want.setdefault(int(h), set()).add(int(t))
    kp = k_pool.reshape(P * ps, Hkv, D)
    vp = v_pool_bits.reshape(P * ps, Hkv, D)
    for b in range(len(begin)):
        Lq = int(end[b] - begin[b])
        Lk = int(seqlens_kv[b])
        if Lq == 0:
            continue
        prow = page_rows(block_table[b], ps, np.arange(Lk))
        kblk = np.arange(Lk) // 128
        qblk = np.arange(Lq) // 128
        vis = causal_visible(Lq, Lk) if causal else None
        for h in range(H):
            sel = np.arange(Lq)
            if want is not None:
                ts = want.get(h, set())
                sel = np.array(sorted(t - int(begin[b]) for t in ts
                                      if begin[b] <= t < end[b]), dtype=np.int64)
                if sel.size == 0:
                    continue
            hk = h // G
            K = quant.dequant_int8(kp[prow, hk], k_scale[b, kblk, hk][:, None])
            if v_scale is None:
                V = cache.bf16_value(vp[prow, hk])
            else:
                V = quant.dequant_fp8(vp[prow, hk], v_scale[b, hk][None, :])
            Q = quant.dequant_int8(q8[begin[b] + sel, h],
                                   q_scale[b, qblk[sel], h][:, None])
            o, l = attend_rows(Q, K, V, scale, None if vis is None else vis[sel])
            O[begin[b] + sel, h] = o
            lse[begin[b] + sel, h] = l
    return O, lse


# ---------------------------------------------- dense FP8 (per-(b, h) descale)

def dense_fp8(q8, k8, v8, q_descale, k_descale, v_descale, scale, causal,
              rows=None):
    """FA-v3-style FP8 attention ("[Triton] FP8 with FA v3 API", the
    flash_attn_func usage): q8/k8/v8 E4M3 codes [B, S, H, D] (BSND),
    descales f32 [B, H] (k/v indexed by kv head), dequantised value =
    code * descale.  ``rows``: optional list of (b, s, h) query rows.
    Returns (O f64[B, Sq, Hq, D], lse f64[B, Sq, Hq]).
    """
    B, Sq, Hq, D = q8.shape
    Sk, Hkv = k8.shape[1], k8.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Sq, Hq, v8.shape[3]))
    lse = np.full((B, Sq, Hq), NEG_INF)
    groups = {}
    if rows is None:
        for b in range(B):
            for h in range(Hq):
                groups[(b, h)] = np.arange(Sq)
    else:
        for b, s, h in rows:
            groups.setdefault((int(b), int(h)), []).append(int(s))
    for (b, h), ss in groups.items():
        ss = np.asarray(sorted(set(np.asarray(ss).tolist())), dtype=np.int64)
        hk = h // G
        Q = e4m3.decode(q8[b, ss, h]) * np.float64(q_descale[b, h])
        K = e4m3.decode(k8[b, :, hk]) * np.float64(k_descale[b, hk])
        V = e4m3.decode(v8[b, :, hk]) * np.float64(v_descale[b, hk])
        vis = causal_visible(Sq, Sk)[ss] if causal else None
        o, l = attend_rows(Q, K, V, scale, vis)
        O[b, ss, h] = o
        lse[b, ss, h] = l
    return O, lse
