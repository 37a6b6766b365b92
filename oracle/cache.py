"""The cache-write step: optional RoPE, quantise, append into pages.

Test infrastructure only (see oracle/__init__.py).

Layout ("KvQuantSparseFlashAttention" README, 参数说明 rows key / block_table
/ actual_seq_lengths_query): pages are PA_BSND ``[block_num, block_size,
KV_N, KV_D]``; ``block_table[b, j]`` is the page holding logical tokens
``[j*block_size, (j+1)*block_size)`` of sequence b; TND query prefix sums are
inclusive, B elements (batch b spans ``[cu[b-1], cu[b])`` with cu[-1] = 0).
RoPE fused into the write follows "[Feature] Sage Attention Support Varlen &
write kv cache BF16/FP16", Description item 1.

A token t of sequence b at position p = start_pos[b] + (t - begin_b) goes to
pool row ``block_table[b, p // ps] * ps + p % ps`` (its "slot").

Three modes:
  fp8_token_head   K and V -> E4M3 with one fp32 scale per (token, head);
                   optional RoPE on q and k first.
  int8_block128    RoPE on q and k, then Q and K -> INT8 with one fp32 scale
                   per (sequence, 128-token logical block, head); V stored
                   as bf16 unchanged.  Whole sequences only (start_pos 0).
                   Optional K smoothing (the role of the Sage varlen
                   "segment_mean" kernel): the per-(sequence, head) mean of
                   the rotated keys is subtracted before quantising, which
                   shifts every logit of a query row by the same amount.
                   Optional FP8 V (Sage-style, for an FP8 P.V product): V
                   -> E4M3 with one fp32 scale per (sequence, head,
                   channel), the channel's absmax over the sequence / 448.
  mla_row          one 656-byte row per token: 512 INT8 nope codes with one
                   fp32 scale per 128-wide tile, the 64-wide rope part as
                   bf16, then the 4 scales (README, 参数说明 row key:
                   "512+64*2+4*4").  Optionally the rope part (and the
                   query's) is rotated first: rotate-half over its 64 dims,
                   the float32 result rounded to bf16 to nearest-even.
"""
import numpy as np

from . import quant, rope

F32 = np.float32


def seq_bounds(cu_seqlens_inclusive: np.ndarray):
    """Inclusive B-element prefix sums -> (begin[B], end[B])."""
    cu = np.asarray(cu_seqlens_inclusive, dtype=np.int64)
    begin = np.concatenate([[0], cu[:-1]])
    return begin, cu


def token_positions(cu_seqlens_inclusive, start_pos):
    """Per token: (sequence index b, position p within its sequence)."""
    begin, end = seq_bounds(cu_seqlens_inclusive)
    T = int(end[-1]) if len(end) else 0
    b_of = np.zeros(T, dtype=np.int64)
    p_of = np.zeros(T, dtype=np.int64)
    for b in range(len(begin)):
        n = int(end[b] - begin[b])
        b_of[begin[b]:end[b]] = b
        p_of[begin[b]:end[b]] = int(start_pos[b]) + np.arange(n)
    return b_of, p_of


def slot_mapping(cu_seqlens_inclusive, start_pos, block_table, page_size):
    """int32 pool row of every new token."""
    b_of, p_of = token_positions(cu_seqlens_inclusive, start_pos)
    bt = np.asarray(block_table, dtype=np.int64)
    page = bt[b_of, p_of // page_size]
    return (page * page_size + p_of % page_size).astype(np.int32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values that are bf16-exact."""
    u = np.asarray(x, dtype=F32).view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), returned
    as float32; NaN stays NaN, infinities stay infinite."""
    u = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(np.asarray(x, dtype=F32))
    r = np.where(nan, (u | 0x400000) >> 16 << 16, r)
    return r.astype(np.uint32).view(F32)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """float64 values of uint16 bf16 bit patterns (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(F32).astype(np.float64)


def write_fp8_token_head(k, v, cu_seqlens_q, start_pos, block_table, page_size,
                         k_pool, v_pool, k_scale_pool, v_scale_pool,
                         q=None, cos=None, sin=None, layout="NHD"):
    """FP8 per-(token, head) write.  k, v: float32 [T, H, D] (bf16 values).

    Pools are updated in place copies and returned:
    (k_pool, v_pool, k_scale_pool, v_scale_pool, slots, q_rot or None).
    With cos/sin given, q and k are rotated first (v never is).  layout
    "HND" takes K/V pools [P, H, page_size, D] (token at page offset o of
    head h in [page, h, o]); the scale pools stay [P, page_size, H].
    """
    k = np.asarray(k, dtype=F32)
    v = np.asarray(v, dtype=F32)
    q_rot = None
    if cos is not None:
        _, p_of = token_positions(cu_seqlens_q, start_pos)
        k = rope.rotate(k, p_of, cos, sin)
        if q is not None:
            q_rot = rope.rotate(np.asarray(q, dtype=F32), p_of, cos, sin)
    slots = slot_mapping(cu_seqlens_q, start_pos, block_table, page_size)
    kc, ks = quant.quant_fp8_last_axis(k)
    vc, vs = quant.quant_fp8_last_axis(v)
    if layout == "HND":
        P, H, ps, D = k_pool.shape
        b_of, p_of = token_positions(cu_seqlens_q, start_pos)
        page = np.asarray(block_table, dtype=np.int64)[b_of, p_of // page_size]
        off = p_of % page_size
        k_pool, v_pool = k_pool.copy(), v_pool.copy()
        k_scale_pool, v_scale_pool = k_scale_pool.copy(), v_scale_pool.copy()
        for hh in range(H):
            k_pool[page, hh, off] = kc[:, hh]
            v_pool[page, hh, off] = vc[:, hh]
            k_scale_pool[page, off, hh] = ks[:, hh]
            v_scale_pool[page, off, hh] = vs[:, hh]
        return k_pool, v_pool, k_scale_pool, v_scale_pool, slots, q_rot
    P, ps, H, D = k_pool.shape
    k_pool = k_pool.copy().reshape(P * ps, H, D)
    v_pool = v_pool.copy().reshape(P * ps, H, D)
    k_scale_pool = k_scale_pool.copy().reshape(P * ps, H)
    v_scale_pool = v_scale_pool.copy().reshape(P * ps, H)
    k_pool[slots] = kc
    v_pool[slots] = vc
    k_scale_pool[slots] = ks
    v_scale_pool[slots] = vs
    return (k_pool.reshape(P, ps, H, D), v_pool.reshape(P, ps, H, D),
            k_scale_pool.reshape(P, ps, H), v_scale_pool.reshape(P, ps, H),
            slots, q_rot)


def block128_quant(x_rot, cu_seqlens_q, num_blocks):
    """INT8 per-(sequence, 128-token block, head) quantisation of [T, H, D].

    Returns (codes int8 [T, H, D], scales f32 [B, num_blocks, H]); blocks past
    a sequence's end keep scale 0.
    """
    x_rot = np.asarray(x_rot, dtype=F32)
    begin, end = seq_bounds(cu_seqlens_q)
    B = len(begin)
    T, H, D = x_rot.shape
    codes = np.zeros((T, H, D), dtype=np.int8)
    scales = np.zeros((B, num_blocks, H), dtype=F32)
    for b in range(B):
        n = int(end[b] - begin[b])
        for blk in range((n + 127) // 128):
            lo = int(begin[b]) + blk * 128
            hi = min(int(begin[b]) + (blk + 1) * 128, int(end[b]))
            seg = x_rot[lo:hi]                                 # [n_blk, H, D]
            amax = np.max(np.abs(seg), axis=(0, 2))            # [H]
            s = quant.absmax_scale(amax, quant.INT8_QMAX)      # [H]
            scales[b, blk] = s
            codes[lo:hi] = quant.quant_int8(seg, s[None, :, None])
    return codes, scales


# K smoothing mean: each rotated key value is clamped to [-2^15, 2^15] and
# rounded (nearest-even) to a multiple of 2^-24; the sum over the sequence
# is then exact (int64), so the mean does not depend on summation order:
#   k_mean = float32( float64(sum) / (n * 2^24) )
K_MEAN_FRAC_BITS = 24
K_MEAN_CLAMP = 32768.0


def k_smoothing_mean(k_rot, cu_seqlens_q):
    """Per-(sequence, head) mean of rotated keys k_rot float32 [T, H, D]:
    float32 [B, H, D] (zero for an empty sequence)."""
    k_rot = np.asarray(k_rot, dtype=F32)
    begin, end = seq_bounds(cu_seqlens_q)
    T, H, D = k_rot.shape
    km = np.zeros((len(begin), H, D), dtype=F32)
    one = float(2 ** K_MEAN_FRAC_BITS)
    for b in range(len(begin)):
        n = int(end[b] - begin[b])
        if n == 0:
            continue
        seg = np.clip(k_rot[begin[b]:end[b]].astype(np.float64), -K_MEAN_CLAMP, K_MEAN_CLAMP)
        total = np.rint(seg * one).astype(np.int64).sum(axis=0)
        km[b] = (total.astype(np.float64) / (n * one)).astype(F32)
    return km


def v_channel_fp8(v, cu_seqlens_q):
    """Per-(sequence, head, channel) E4M3 quantisation of V float32 [T, H, D]:
    scale = absmax over the sequence's tokens / 448 (float32 division), codes
    RNE-satfinite of v / scale.  Returns (codes u8 [T, H, D], scale f32
    [B, H, D]); a channel that is all zero has scale 0 and zero codes."""
    v = np.asarray(v, dtype=F32)
    begin, end = seq_bounds(cu_seqlens_q)
    T, H, D = v.shape
    codes = np.zeros((T, H, D), dtype=np.uint8)
    scales = np.zeros((len(begin), H, D), dtype=F32)
    for b in range(len(begin)):
        if end[b] == begin[b]:
            continue
        seg = v[begin[b]:end[b]]
        s = quant.absmax_scale(np.max(np.abs(seg), axis=0), quant.FP8_QMAX)
        scales[b] = s
        codes[begin[b]:end[b]] = quant.quant_fp8(seg, s[None])
    return codes, scales


def write_int8_block128_rope(q, k, v, cu_seqlens_q, block_table, page_size,
                             cos, sin, num_blocks, k_pool, v_pool_bits, smooth_k=False,
                             v_fp8=False):
    """Sage-style write: RoPE(q, k), block-INT8 Q and K, bf16 V into pages.

    q, k, v: float32 [T, H, D] (bf16 values).  Whole sequences (positions
    start at 0).  Returns (k_pool int8, v_pool_bits uint16, k_scale
    [B, nb, H], q8 int8 [T, H, D], q_scale [B, nb, H], slots), and with
    smooth_k the keys quantised are k_rot - k_mean (float32 subtraction)
    and k_mean float32 [B, H, D] is appended; with v_fp8 the V pool holds
    E4M3 codes (u8) and the per-channel scales float32 [B, H, D] are appended
    last.
    """
    B = len(cu_seqlens_q)
    start = np.zeros(B, dtype=np.int64)
    b_of, p_of = token_positions(cu_seqlens_q, start)
    q_rot = rope.rotate(np.asarray(q, dtype=F32), p_of, cos, sin)
    k_rot = rope.rotate(np.asarray(k, dtype=F32), p_of, cos, sin)
    km = None
    if smooth_k:
        km = k_smoothing_mean(k_rot, cu_seqlens_q)
        k_rot = (k_rot - km[b_of]).astype(F32)
    q8, q_scale = block128_quant(q_rot, cu_seqlens_q, num_blocks)
    k8, k_scale = block128_quant(k_rot, cu_seqlens_q, num_blocks)
    slots = slot_mapping(cu_seqlens_q, start, block_table, page_size)
    P, ps, H, D = k_pool.shape
    k_pool = k_pool.copy().reshape(P * ps, H, D)
    v_pool_bits = v_pool_bits.copy().reshape(P * ps, H, D)
    k_pool[slots] = k8
    extra = (km,) if smooth_k else ()
    if v_fp8:
        v_codes, v_scale = v_channel_fp8(v, cu_seqlens_q)
        v_pool_bits[slots] = v_codes
        extra = extra + (v_scale,)
    else:
        v_pool_bits[slots] = bf16_bits(v)
    out = (k_pool.reshape(P, ps, H, D), v_pool_bits.reshape(P, ps, H, D),
           k_scale, q8, q_scale, slots)
    return out + extra


MLA_NOPE = 512
MLA_ROPE = 64
MLA_TILE = 128
MLA_ROW_BYTES = MLA_NOPE + 2 * MLA_ROPE + 4 * (MLA_NOPE // MLA_TILE)   # 656


def mla_pack_rows(kv):
    """[T, 576] float32 (bf16 values) -> [T, 656] uint8 combined rows."""
    kv = np.asarray(kv, dtype=F32)
    T = kv.shape[0]
    nope = kv[:, :MLA_NOPE].reshape(T, MLA_NOPE // MLA_TILE, MLA_TILE)
    codes, scales = quant.quant_int8_last_axis(nope)            # [T,4,128], [T,4]
    rows = np.zeros((T, MLA_ROW_BYTES), dtype=np.uint8)
    rows[:, :MLA_NOPE] = codes.reshape(T, MLA_NOPE).view(np.uint8)
    rows[:, MLA_NOPE:MLA_NOPE + 2 * MLA_ROPE] = (
        bf16_bits(kv[:, MLA_NOPE:]).astype("<u2").view(np.uint8).reshape(T, -1))
    rows[:, MLA_NOPE + 2 * MLA_ROPE:] = (
        scales.astype("<f4").view(np.uint8).reshape(T, -1))
    return rows


def mla_unpack_rows(rows):
    """[n, 656] uint8 -> (K f64 [n, 576] dequantised, V f64 [n, 512])."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    codes = rows[:, :MLA_NOPE].view(np.int8).reshape(n, MLA_NOPE // MLA_TILE, MLA_TILE)
    rope_bits = rows[:, MLA_NOPE:MLA_NOPE + 2 * MLA_ROPE].copy().view("<u2")
    scales = rows[:, MLA_NOPE + 2 * MLA_ROPE:].copy().view("<f4").astype(np.float64)
    nope = quant.dequant_int8(codes, scales[:, :, None]).reshape(n, MLA_NOPE)
    k = np.concatenate([nope, bf16_value(rope_bits)], axis=1)
    return k, nope


def mla_rope(x, cu_seqlens_q, start_pos, cos, sin):
    """Rotate the 64-wide rope part (last 64 of 576 dims) of every row of
    x float32 [T, 576] or [T, N, 576] at its token's position; the rotated
    values are rounded to bf16.  cos/sin: float32 [max_pos, 32]."""
    x = np.array(x, dtype=F32)
    _, p_of = token_positions(cu_seqlens_q, start_pos)
    rot = rope.rotate(x[..., MLA_NOPE:], p_of, cos, sin)
    x[..., MLA_NOPE:] = bf16_round(rot)
    return x


def write_mla_rows(kv, cu_seqlens_q, start_pos, block_table, page_size, pool,
                   cos=None, sin=None):
    """MLA combined-row write of [T, 576] tokens into pool [P, bs, 1, 656];
    with cos/sin the rope part is rotated first (mla_rope)."""
    if cos is not None:
        kv = mla_rope(kv, cu_seqlens_q, start_pos, cos, sin)
    slots = slot_mapping(cu_seqlens_q, start_pos, block_table, page_size)
    P, bs, one, W = pool.shape
    pool = pool.copy().reshape(P * bs, W)
    pool[slots] = mla_pack_rows(kv)
    return pool.reshape(P, bs, one, W), slots
