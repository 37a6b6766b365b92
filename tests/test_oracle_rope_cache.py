"""Pins for the oracle's RoPE, slot mapping and cache-write modes (CPU only)."""
import numpy as np

from oracle import cache, e4m3, quant, rope
from quantized_paged_kv_varlen_gb300 import synth


def test_rope_table_closed_form():
    cos, sin = rope.cos_sin_table(50, 8, 1.0e4)
    assert cos.dtype == np.float32 and cos.shape == (50, 4)
    pos = np.arange(50, dtype=np.float64)
    # i = 0 has inverse frequency 1; i = 2 (2i/D = 1/2) has theta^(-1/2) = 0.01
    assert np.array_equal(cos[:, 0], np.cos(pos).astype(np.float32))
    assert np.array_equal(sin[:, 0], np.sin(pos).astype(np.float32))
    assert np.allclose(cos[:, 2], np.cos(pos * 0.01), atol=1e-7)
    assert np.all(cos[0] == 1) and np.all(sin[0] == 0)


def test_rope_identity_norm_and_direction():
    rng = np.random.default_rng(0)
    D = 16
    cos, sin = rope.cos_sin_table(64, D, 1.0e4)
    x = rng.standard_normal((64, 3, D)).astype(np.float32)
    pos = np.arange(64)
    y = rope.rotate(x, pos, cos, sin)
    assert np.array_equal(y[0], x[0])                      # position 0: identity
    pair_in = x[..., :D // 2].astype(np.float64) ** 2 + x[..., D // 2:].astype(np.float64) ** 2
    pair_out = y[..., :D // 2].astype(np.float64) ** 2 + y[..., D // 2:].astype(np.float64) ** 2
    assert np.allclose(pair_out, pair_in, rtol=2e-6, atol=1e-12)
    # one pair (1, 0) at angle a goes to (cos a, sin a): counter-clockwise, pairs (i, i+D/2)
    e = np.zeros((1, D), dtype=np.float32)
    e[0, 0] = 1.0
    r = rope.rotate(e, np.array([5]), cos, sin)
    assert r[0, 0] == cos[5, 0] and r[0, D // 2] == sin[5, 0]


def test_rope_dot_depends_only_on_relative_position():
    rng = np.random.default_rng(1)
    D = 32
    cos, sin = rope.cos_sin_table(400, D, 1.0e4)
    q = rng.standard_normal((1, D)).astype(np.float32)
    k = rng.standard_normal((1, D)).astype(np.float32)
    dots = []
    for m, n in [(10, 3), (107, 100), (307, 300)]:
        qm = rope.rotate(q, np.array([m]), cos, sin).astype(np.float64)
        kn = rope.rotate(k, np.array([n]), cos, sin).astype(np.float64)
        dots.append(float(qm[0] @ kn[0]))
    assert np.allclose(dots, dots[0], rtol=1e-4, atol=1e-4)


def test_rope_products_rounded_separately():
    """x'_i = fl(fl(x_i c) - fl(x_j s)): differs from a fused evaluation."""
    x = np.array([[1.0000001, 3.0000002]], dtype=np.float32)
    c = np.array([[0.7]], dtype=np.float32)
    s = np.array([[0.3000001]], dtype=np.float32)
    y = rope.rotate(x, np.array([0]), c, s)
    want0 = np.float32(np.float32(x[0, 0] * c[0, 0]) - np.float32(x[0, 1] * s[0, 0]))
    want1 = np.float32(np.float32(x[0, 1] * c[0, 0]) + np.float32(x[0, 0] * s[0, 0]))
    assert y[0, 0] == want0 and y[0, 1] == want1


def _walk_slots(lengths, start_pos, bt, ps):
    """Brute force: walk every request's tokens page by page."""
    out = []
    for b, L in enumerate(lengths):
        page_idx, off = divmod(int(start_pos[b]), ps)
        for _ in range(int(L)):
            out.append(int(bt[b][page_idx]) * ps + off)
            off += 1
            if off == ps:
                off = 0
                page_idx += 1
    return np.array(out, dtype=np.int32)


def test_slot_mapping_matches_page_walk():
    rng = np.random.default_rng(3)
    lengths = np.array([5, 0, 33, 16, 1])
    start = np.array([0, 7, 12, 16, 31])
    total = [int(s + L) for s, L in zip(start, lengths)]
    bt, _ = synth.page_tables(rng, total, 16)
    cu = np.cumsum(lengths)
    got = cache.slot_mapping(cu, start, bt, 16)
    assert np.array_equal(got, _walk_slots(lengths, start, bt, 16))


def test_fp8_write_bytes_and_untouched_slots():
    wl = synth.tiny_decode(0)
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, 16, wl.Hkv, wl.D
    fill = np.full((P, ps, H, D), 0x5A, dtype=np.uint8)
    sfill = np.full((P, ps, H), -7.0, dtype=np.float32)
    kp, vp, ks, vs, slots, _ = cache.write_fp8_token_head(
        k, v, wl.cu_seqlens, np.zeros(2, np.int64), wl.block_table, ps,
        fill, fill, sfill, sfill)
    kc, kscale = quant.quant_fp8_last_axis(k)
    flat = kp.reshape(P * ps, H, D)
    assert np.array_equal(flat[slots], kc)
    assert np.array_equal(ks.reshape(P * ps, H)[slots], kscale)
    untouched = np.setdiff1d(np.arange(P * ps), slots)
    assert np.all(flat[untouched] == 0x5A) and np.all(ks.reshape(-1, H)[untouched] == -7.0)
    # each token's absmax element sits at +-448
    deq = e4m3.decode(flat[slots]) * ks.reshape(P * ps, H)[slots][..., None]
    assert np.allclose(np.abs(deq).max(-1), np.abs(k).max(-1), rtol=2 ** -4)


def test_int8_block_scales_stay_inside_sequences():
    """Blocks never straddle two sequences: a loud and a quiet sequence get
    their own scales, and each block's absmax element is +-127."""
    lengths = np.array([130, 70])
    T, H, D = 200, 2, 8
    rng = np.random.default_rng(4)
    x = rng.standard_normal((T, H, D)).astype(np.float32)
    x[:130] *= 100.0
    cu = np.cumsum(lengths)
    codes, scales = cache.block128_quant(x, cu, 2)
    assert scales.shape == (2, 2, H)
    assert np.all(scales[1, 1] == 0)                       # sequence 1 has one block
    assert np.all(scales[0, 0] > 10 * scales[1, 0])
    for (lo, hi, b, blk) in [(0, 128, 0, 0), (128, 130, 0, 1), (130, 200, 1, 0)]:
        amax = np.abs(x[lo:hi]).max(axis=(0, 2))
        assert np.array_equal(scales[b, blk], (amax / np.float32(127)).astype(np.float32))
        assert np.all(np.abs(codes[lo:hi]).max(axis=(0, 2)) == 127)


def test_mla_row_layout_roundtrip():
    rng = np.random.default_rng(5)
    kv = synth.bf16_normal(rng, (9, 576))
    kv[3, :128] = 0.0                                       # a zero tile
    rows = cache.mla_pack_rows(kv)
    assert rows.shape == (9, 656)
    # rope part: bytes 512..640 are the bf16 bits, little-endian
    rope_bits = rows[:, 512:640].copy().view("<u2")
    assert np.array_equal(cache.bf16_value(rope_bits), kv[:, 512:].astype(np.float64))
    scales = rows[:, 640:].copy().view("<f4")
    amax = np.abs(kv[:, :512].reshape(9, 4, 128)).max(-1)
    assert np.array_equal(scales, (amax / np.float32(127)).astype(np.float32))
    assert scales[3, 0] == 0 and np.all(rows[3, :128] == 0)
    K, V = cache.mla_unpack_rows(rows)
    assert np.array_equal(K[:, 512:], kv[:, 512:].astype(np.float64))
    err = np.abs(V - kv[:, :512]).reshape(9, 4, 128)
    assert np.all(err <= scales[..., None].astype(np.float64) * 0.5 * (1 + 1e-5))
    assert np.array_equal(K[:, :512], V)


def test_bf16_round_matches_library_cast():
    """The oracle's nearest-even bf16 rounding against torch's CPU cast (a
    library routine), ties included; NaN stays NaN."""
    import torch
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(20000) * 3).astype(np.float32)
    hi = rng.integers(0, 0x7F7F, 2000).astype(np.uint32)
    ties = ((hi << 16) | 0x8000).view(np.float32) * np.where(rng.random(2000) < 0.5, 1, -1).astype(np.float32)
    x = np.concatenate([x, ties, np.array([np.inf, -np.inf, 0.0, -0.0, 3.4e38, np.nan], np.float32)])
    got = cache.bf16_round(x)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin].view(np.uint32), want[fin].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(want))


def _mla_case(rng, lengths, start):
    lengths = np.asarray(lengths, np.int32)
    bt, P = synth.page_tables(rng, lengths + np.asarray(start), 16)
    kv = synth.bf16_normal(rng, (int(lengths.sum()), 576))
    pool = np.zeros((P, 16, 1, 656), np.uint8)
    return kv, synth.inclusive_prefix(lengths), np.asarray(start, np.int64), bt, pool


def test_mla_rope_position_zero_is_identity():
    rng = np.random.default_rng(12)
    kv, cu, start, bt, pool = _mla_case(rng, [1, 1, 1], [0, 0, 0])
    cos, sin = rope.cos_sin_table(8, 64, 1.0e4)
    a, _ = cache.write_mla_rows(kv, cu, start, bt, 16, pool, cos, sin)
    b, _ = cache.write_mla_rows(kv, cu, start, bt, 16, pool)
    assert np.array_equal(a, b)


def test_mla_rope_quarter_turn_pins_pairs_and_sign():
    """A table with cos = 0, sin = 1 at every position maps the rope pair
    (x_i, x_{i+32}) to (-x_{i+32}, x_i) exactly; the nope bytes and scales
    do not change."""
    rng = np.random.default_rng(13)
    kv, cu, start, bt, pool = _mla_case(rng, [5, 3], [7, 0])
    cos = np.zeros((32, 32), np.float32)
    sin = np.ones((32, 32), np.float32)
    rot, _ = cache.write_mla_rows(kv, cu, start, bt, 16, pool, cos, sin)
    plain, slots = cache.write_mla_rows(kv, cu, start, bt, 16, pool)
    r = rot.reshape(-1, 656)[slots]
    p = plain.reshape(-1, 656)[slots]
    assert np.array_equal(r[:, :512], p[:, :512]) and np.array_equal(r[:, 640:], p[:, 640:])
    got = cache.bf16_value(r[:, 512:640].copy().view("<u2"))
    x = kv[:, 512:].astype(np.float64)
    assert np.array_equal(got[:, :32], -x[:, 32:]) and np.array_equal(got[:, 32:], x[:, :32])


def test_mla_rope_dot_depends_on_relative_position():
    """Rotated query and key rope parts (decoded from the rows, bf16) give
    the same dot product when both positions shift by the same amount, to
    the bf16 rounding of the stored values."""
    rng = np.random.default_rng(14)
    cos, sin = rope.cos_sin_table(512, 64, 1.0e4)
    q = synth.bf16_normal(rng, (1, 576))
    kv = synth.bf16_normal(rng, (1, 576))
    cu = np.array([1], np.int32)

    def dot(m, n):
        qr = cache.mla_rope(q, cu, np.array([m]), cos, sin)[0, 512:].astype(np.float64)
        pool = np.zeros((40, 16, 1, 656), np.uint8)
        bt = np.arange(40, dtype=np.int32)[None]
        rows, slots = cache.write_mla_rows(kv, cu, np.array([n]), bt, 16, pool, cos, sin)
        k, _ = cache.mla_unpack_rows(rows.reshape(-1, 656)[slots])
        return float(qr @ k[0, 512:])
    for m, n, d in [(5, 2, 100), (300, 17, 150), (9, 9, 400)]:
        assert abs(dot(m, n) - dot(m + d, n + d)) < 0.1
    assert abs(dot(5, 2) - dot(5, 100)) > 0.1          # and does depend on the offset


def test_k_smoothing_mean_is_exact_and_order_free():
    """The smoothing mean is the exact mean of the 2^-24-rounded keys: within
    2^-25 (plus float32 rounding) of the float64 mean, and bit-identical when
    a sequence's tokens are permuted; values beyond 2^15 are clamped."""
    rng = np.random.default_rng(31)
    lengths = [130, 1, 257]
    T = sum(lengths)
    x = (rng.standard_normal((T, 3, 128)) * 4).astype(np.float32)
    x[5, 0, :7] = np.float32(1e-9)                            # below the fixed-point step
    cu = synth.inclusive_prefix(lengths)
    km = cache.k_smoothing_mean(x, cu)
    begin = [0, 130, 131]
    for b, n in enumerate(lengths):
        mean = x[begin[b]:begin[b] + n].astype(np.float64).mean(axis=0)
        bound = 2.0 ** -25 + np.spacing(np.abs(mean).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(km[b].astype(np.float64) - mean) <= bound)
    perm = np.concatenate([rng.permutation(130), 130 + np.arange(1), 131 + rng.permutation(257)])
    assert np.array_equal(cache.k_smoothing_mean(x[perm], cu).view(np.uint32), km.view(np.uint32))
    big = x.copy()
    big[0, 0, 0] = np.float32(1e6)
    kb = cache.k_smoothing_mean(big, cu)
    want = (np.rint(np.clip(big[:130, 0, 0].astype(np.float64), -32768, 32768) * 2.0 ** 24).sum()
            / (130 * 2.0 ** 24))
    assert kb[0, 0, 0] == np.float32(want)


def test_k_smoothing_shrinks_int8_error_with_a_key_offset():
    """Keys with a common per-head offset on the slowest-rotating RoPE pairs
    (channels the rotation barely moves over the sequence) lose most of their
    resolution to block-INT8; subtracting the mean first keeps attention
    much closer to exact float64 attention on the rotated keys, and the
    cache otherwise equals the unsmoothed one (V, Q)."""
    from oracle import attention as oatt
    rng = np.random.default_rng(32)
    lengths = np.array([300, 170], np.int32)
    T, H, D, ps = int(lengths.sum()), 2, 128, 64
    q = synth.bf16_normal(rng, (T, H, D))
    off = np.zeros((H, D), np.float32)
    off[:, 56:64] = 12.0
    off[:, 120:128] = 12.0
    k = cache.bf16_round((rng.standard_normal((T, H, D)) + off).astype(np.float32))
    v = synth.bf16_normal(rng, (T, H, D))
    bt, P = synth.page_tables(rng, lengths, ps)
    cu = synth.inclusive_prefix(lengths)
    cos, sin = rope.cos_sin_table(512, D, 1.0e4)
    nb = 3
    args = (q, k, v, cu, bt, ps, cos, sin, nb, np.zeros((P, ps, H, D), np.int8),
            np.zeros((P, ps, H, D), np.uint16))
    plain = cache.write_int8_block128_rope(*args)
    smooth = cache.write_int8_block128_rope(*args, smooth_k=True)
    km = smooth[6]
    assert np.array_equal(plain[1], smooth[1]) and np.array_equal(plain[3], smooth[3])
    b_of, p_of = cache.token_positions(cu, np.zeros(2, np.int64))
    q_rot = rope.rotate(q, p_of, cos, sin).astype(np.float64)
    k_rot = rope.rotate(k, p_of, cos, sin).astype(np.float64)
    scale = 1.0 / np.sqrt(D)
    errs = []
    for out in (plain, smooth):
        O, _ = oatt.paged_prefill_int8(out[3], out[4], out[0], out[2], out[1], bt, cu, lengths, scale)
        err = 0.0
        for b, (lo, n) in enumerate([(0, 300), (300, 170)]):
            for h in range(H):
                vis = oatt.causal_visible(n, n)
                ref, _ = oatt.attend_rows(q_rot[lo:lo + n, h], k_rot[lo:lo + n, h],
                                          cache.bf16_value(cache.bf16_bits(v[lo:lo + n, h])), scale, vis)
                err = max(err, np.abs(O[lo:lo + n, h] - ref).max())
        errs.append(err)
    assert errs[1] < 0.5 * errs[0], errs
    # the codes are those of the shifted keys
    assert np.all(np.abs(km[:, :, 120:128] - 12.0) < 0.6)


def test_v_channel_fp8_scales_per_sequence_head_channel():
    """FP8 V: one scale per (sequence, head, channel) from that channel's
    absmax over the sequence (checked by explicit loops), the absmax element
    coding to +-448, a channel scaled by a power of two keeping its codes,
    and an all-zero channel giving scale 0 and zero codes."""
    rng = np.random.default_rng(33)
    lengths = [5, 9]
    v = synth.bf16_normal(rng, (14, 2, 8))
    v[5:, 1, 3] = 0.0
    v[:5, 0, 2] *= np.float32(8.0)
    cu = synth.inclusive_prefix(lengths)
    codes, scales = cache.v_channel_fp8(v, cu)
    for b, (lo, hi) in enumerate([(0, 5), (5, 14)]):
        for h in range(2):
            for c in range(8):
                amax = max(abs(float(x)) for x in v[lo:hi, h, c])
                assert scales[b, h, c] == np.float32(np.float32(amax) / np.float32(448.0))
                if amax > 0:
                    j = lo + int(np.argmax(np.abs(v[lo:hi, h, c])))
                    assert e4m3.decode(codes[j, h, c]) == (448.0 if v[j, h, c] > 0 else -448.0)
    assert scales[1, 1, 3] == 0 and np.all(codes[5:, 1, 3] == 0)
    v2 = v.copy()
    v2[:5, 0, 2] /= np.float32(8.0)
    codes2, scales2 = cache.v_channel_fp8(v2, cu)
    assert np.array_equal(codes2[:5, 0, 2], codes[:5, 0, 2])
    assert scales2[0, 0, 2] * 8 == scales[0, 0, 2]


def test_prefill_with_fp8_v_factors_the_channel_scale():
    """O over FP8 V is (attention over the raw E4M3 values) times each
    channel's scale: the per-channel scale factors out of P.V."""
    from oracle import attention as oatt
    rng = np.random.default_rng(34)
    lengths = np.array([70, 150], np.int32)
    T, H, D, ps = int(lengths.sum()), 2, 128, 64
    q, k, v = (synth.bf16_normal(rng, (T, H, D)) for _ in range(3))
    bt, P = synth.page_tables(rng, lengths, ps)
    cu = synth.inclusive_prefix(lengths)
    cos, sin = rope.cos_sin_table(256, D, 1.0e4)
    out = cache.write_int8_block128_rope(q, k, v, cu, bt, ps, cos, sin, 2,
                                         np.zeros((P, ps, H, D), np.int8),
                                         np.zeros((P, ps, H, D), np.uint8), v_fp8=True)
    kp, vp, ks, q8, qs, slots, vscale = out
    scale = 1.0 / np.sqrt(D)
    O, lse = oatt.paged_prefill_int8(q8, qs, kp, ks, vp, bt, cu, lengths, scale, v_scale=vscale)
    ones = np.ones_like(vscale)
    O1, lse1 = oatt.paged_prefill_int8(q8, qs, kp, ks, vp, bt, cu, lengths, scale, v_scale=ones)
    b_of, _ = cache.token_positions(cu, np.zeros(2, np.int64))
    assert np.allclose(O, O1 * vscale[b_of].astype(np.float64), rtol=1e-12, atol=1e-14)
    assert np.array_equal(lse, lse1)
    # and against the bf16 V it quantises: each value moves by at most 2^-4 of
    # itself, so O by at most 2^-4 of the channel's absmax (448 * scale)
    plain = cache.write_int8_block128_rope(q, k, v, cu, bt, ps, cos, sin, 2,
                                           np.zeros((P, ps, H, D), np.int8),
                                           np.zeros((P, ps, H, D), np.uint16))
    Ob, _ = oatt.paged_prefill_int8(q8, qs, kp, ks, plain[1], bt, cu, lengths, scale)
    bound = 2.0 ** -4 * 448.0 * vscale[b_of].astype(np.float64) * (1 + 1e-6)
    assert np.all(np.abs(O - Ob) <= bound)
