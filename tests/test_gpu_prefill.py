"""GPU parity: the Sage-style INT8 cache write (bit-exact) and the varlen
INT8-QK paged prefill against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import cache as ocache
from oracle import rope as orope
from quantized_paged_kv_varlen_gb300 import synth
from tests.gpu_util import (REL_L2_FP8_P, assert_attention_close,
                            assert_lse_close, bf16_to_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# --------------------------------------------------------- INT8 cache write

def _gpu_write(lib, q, k, v, lengths, bt, P, ps, cos, sin):
    """GPU RoPE + block-INT8 write of whole sequences; tables are inputs."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = len(lengths)
    nb = max(1, (int(max(lengths)) + 127) // 128)
    k_pool = torch.full((P, ps, Hkv, D), 99, dtype=torch.int8, device=DEV)
    v_pool = torch.full((P, ps, Hkv, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ks = torch.full((B, nb, Hkv), float("nan"), dtype=torch.float32, device=DEV)
    qs = torch.full((B, nb, Hq), float("nan"), dtype=torch.float32, device=DEV)
    q8 = torch.full((T, Hq, D), 99, dtype=torch.int8, device=DEV)
    slots = torch.full((T,), -1, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cu = _t(synth.inclusive_prefix(lengths))
    lib.write_cache_int8_block128_rope(
        _t(q).to(torch.bfloat16), _t(k).to(torch.bfloat16), _t(v).to(torch.bfloat16), cu, _t(bt),
        int(max(lengths)), _t(cos), _t(sin), k_pool, v_pool, ks, q8, qs, slot_mapping=slots,
        error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return dict(k_pool=k_pool, v_pool=v_pool, ks=ks, qs=qs, q8=q8, slots=slots, cu=cu, nb=nb)


def test_write_cache_int8_bit_exact(lib):
    lengths = np.array([1, 130, 300], dtype=np.int32)
    wl = synth.varlen_prefill(seed=11, H=4, page_size=64, lengths=lengths)
    Hkv = 2
    k, v = wl.k[:, :Hkv], wl.v[:, :Hkv]
    cos, sin = orope.cos_sin_table(512, 128, wl.theta)
    d = _gpu_write(lib, wl.q, k, v, lengths, wl.block_table, wl.num_pages, 64, cos, sin)
    P, ps, D = wl.num_pages, 64, 128
    kp0 = np.full((P, ps, Hkv, D), 99, np.int8)
    vp0 = np.full((P, ps, Hkv, D), 0x7FC0, np.uint16)
    kp, vp, kscale, q8, qscale, slots = ocache.write_int8_block128_rope(
        wl.q, k, v, wl.cu_seqlens, wl.block_table, ps, cos, sin, d["nb"], kp0, vp0)
    assert np.array_equal(d["slots"].cpu().numpy(), slots)
    got_k = d["k_pool"].cpu().numpy().reshape(P * ps, Hkv, D)
    got_v = d["v_pool"].cpu().view(torch.int16).numpy().view(np.uint16).reshape(P * ps, Hkv, D)
    assert np.array_equal(got_k[slots], kp.reshape(P * ps, Hkv, D)[slots])
    assert np.array_equal(got_v[slots], vp.reshape(P * ps, Hkv, D)[slots])
    assert np.array_equal(d["q8"].cpu().numpy(), q8)
    # scales of the blocks a sequence has; the rest stay as the caller left them
    for b, L in enumerate(lengths):
        n = (int(L) + 127) // 128
        assert np.array_equal(_u32(d["ks"].cpu().numpy()[b, :n]), _u32(kscale[b, :n]))
        assert np.array_equal(_u32(d["qs"].cpu().numpy()[b, :n]), _u32(qscale[b, :n]))


def test_write_cache_int8_smooth_k_bit_exact_and_attention(lib):
    """K smoothing: codes, block scales and the per-(sequence, head) mean
    bit-exact; the prefill over the smoothed cache matches the oracle on the
    same cache, and (the softmax being shift-invariant) the oracle on the
    unsmoothed cache to the INT8 tolerance."""
    rng = np.random.default_rng(51)
    lengths = np.array([1, 300, 129], dtype=np.int32)
    T, Hq, Hkv, D, ps = int(lengths.sum()), 4, 2, 128, 64
    q = synth.bf16_normal(rng, (T, Hq, D))
    off = np.zeros((Hkv, D), np.float32)
    off[:, 120:128] = 9.0
    k = ocache.bf16_round((rng.standard_normal((T, Hkv, D)) + off).astype(np.float32))
    v = synth.bf16_normal(rng, (T, Hkv, D))
    bt, P = synth.page_tables(rng, lengths, ps)
    cos, sin = orope.cos_sin_table(512, 128, 1.0e4)
    B, nb = 3, 3
    k_pool = torch.full((P, ps, Hkv, D), 99, dtype=torch.int8, device=DEV)
    v_pool = torch.zeros((P, ps, Hkv, D), dtype=torch.bfloat16, device=DEV)
    ks = torch.full((B, nb, Hkv), float("nan"), dtype=torch.float32, device=DEV)
    qs = torch.full((B, nb, Hq), float("nan"), dtype=torch.float32, device=DEV)
    q8 = torch.zeros((T, Hq, D), dtype=torch.int8, device=DEV)
    km = torch.full((B, Hkv, D), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cu = synth.inclusive_prefix(lengths)
    lib.write_cache_int8_block128_rope(
        _t(q).to(torch.bfloat16), _t(k).to(torch.bfloat16), _t(v).to(torch.bfloat16), _t(cu), _t(bt),
        300, _t(cos), _t(sin), k_pool, v_pool, ks, q8, qs, error_word=err, k_mean=km)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp0 = np.full((P, ps, Hkv, D), 99, np.int8)
    vp0 = np.zeros((P, ps, Hkv, D), np.uint16)
    kp, vp, kscale, q8w, qscale, slots, kmw = ocache.write_int8_block128_rope(
        q, k, v, cu, bt, ps, cos, sin, nb, kp0, vp0, smooth_k=True)
    assert np.array_equal(_u32(km.cpu().numpy()), _u32(kmw))
    got_k = k_pool.cpu().numpy().reshape(P * ps, Hkv, D)
    assert np.array_equal(got_k[slots], kp.reshape(P * ps, Hkv, D)[slots])
    assert np.array_equal(q8.cpu().numpy(), q8w)
    for b, L in enumerate(lengths):
        n = (int(L) + 127) // 128
        assert np.array_equal(_u32(ks.cpu().numpy()[b, :n]), _u32(kscale[b, :n]))
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=DEV)
    lib.prefill_paged(q8, qs, k_pool, ks, v_pool, _t(bt), _t(cu), _t(lengths), causal=True,
                      out=out, lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    scale = 1.0 / np.sqrt(128.0)
    want_o, want_lse = oatt.paged_prefill_int8(q8w, qscale, kp, kscale, vp, bt, cu, lengths, scale)
    assert_attention_close(bf16_to_f64(out), want_o)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)
    plain = ocache.write_int8_block128_rope(q, k, v, cu, bt, ps, cos, sin, nb, kp0, vp0)
    o_plain, _ = oatt.paged_prefill_int8(plain[3], plain[4], plain[0], plain[2], plain[1], bt, cu,
                                         lengths, scale)
    assert np.abs(bf16_to_f64(out) - o_plain).max() < 0.1


def test_rope_table_matches_oracle(lib):
    """The library's table (double precision on the device, rounded to
    float) against the oracle's numpy float64 table: equal or 1 ulp apart."""
    cos, sin = lib.rope_table(1.0e4, 4096, 128)
    ocos, osin = orope.cos_sin_table(4096, 128, 1.0e4)
    for g, w in ((cos.cpu().numpy(), ocos), (sin.cpu().numpy(), osin)):
        du = np.abs(_u32(g).astype(np.int64) - _u32(w).astype(np.int64))
        same_sign = np.sign(g) == np.sign(w)
        assert np.all((du <= 1) | (~same_sign & (np.abs(g) < 1e-6)))
        assert np.mean(du == 0) > 0.99


# ------------------------------------------------------------------ prefill

def _random_case(seed, Lq, Lk, Hq, Hkv, ps, qmag=3.0, kmag=3.0):
    """Random INT8 Q/K codes with block scales and bf16 V in a permuted pool."""
    rng = np.random.default_rng((seed, 77))
    Lq = np.asarray(Lq, dtype=np.int32)
    Lk = np.asarray(Lk, dtype=np.int32)
    B, T = len(Lq), int(Lq.sum())
    nb = max(1, (int(max(Lq.max(), Lk.max())) + 127) // 128)
    q8 = rng.integers(-127, 128, (T, Hq, 128), dtype=np.int8)
    qs = (rng.uniform(0.5, 1.5, (B, nb, Hq)) * qmag / 127).astype(np.float32)
    bt, P = synth.page_tables(rng, Lk, ps, extra_pages=2)
    k_pool = rng.integers(-127, 128, (P, ps, Hkv, 128), dtype=np.int8)
    ks = (rng.uniform(0.5, 1.5, (B, nb, Hkv)) * kmag / 127).astype(np.float32)
    v_bits = ocache.bf16_bits(synth.bf16_normal(rng, (P, ps, Hkv, 128)))
    return dict(q8=q8, qs=qs, k_pool=k_pool, ks=ks, v_bits=v_bits, bt=bt,
                cu=synth.inclusive_prefix(Lq), Lk=Lk)


def _run_prefill(lib, c, causal, scale=None):
    T, Hq, _ = c["q8"].shape
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((T, Hq, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    v_pool = _t(c["v_bits"].view(np.int16)).view(torch.bfloat16)
    lib.prefill_paged(_t(c["q8"]), _t(c["qs"]), _t(c["k_pool"]), _t(c["ks"]), v_pool, _t(c["bt"]),
                      _t(c["cu"]), _t(c["Lk"]), sm_scale=scale, causal=causal, out=out, lse=lse,
                      error_word=err)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), int(err.item())


def _oracle(c, causal, scale=1.0 / np.sqrt(128.0), rows=None):
    return oatt.paged_prefill_int8(c["q8"], c["qs"], c["k_pool"], c["ks"], c["v_bits"], c["bt"],
                                   c["cu"], c["Lk"], scale, causal, rows=rows)


@pytest.mark.parametrize("Lq,Lk,Hq,Hkv,ps,causal", [
    ([1, 130, 300], [1, 130, 300], 2, 2, 64, True),        # ragged tails, one-token sequence
    ([200, 0, 385], [200, 0, 385], 4, 2, 16, True),        # an empty sequence, GQA 2:1
    ([77, 128, 1], [300, 128, 513], 4, 1, 32, True),       # cached prefix: L_q < L_kv
    ([300, 50], [40, 0], 2, 2, 64, True),                  # L_q > L_kv: leading rows see nothing
    ([130, 257], [390, 100], 2, 1, 128, False),            # no mask
    ([600], [600], 2, 2, 256, True),                       # pages longer than a tile
    ([900, 300], [1000, 300], 4, 2, 384, True),            # three tiles per page
    ([640, 520], [640, 520], 1, 1, 64, True),              # several q tiles: pairs (0,4) (1,3) (2)
])
def test_prefill_shapes(lib, Lq, Lk, Hq, Hkv, ps, causal):
    c = _random_case(sum(Lq) + 7 * ps, Lq, Lk, Hq, Hkv, ps)
    got_o, got_lse, err = _run_prefill(lib, c, causal)
    assert err == 0
    want_o, want_lse = _oracle(c, causal)
    assert_attention_close(got_o, want_o)
    assert_lse_close(got_lse, want_lse)
    none = np.isneginf(want_lse)
    assert np.all(got_o[none] == 0.0)



@pytest.mark.parametrize("Lq,Lk,Hq,Hkv,causal", [
    ([1, 130, 300], [1, 130, 300], 2, 2, True),      # sequences back to back, ragged tails
    ([77, 128, 1], [300, 128, 513], 4, 1, True),     # cached prefixes, GQA 4:1
    ([300, 50], [40, 0], 2, 2, True),                # rows that see nothing, an empty sequence
    ([130, 257], [390, 100], 2, 2, False),           # no mask
])
def test_prefill_ragged_kv(lib, Lq, Lk, Hq, Hkv, causal):
    """Ragged (non-paged) K/V: sequence b's keys are rows [cu[b-1], cu[b]) of
    one packed tensor.  The oracle sees the same rows as a page-size-1 pool
    whose block table points at them."""
    rng = np.random.default_rng((sum(Lk), 23))
    Lq, Lk = np.asarray(Lq, np.int32), np.asarray(Lk, np.int32)
    B, T, Tkv = len(Lq), int(Lq.sum()), int(Lk.sum())
    nb = max(1, (int(max(Lq.max(), Lk.max())) + 127) // 128)
    q8 = rng.integers(-127, 128, (T, Hq, 128), dtype=np.int8)
    qs = (rng.uniform(0.5, 1.5, (B, nb, Hq)) * 3.0 / 127).astype(np.float32)
    k8 = rng.integers(-127, 128, (max(Tkv, 1), Hkv, 128), dtype=np.int8)
    ks = (rng.uniform(0.5, 1.5, (B, nb, Hkv)) * 3.0 / 127).astype(np.float32)
    v_bits = ocache.bf16_bits(synth.bf16_normal(rng, (max(Tkv, 1), Hkv, 128)))
    cu_kv = synth.inclusive_prefix(Lk)
    kvb = np.concatenate([[0], cu_kv[:-1]]).astype(np.int32)
    bt = np.full((B, max(1, int(Lk.max()))), -1, np.int32)
    for b in range(B):
        bt[b, :Lk[b]] = kvb[b] + np.arange(Lk[b])
    cu_q = synth.inclusive_prefix(Lq)
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    v_t = _t(v_bits[:Tkv].view(np.int16)).view(torch.bfloat16)
    out = lib.prefill_paged(_t(q8), _t(qs), _t(k8[:Tkv]), _t(ks), v_t, None, _t(cu_q), None,
                            causal=causal, lse=lse, error_word=err, cu_seqlens_kv=_t(cu_kv))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_o, want_lse = oatt.paged_prefill_int8(q8, qs, k8.reshape(-1, 1, Hkv, 128), ks,
                                               v_bits.reshape(-1, 1, Hkv, 128), bt, cu_q, Lk,
                                               1.0 / np.sqrt(128.0), causal)
    assert_attention_close(bf16_to_f64(out), want_o)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)

def test_prefill_zero_scale_blocks(lib):
    """A key block and a query block whose scale is 0 (all-zero input
    blocks): their logits are exactly 0 and nothing turns into NaN."""
    c = _random_case(5, [300], [300], 2, 2, 64)
    c["ks"][0, 1, :] = 0.0
    c["qs"][0, 2, 1] = 0.0
    got_o, got_lse, err = _run_prefill(lib, c, True)
    assert err == 0
    want_o, want_lse = _oracle(c, True)
    assert_attention_close(got_o, want_o)
    assert_lse_close(got_lse, want_lse)


def test_prefill_running_max_jumps(lib):
    """Key scales grow 4x per block: later tiles beat the running maximum by
    far more than 2^8 and the accumulated O rows are rescaled (the lse stays
    near 1.5e3, where one fp32 ulp is well inside the 1e-3 bound)."""
    c = _random_case(9, [700], [700], 2, 2, 64, kmag=0.5)
    c["ks"][0] *= (4.0 ** np.arange(c["ks"].shape[1]))[:, None].astype(np.float32)
    got_o, got_lse, err = _run_prefill(lib, c, True)
    assert err == 0
    want_o, want_lse = _oracle(c, True)
    assert_attention_close(got_o, want_o)
    assert_lse_close(got_lse, want_lse)


def test_prefill_bad_page_sets_error_word(lib):
    """A block_table entry outside the pool is read as zeros and flagged."""
    c = _random_case(3, [256], [256], 1, 1, 64)
    P = c["k_pool"].shape[0]
    c["bt"][0, 1] = P + 5
    _, _, err = _run_prefill(lib, c, True)
    assert err & 2


def test_prefill_full_size_sampled(lib):
    """8 sequences, L ~ U{256..4096}, 32 heads, page 64: the GPU writes the
    cache and runs the prefill (the benchmark's launch); the oracle rebuilds
    two sequences' caches from the same bf16 draws, which must match the
    written bytes and scales exactly (about 30M codes, so thousands sit near
    a rounding boundary), and checks sampled attention rows."""
    wl = synth.varlen_prefill(0)
    lengths = wl.lengths
    cos, sin = orope.cos_sin_table(int(lengths.max()), 128, wl.theta)
    d = _gpu_write(lib, wl.q, wl.k, wl.v, lengths, wl.block_table, wl.num_pages, 64, cos, sin)
    T, H = wl.q.shape[0], wl.H
    lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lk = _t(lengths)
    out = lib.prefill_paged(d["q8"], d["qs"], d["k_pool"], d["ks"], d["v_pool"], _t(wl.block_table),
                            d["cu"], lk, causal=True, lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    begin = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    for b in (int(np.argmax(lengths)), int(np.argmin(lengths))):
        L = int(lengths[b])
        sl = slice(int(begin[b]), int(begin[b]) + L)
        npg = (L + 63) // 64
        bt1 = np.arange(npg, dtype=np.int32)[None]
        kp, vp, kscale, q8, qscale, _ = ocache.write_int8_block128_rope(
            wl.q[sl], wl.k[sl], wl.v[sl], np.array([L], np.int32), bt1, 64, cos, sin,
            (L + 127) // 128, np.zeros((npg, 64, H, 128), np.int8),
            np.zeros((npg, 64, H, 128), np.uint16))
        rows_b = d["slots"][begin[b]:begin[b] + L].long()
        got_k = d["k_pool"].reshape(-1, H, 128)[rows_b].cpu().numpy()
        got_v = d["v_pool"].reshape(-1, H, 128)[rows_b].cpu().view(torch.int16).numpy()
        assert np.array_equal(got_k, kp.reshape(-1, H, 128)[:L])
        assert np.array_equal(got_v.view(np.uint16), vp.reshape(-1, H, 128)[:L])
        assert np.array_equal(d["q8"][begin[b]:begin[b] + L].cpu().numpy(), q8)
        nblk = (L + 127) // 128
        assert np.array_equal(_u32(d["ks"][b, :nblk].cpu().numpy()), _u32(kscale[0, :nblk]))
        assert np.array_equal(_u32(d["qs"][b, :nblk].cpu().numpy()), _u32(qscale[0, :nblk]))
        toks = sorted({0, 1, 127, 128, L // 2, L - 2, L - 1})
        rows = [(t, h) for t in toks for h in (0, 13, 31)]
        want_o, want_lse = oatt.paged_prefill_int8(q8, qscale, kp, kscale, vp, bt1,
                                                   np.array([L], np.int32), np.array([L], np.int32),
                                                   wl.scale, True, rows=rows)
        ti = np.array([t for t, _ in rows])
        hi = np.array([h for _, h in rows])
        got_o = bf16_to_f64(out[torch.from_numpy(begin[b] + ti).long(), torch.from_numpy(hi).long()])
        got_l = lse[torch.from_numpy(begin[b] + ti).long(), torch.from_numpy(hi).long()]
        assert_attention_close(got_o, want_o[ti, hi])
        assert_lse_close(got_l.cpu().numpy().astype(np.float64), want_lse[ti, hi])


# ------------------------------------------------------------------ FP8 V

def _fp8v_case(seed, Lq, Lk, Hq, Hkv, ps):
    """INT8 Q/K as in _random_case, V as E4M3 codes with per-(sequence, head,
    channel) scales from the oracle's FP8-V quantiser of bf16 draws."""
    c = _random_case(seed, Lq, Lk, Hq, Hkv, ps)
    rng = np.random.default_rng((seed, 78))
    Lk = np.asarray(Lk, np.int32)
    v = synth.bf16_normal(rng, (int(Lk.sum()), Hkv, 128))
    codes, vscale = ocache.v_channel_fp8(v, synth.inclusive_prefix(Lk))
    P, ps_, _, _ = c["k_pool"].shape
    vpool = np.full((P, ps_, Hkv, 128), 0x7F, np.uint8)     # NaN codes off the written rows
    begin = np.concatenate([[0], np.cumsum(Lk)[:-1]])
    for b, L in enumerate(Lk):
        rows = ocache.slot_mapping(np.array([int(L)]), np.zeros(1, np.int64), c["bt"][b:b + 1], ps_)
        vpool.reshape(P * ps_, Hkv, 128)[rows] = codes[begin[b]:begin[b] + int(L)]
    c["v_codes"], c["vscale"] = vpool, vscale
    return c


@pytest.mark.parametrize("Lq,Lk,Hq,Hkv,ps,causal", [
    ([1, 130, 300], [1, 130, 300], 2, 2, 64, True),
    ([77, 128, 1], [300, 128, 513], 4, 1, 32, True),       # cached prefix, GQA 4:1
    ([130, 257], [390, 100], 2, 1, 128, False),
    ([640, 520], [640, 520], 1, 1, 16, True),
])
def test_prefill_fp8_v(lib, Lq, Lk, Hq, Hkv, ps, causal):
    """FP8 V with channel scales: P.V as an FP8 product (P in two E4M3
    terms) against the oracle on the same codes."""
    c = _fp8v_case(sum(Lq) + ps, Lq, Lk, Hq, Hkv, ps)
    T = c["q8"].shape[0]
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = lib.prefill_paged(_t(c["q8"]), _t(c["qs"]), _t(c["k_pool"]), _t(c["ks"]), _t(c["v_codes"]),
                            _t(c["bt"]), _t(c["cu"]), _t(c["Lk"]), causal=causal, lse=lse,
                            error_word=err, v_scale=_t(c["vscale"]))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_o, want_lse = oatt.paged_prefill_int8(c["q8"], c["qs"], c["k_pool"], c["ks"], c["v_codes"],
                                               c["bt"], c["cu"], c["Lk"], 1.0 / np.sqrt(128.0), causal,
                                               v_scale=c["vscale"])
    assert_attention_close(bf16_to_f64(out), want_o, rel=REL_L2_FP8_P)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)


def test_write_cache_int8_v_fp8_bit_exact_and_ragged_prefill(lib):
    """The write's FP8 V (codes and channel scales) bit-exact against the
    oracle, then a ragged (packed K/V) prefill over those codes."""
    rng = np.random.default_rng(61)
    lengths = np.array([200, 1, 333], dtype=np.int32)
    T, Hq, Hkv, D, ps = int(lengths.sum()), 4, 2, 128, 64
    q = synth.bf16_normal(rng, (T, Hq, D))
    k = synth.bf16_normal(rng, (T, Hkv, D))
    v = synth.bf16_normal(rng, (T, Hkv, D))
    v[:, 1, 5] = 0.0                                           # an all-zero channel
    bt, P = synth.page_tables(rng, lengths, ps)
    cos, sin = orope.cos_sin_table(512, 128, 1.0e4)
    B, nb = 3, 3
    k_pool = torch.zeros((P, ps, Hkv, D), dtype=torch.int8, device=DEV)
    v_pool = torch.full((P, ps, Hkv, D), 0x7F, dtype=torch.uint8, device=DEV)
    ks = torch.zeros((B, nb, Hkv), dtype=torch.float32, device=DEV)
    qs = torch.zeros((B, nb, Hq), dtype=torch.float32, device=DEV)
    q8 = torch.zeros((T, Hq, D), dtype=torch.int8, device=DEV)
    vsc = torch.full((B, Hkv, D), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cu = synth.inclusive_prefix(lengths)
    lib.write_cache_int8_block128_rope(
        _t(q).to(torch.bfloat16), _t(k).to(torch.bfloat16), _t(v).to(torch.bfloat16), _t(cu), _t(bt),
        333, _t(cos), _t(sin), k_pool, v_pool, ks, q8, qs, error_word=err, v_channel_scale=vsc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp, vp, kscale, q8w, qscale, slots, vscw = ocache.write_int8_block128_rope(
        q, k, v, cu, bt, ps, cos, sin, nb, np.zeros((P, ps, Hkv, D), np.int8),
        np.full((P, ps, Hkv, D), 0x7F, np.uint8), v_fp8=True)
    assert np.array_equal(_u32(vsc.cpu().numpy()), _u32(vscw))
    got_v = v_pool.cpu().numpy().reshape(P * ps, Hkv, D)
    assert np.array_equal(got_v[slots], vp.reshape(P * ps, Hkv, D)[slots])
    assert np.array_equal(q8.cpu().numpy(), q8w)
    # ragged prefill over the packed rows
    k_rag = k_pool.reshape(P * ps, Hkv, D)[torch.from_numpy(slots).long().to(DEV)].contiguous()
    v_rag = v_pool.reshape(P * ps, Hkv, D)[torch.from_numpy(slots).long().to(DEV)].contiguous()
    lse = torch.empty((T, Hq), dtype=torch.float32, device=DEV)
    out = lib.prefill_paged(q8, qs, k_rag, ks, v_rag, None, _t(cu), _t(lengths), causal=True,
                            lse=lse, error_word=err, cu_seqlens_kv=_t(cu), v_scale=vsc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_o, want_lse = oatt.paged_prefill_int8(q8w, qscale, kp, kscale, vp, bt, cu, lengths,
                                               1.0 / np.sqrt(128.0), True, v_scale=vscw)
    assert_attention_close(bf16_to_f64(out), want_o, rel=REL_L2_FP8_P)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)
