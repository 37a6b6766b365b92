"""GPU parity: the MLA combined-row cache write (bit-exact) and the MLA-absorb
sparse paged decode against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import cache as ocache
from oracle import mla as omla
from quantized_paged_kv_varlen_gb300 import synth
from tests.gpu_util import assert_attention_close, assert_lse_close, bf16_to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
FILL = 0xA5          # every unwritten pool byte


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(seed, lengths, q_per_seq, QN, bs, sparse_size, n_ids):
    """Per-sequence kv draws written into a permuted pool; q_per_seq query
    tokens per sequence, each listing n_ids distinct ids (then -1)."""
    rng = np.random.default_rng((seed, 19))
    lengths = np.asarray(lengths, dtype=np.int32)
    B = len(lengths)
    bt, P = synth.page_tables(rng, lengths, bs, extra_pages=1)
    kv = synth.bf16_normal(rng, (int(lengths.sum()), 576))
    T = B * q_per_seq
    q = synth.bf16_normal(rng, (T, QN, 576))
    idx = np.full((T, 1, sparse_size), -1, dtype=np.int32)
    for t in range(T):
        b = t // q_per_seq
        n = min(n_ids, int(lengths[b]), sparse_size)
        idx[t, 0, :n] = rng.permutation(int(lengths[b]))[:n]
    cu_q = np.arange(1, B + 1, dtype=np.int32) * q_per_seq
    return dict(lengths=lengths, bt=bt, P=P, bs=bs, kv=kv, q=q, idx=idx, cu_q=cu_q,
                scale=1.0 / np.sqrt(576.0))


def _gpu_pool(lib, c):
    pool = torch.full((c["P"], c["bs"], 1, 656), FILL, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.write_cache_mla(_t(c["kv"]).to(torch.bfloat16), _t(synth.inclusive_prefix(c["lengths"])),
                        _t(c["bt"]), pool, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return pool


def _oracle_pool(c):
    pool = np.full((c["P"], c["bs"], 1, 656), FILL, dtype=np.uint8)
    B = len(c["lengths"])
    pool, _ = ocache.write_mla_rows(c["kv"], synth.inclusive_prefix(c["lengths"]),
                                    np.zeros(B, np.int64), c["bt"], c["bs"], pool)
    return pool


def _run(lib, c, pool, mode):
    T, QN = c["q"].shape[:2]
    lse = torch.full((T, QN), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = lib.mla_sparse_decode(_t(c["q"]).to(torch.bfloat16), pool, _t(c["idx"]), _t(c["bt"]),
                                _t(c["lengths"]), _t(c["cu_q"]), scale=c["scale"], sparse_mode=mode,
                                lse=lse, error_word=err)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), int(err.item())


def test_write_cache_mla_bit_exact(lib):
    c = _case(1, [300, 77, 130], 1, 4, 64, 128, 64)
    got = _gpu_pool(lib, c).cpu().numpy()
    assert np.array_equal(got, _oracle_pool(c))


def test_write_cache_mla_rope_bit_exact(lib):
    """RoPE on the rope part of the rows and of the queries, at positions
    start_pos[b] + i: pool bytes and rotated queries bit-exact; q_out may be
    q itself."""
    from oracle import rope as orope
    rng = np.random.default_rng(41)
    lengths = np.array([37, 5, 90], np.int32)
    start = np.array([3, 200, 0], np.int32)
    bt, P = synth.page_tables(rng, lengths + start, 64, extra_pages=1)
    kv = synth.bf16_normal(rng, (int(lengths.sum()), 576))
    q = synth.bf16_normal(rng, (int(lengths.sum()), 8, 576))
    cos, sin = orope.cos_sin_table(400, 64, 1.0e4)
    cu = synth.inclusive_prefix(lengths)
    pool = torch.full((P, 64, 1, 656), FILL, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    qd = _t(q).to(torch.bfloat16)
    q_out = lib.write_cache_mla(_t(kv).to(torch.bfloat16), _t(cu), _t(bt), pool, start_pos=_t(start),
                                error_word=err, rope_cos=_t(cos), rope_sin=_t(sin), q=qd, q_out=qd)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and q_out.data_ptr() == qd.data_ptr()
    want_pool = np.full((P, 64, 1, 656), FILL, dtype=np.uint8)
    want_pool, _ = ocache.write_mla_rows(kv, cu, start.astype(np.int64), bt, 64, want_pool, cos, sin)
    assert np.array_equal(pool.cpu().numpy(), want_pool)
    want_q = ocache.mla_rope(q, cu, start.astype(np.int64), cos, sin)
    assert np.array_equal(q_out.float().cpu().numpy(), want_q)


def test_write_cache_mla_rope_position_past_table(lib):
    """A token whose position lies past the RoPE tables is not written and
    flags the length error."""
    from oracle import rope as orope
    rng = np.random.default_rng(42)
    lengths = np.array([4], np.int32)
    bt, P = synth.page_tables(rng, lengths + 30, 16)
    kv = synth.bf16_normal(rng, (4, 576))
    cos, sin = orope.cos_sin_table(32, 64, 1.0e4)
    pool = torch.full((P, 16, 1, 656), FILL, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.write_cache_mla(_t(kv).to(torch.bfloat16), _t(synth.inclusive_prefix(lengths)), _t(bt), pool,
                        start_pos=_t(np.array([30], np.int32)), error_word=err,
                        rope_cos=_t(cos), rope_sin=_t(sin))
    torch.cuda.synchronize()
    assert int(err.item()) & 8
    got = pool.cpu().numpy().reshape(-1, 656)
    want = np.full((P, 16, 1, 656), FILL, dtype=np.uint8)
    want, slots = ocache.write_mla_rows(kv[:2], np.array([2], np.int32), np.array([30]), bt, 16, want, cos, sin)
    assert np.array_equal(got[slots], want.reshape(-1, 656)[slots])     # positions 30, 31 written
    untouched = np.ones(got.shape[0], bool)
    untouched[slots] = False
    assert np.all(got[untouched] == FILL)                                # 32, 33 not


@pytest.mark.parametrize("lengths,qps,QN,bs,S,n,mode", [
    ([300, 700], 1, 16, 64, 256, 200, 0),         # -1 tails, ragged last tile
    ([1000, 513], 1, 128, 64, 640, 640, 0),       # full head tile, S past one 512-key group
    ([257, 400], 3, 32, 16, 384, 300, 3),         # three query rows per sequence, causal drop
    ([90, 1200], 2, 128, 128, 128, 100, 0),       # two query rows, one key tile
])
def test_mla_shapes(lib, lengths, qps, QN, bs, S, n, mode):
    c = _case(sum(lengths) + S, lengths, qps, QN, bs, S, n)
    pool = _gpu_pool(lib, c)
    got_o, got_lse, err = _run(lib, c, pool, mode)
    assert err == 0
    want_o, want_lse = omla.mla_sparse_decode(c["q"], _oracle_pool(c), c["idx"], c["bt"],
                                              c["lengths"], c["cu_q"], c["scale"], sparse_mode=mode)
    assert_attention_close(got_o, want_o)
    assert_lse_close(got_lse, want_lse)


def test_mla_empty_lists_and_bad_ids(lib):
    """A token whose list starts with -1 sees nothing (O = 0, lse = -inf);
    an id past L_kv is skipped and flagged; entries after the first -1 are
    ignored even when they hold valid ids."""
    c = _case(3, [200, 300], 1, 8, 64, 128, 100)
    c["idx"][0, 0, :] = -1
    c["idx"][1, 0, 100] = -1
    c["idx"][1, 0, 101:110] = 5          # after the first -1: ignored
    pool = _gpu_pool(lib, c)
    got_o, got_lse, err = _run(lib, c, pool, 0)
    assert err == 0
    want_o, want_lse = omla.mla_sparse_decode(c["q"], _oracle_pool(c), c["idx"], c["bt"],
                                              c["lengths"], c["cu_q"], c["scale"])
    assert np.all(got_o[0] == 0.0) and np.all(np.isneginf(got_lse[0]))
    assert_attention_close(got_o, want_o)
    assert_lse_close(got_lse, want_lse)
    c["idx"][1, 0, 3] = 300              # = L_kv of sequence 1: out of range
    _, _, err = _run(lib, c, pool, 0)
    assert err & 4


def test_mla_full_size_sampled(lib):
    """B=32, 128 heads, L ~ U{32768..65536}, block 64, 2048 ids per token:
    the GPU writes the whole cache and runs the decode (the benchmark's
    launch); the oracle packs the listed rows from the same bf16 draws and
    checks three tokens, all heads."""
    d = synth.mla_sparse_device(0, DEV)
    pool = torch.empty((d["num_pages"], 64, 1, 656), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.write_cache_mla(d["kv"], d["cu_kv"], d["bt"], pool, error_word=err)
    lse = torch.empty((32, 128), dtype=torch.float32, device=DEV)
    out = lib.mla_sparse_decode(d["q"], pool, d["idx"], d["bt"], d["lk"], d["cu_q"],
                                scale=d["scale"], lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    begin = np.concatenate([[0], np.cumsum(d["lengths"])[:-1]])
    for t in (0, 13, 31):
        ids = d["idx"][t, 0].cpu().numpy()
        ids = ids[ids >= 0]
        rows = d["kv"][torch.from_numpy(begin[t] + ids).long().to(DEV)].float().cpu().numpy()
        n = len(ids)
        mini = ocache.mla_pack_rows(rows).reshape(n, 1, 1, 656)
        want_o, want_lse = omla.mla_sparse_decode(
            d["q"][t:t + 1].float().cpu().numpy(), mini,
            np.arange(n, dtype=np.int32).reshape(1, 1, n), np.arange(n, dtype=np.int32)[None],
            np.array([n], np.int32), np.array([1], np.int32), d["scale"])
        assert_attention_close(bf16_to_f64(out[t:t + 1]), want_o)
        assert_lse_close(lse[t:t + 1].cpu().numpy().astype(np.float64), want_lse)


@pytest.mark.parametrize("lengths,qps,QN,bs,S,n_ids,sbs,mode", [
    ([300, 701], 1, 16, 64, 80, 60, 4, 0),        # partial last block, -1 tail, S*n past 256
    ([1000, 517], 2, 32, 64, 40, 33, 16, 3),      # two query rows, causal drop inside blocks
    ([900, 130], 1, 128, 128, 8, 7, 128, 0),      # whole-tile blocks
])
def test_mla_block_sparse(lib, lengths, qps, QN, bs, S, n_ids, sbs, mode):
    """sparse_block_size > 1: each listed id names sbs consecutive tokens."""
    rng = np.random.default_rng((sum(lengths), sbs))
    c = _case(sum(lengths) + sbs, lengths, qps, QN, bs, S, 0)
    T = c["q"].shape[0]
    idx = np.full((T, 1, S), -1, dtype=np.int32)
    for t in range(T):
        nblk = (int(c["lengths"][t // qps]) + sbs - 1) // sbs
        k = min(n_ids, nblk, S)
        idx[t, 0, :k] = rng.permutation(nblk)[:k]
    c["idx"] = idx
    pool = _gpu_pool(lib, c)
    lse = torch.full((T, QN), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = lib.mla_sparse_decode(_t(c["q"]).to(torch.bfloat16), pool, _t(idx), _t(c["bt"]),
                                _t(c["lengths"]), _t(c["cu_q"]), scale=c["scale"], sparse_mode=mode,
                                lse=lse, error_word=err, sparse_block_size=sbs)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_o, want_lse = omla.mla_sparse_decode(c["q"], _oracle_pool(c), idx, c["bt"], c["lengths"],
                                              c["cu_q"], c["scale"], sparse_mode=mode,
                                              sparse_block_size=sbs)
    assert_attention_close(bf16_to_f64(out), want_o)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)


def test_mla_tnd_keys_through_block_size_one(lib):
    """A packed TND key tensor [KV_T, 1, 656] read as a pool of block size 1
    whose block-table row b lists sequence b's rows."""
    rng = np.random.default_rng(71)
    lengths = np.array([150, 61, 300], np.int32)
    KV_T, QN, S = int(lengths.sum()), 16, 128
    kv = synth.bf16_normal(rng, (KV_T, 576))
    rows = ocache.mla_pack_rows(kv)                              # packed TND rows
    begin = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    bt = np.full((3, int(lengths.max())), -1, np.int32)
    for b in range(3):
        bt[b, :lengths[b]] = begin[b] + np.arange(lengths[b])
    q = synth.bf16_normal(rng, (3, QN, 576))
    idx = np.full((3, 1, S), -1, np.int32)
    for t in range(3):
        n = min(100, int(lengths[t]))
        idx[t, 0, :n] = rng.permutation(int(lengths[t]))[:n]
    cu_q = np.arange(1, 4, dtype=np.int32)
    pool = _t(rows.reshape(KV_T, 1, 1, 656))
    lse = torch.empty((3, QN), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = lib.mla_sparse_decode(_t(q).to(torch.bfloat16), pool, _t(idx), _t(bt), _t(lengths), _t(cu_q),
                                scale=1.0 / 24.0, lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_o, want_lse = omla.mla_sparse_decode(q, rows.reshape(KV_T, 1, 1, 656), idx, bt, lengths,
                                              cu_q, 1.0 / 24.0)
    assert_attention_close(bf16_to_f64(out), want_o)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), want_lse)


def test_mla_permuted_ids_give_the_same_output(lib):
    """The kernel regroups a token's keys by pool row; any order of the
    listed ids gives the oracle's result (which does not depend on it), over
    several 512-key groups."""
    c = _case(77, [1500, 900], 1, 64, 64, 1280, 1100)
    pool = _gpu_pool(lib, c)
    got_o, got_lse, err = _run(lib, c, pool, 0)
    assert err == 0
    rng = np.random.default_rng(78)
    c2 = dict(c)
    idx2 = c["idx"].copy()
    for t in range(idx2.shape[0]):
        n = int((idx2[t, 0] >= 0).sum())
        idx2[t, 0, :n] = idx2[t, 0, :n][rng.permutation(n)]
    c2["idx"] = idx2
    got2_o, got2_lse, err2 = _run(lib, c2, pool, 0)
    assert err2 == 0
    want_o, want_lse = omla.mla_sparse_decode(c["q"], _oracle_pool(c), c["idx"], c["bt"],
                                              c["lengths"], c["cu_q"], c["scale"])
    for o, l in ((got_o, got_lse), (got2_o, got2_lse)):
        assert_attention_close(o, want_o)
        assert_lse_close(l, want_lse)
