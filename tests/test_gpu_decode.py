"""GPU parity: FP8 cache write (bit-exact) and split-KV paged decode against
the CPU oracle, on the tiny workload, edge cases and the full Llama-3-8B
shaped batch (sampled requests), through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import cache as ocache
from quantized_paged_kv_varlen_gb300 import synth
from tests.gpu_util import DECODE_TIGHT, assert_attention_close, assert_lse_close, bf16_to_f64

pytestmark = pytest.mark.gpu

FILL = 0x7F                # an E4M3 NaN code in every unwritten pool byte
SCALE_FILL = np.float32("nan")


def _pool_shape(P, ps, H, D, layout):
    return (P, H, ps, D) if layout == "HND" else (P, ps, H, D)


def _dev_inputs(lib, wl, k, v, layout="NHD"):
    dev = "cuda"
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    k_pool = torch.full(_pool_shape(P, ps, H, D, layout), FILL, dtype=torch.uint8, device=dev)
    v_pool = torch.full_like(k_pool, FILL)
    ks = torch.full((P, ps, H), float("nan"), dtype=torch.float32, device=dev)
    vs = torch.full_like(ks, float("nan"))
    bt = torch.from_numpy(wl.block_table).to(dev)
    cu = torch.from_numpy(np.cumsum(wl.lengths).astype(np.int32)).to(dev)
    slots = torch.full((k.shape[0],), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kt = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vt = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    lib.write_cache_fp8(kt, vt, cu, bt, k_pool, v_pool, ks, vs, slot_mapping=slots,
                        error_word=err, kv_layout=layout)
    return dict(k_pool=k_pool, v_pool=v_pool, ks=ks, vs=vs, bt=bt, slots=slots, err=err)


def _oracle_cache(wl, k, v, reqs=None, layout="NHD"):
    """Oracle pools; with reqs given, a compact pool holding only their pages
    (and a block table remapped to it)."""
    lens = wl.lengths
    if reqs is None:
        reqs = list(range(wl.B))
        bt = wl.block_table
        P = wl.num_pages
        kk, vv, cu = k, v, np.cumsum(lens)
    else:
        offs = np.concatenate([[0], np.cumsum(lens)])
        bt = np.full((len(reqs), wl.block_table.shape[1]), -1, np.int32)
        P = 0
        parts_k, parts_v = [], []
        for i, b in enumerate(reqs):
            n = (int(lens[b]) + wl.page_size - 1) // wl.page_size
            bt[i, :n] = np.arange(P, P + n)
            P += n
            parts_k.append(k[offs[b]:offs[b + 1]])
            parts_v.append(v[offs[b]:offs[b + 1]])
        kk, vv = np.concatenate(parts_k), np.concatenate(parts_v)
        cu = np.cumsum(lens[reqs])
    fill = np.full(_pool_shape(max(P, 1), wl.page_size, wl.Hkv, wl.D, layout), FILL, np.uint8)
    sfill = np.full((max(P, 1), wl.page_size, wl.Hkv), SCALE_FILL, np.float32)
    kp, vp, ksp, vsp, slots, _ = ocache.write_fp8_token_head(
        kk, vv, cu, np.zeros(len(reqs), np.int64), bt, wl.page_size, fill, fill, sfill, sfill,
        layout=layout)
    return kp, vp, ksp, vsp, bt, reqs


def _u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _check_decode(lib, wl, reqs=None, check_pool_bytes=True, kv=None, layout="NHD"):
    k, v = wl.kv_all() if kv is None else kv
    d = _dev_inputs(lib, wl, k, v, layout)
    plan = lib.DecodePlan(wl.lengths, wl.Hq, wl.Hkv, wl.page_size, wl.D, kv_layout=layout)
    q = torch.from_numpy(wl.q).cuda().to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
    plan.run(q, d["k_pool"], d["v_pool"], d["ks"], d["vs"], d["bt"], wl.scale, out=out, lse=lse,
             error_word=d["err"])
    torch.cuda.synchronize()
    assert int(d["err"].item()) == 0

    kp, vp, ksp, vsp, obt, reqs = _oracle_cache(wl, k, v, reqs, layout)
    want_o, want_lse = oatt.paged_decode_fp8(wl.q[reqs], kp, vp, ksp, vsp, obt,
                                             wl.lengths[reqs], wl.scale, layout=layout)
    got_o = bf16_to_f64(out)[reqs]
    got_lse = lse.cpu().numpy().astype(np.float64)[reqs]
    assert_attention_close(got_o, want_o, tight=DECODE_TIGHT)
    assert_lse_close(got_lse, want_lse)

    if check_pool_bytes:
        # the cache rows of the checked requests, bit for bit (scales as bits)
        gk = d["k_pool"].cpu().numpy()
        gks = d["ks"].cpu().numpy()
        for i, b in enumerate(reqs):
            n = (int(wl.lengths[b]) + wl.page_size - 1) // wl.page_size
            gp = wl.block_table[b, :n]
            op = obt[i, :n]
            assert np.array_equal(gk[gp], kp[op]), f"k bytes differ for request {b}"
            assert np.array_equal(_u32(gks[gp]), _u32(ksp[op])), f"k scales differ ({b})"
    return d, plan


def test_write_cache_fp8_bit_exact_tiny(lib):
    wl = synth.tiny_decode(0)
    k, v = wl.kv_all()
    d = _dev_inputs(lib, wl, k, v)
    torch.cuda.synchronize()
    kp, vp, ksp, vsp, bt, _ = _oracle_cache(wl, k, v)
    assert np.array_equal(d["k_pool"].cpu().numpy(), kp)
    assert np.array_equal(d["v_pool"].cpu().numpy(), vp)
    assert np.array_equal(_u32(d["ks"].cpu().numpy()), _u32(ksp))
    assert np.array_equal(_u32(d["vs"].cpu().numpy()), _u32(vsp))
    want_slots = ocache.slot_mapping(np.cumsum(wl.lengths), np.zeros(2, np.int64), bt, 16)
    assert np.array_equal(d["slots"].cpu().numpy(), want_slots)
    assert int(d["err"].item()) == 0


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 1, 64)])
def test_write_cache_fp8_rope_bit_exact(lib, Hq, Hkv, D):
    """RoPE fused into the FP8 write: k rotated at each token's position
    (start_pos > 0 on some requests) before it is quantised, v not rotated,
    the rotated queries rounded to bf16; bytes, scale bits, slots and
    rotated query bits against the oracle."""
    from oracle import rope as orope
    rng = np.random.default_rng(31)
    lengths = np.array([20, 7, 45], np.int32)
    start = np.array([0, 9, 30], np.int32)
    ps = 16
    bt, P = synth.page_tables(rng, lengths + start, ps)
    T = int(lengths.sum())
    k = synth.bf16_normal(rng, (T, Hkv, D))
    v = synth.bf16_normal(rng, (T, Hkv, D))
    qv = synth.bf16_normal(rng, (T, Hq, D))
    max_pos = int((lengths + start).max())
    cos, sin = orope.cos_sin_table(max_pos, D, 1.0e4)
    gcos, gsin = lib.rope_table(1.0e4, max_pos, D)
    assert np.array_equal(gcos.cpu().numpy().view(np.uint32), cos.view(np.uint32))
    dev = "cuda"
    k_pool = torch.full((P, ps, Hkv, D), FILL, dtype=torch.uint8, device=dev)
    v_pool = torch.full_like(k_pool, FILL)
    ks = torch.full((P, ps, Hkv), float("nan"), dtype=torch.float32, device=dev)
    vs = torch.full_like(ks, float("nan"))
    slots = torch.full((T,), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q_out = lib.write_cache_fp8(tt(k).bfloat16(), tt(v).bfloat16(), tt(np.cumsum(lengths).astype(np.int32)),
                                tt(bt), k_pool, v_pool, ks, vs, start_pos=tt(start),
                                slot_mapping=slots, error_word=err, rope_cos=gcos, rope_sin=gsin,
                                q=tt(qv).bfloat16())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    fill = np.full((P, ps, Hkv, D), FILL, np.uint8)
    sfill = np.full((P, ps, Hkv), SCALE_FILL, np.float32)
    kp, vp, ksp, vsp, oslots, q_rot = ocache.write_fp8_token_head(
        k, v, np.cumsum(lengths), start, bt, ps, fill, fill, sfill, sfill, q=qv, cos=cos, sin=sin)
    assert np.array_equal(k_pool.cpu().numpy(), kp)
    assert np.array_equal(v_pool.cpu().numpy(), vp)
    assert np.array_equal(_u32(ks.cpu().numpy()), _u32(ksp))
    assert np.array_equal(_u32(vs.cpu().numpy()), _u32(vsp))
    assert np.array_equal(slots.cpu().numpy(), oslots)
    got_q = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
    want_q = ocache.bf16_bits(ocache.bf16_round(q_rot))
    assert np.array_equal(got_q, want_q)
    # the rotation did something: unrotated keys give other bytes
    kp0, _, _, _, _, _ = ocache.write_fp8_token_head(k, v, np.cumsum(lengths), start, bt, ps,
                                                     fill, fill, sfill, sfill)
    assert not np.array_equal(kp0, kp)


def test_decode_tiny_gqa4_d64(lib):
    _check_decode(lib, synth.tiny_decode(0))


@pytest.mark.parametrize("lengths,ps,Hq,Hkv,D,kind", [
    ([0, 1, 127, 128, 129], 16, 4, 1, 64, 0),
    ([255, 256, 257, 1000, 3], 32, 8, 1, 128, 0),
    ([300, 64, 17], 64, 8, 2, 128, 0),
    ([513, 200], 128, 8, 8, 128, 1),
    ([700, 33, 256], 256, 16, 2, 128, 0),
    ([1200, 5], 16, 32, 8, 128, 1),
    ([900, 130, 17], 16, 64, 8, 128, 0),       # 3*Hq > 96: one kv head per work item
    ([777, 64], 32, 16, 8, 128, 1),            # a tile is half a page of 32
    ([300, 64, 17, 1], 32, 16, 4, 128, 1),     # 4 kv heads: 32-token tiles
    ([1000, 33], 64, 32, 4, 64, 1),            # 8 query heads per kv head, D = 64
    ([129, 16, 1, 250], 16, 8, 8, 64, 1),
    ([600, 31], 16, 16, 4, 128, 0),            # 32-token tiles would cross 16-token pages
])
def test_decode_edge_shapes(lib, lengths, ps, Hq, Hkv, D, kind):
    _, plan = _check_decode(lib, _edge_workload(lengths, ps, Hq, Hkv, D))
    assert plan.kind == kind


def _edge_workload(lengths, ps, Hq, Hkv, D):
    rng = np.random.default_rng(11)
    lengths = np.asarray(lengths, dtype=np.int32)
    bt, P = synth.page_tables(rng, lengths, ps, extra_pages=3)
    return synth.DecodeWorkload(seed=11, B=len(lengths), Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                                lengths=lengths, block_table=bt, num_pages=P,
                                q=synth.bf16_normal(rng, (len(lengths), Hq, D)),
                                scale=1.0 / np.sqrt(D), workload_id=9)


@pytest.mark.parametrize("lengths,ps,Hq,Hkv,D,kind", [
    ([0, 1, 127, 128, 129], 16, 4, 1, 64, 0),
    ([300, 64, 17], 64, 8, 2, 128, 0),
    ([700, 33, 256], 256, 16, 2, 128, 0),
    ([1200, 5], 16, 32, 8, 128, 1),
    ([777, 64], 32, 16, 8, 128, 1),            # a tile is half a page of 32
    ([300, 64, 17, 1], 32, 16, 4, 128, 1),     # 4 kv heads: 32-token tiles, partial tails
])
def test_decode_hnd_layout(lib, lengths, ps, Hq, Hkv, D, kind):
    """K/V pools [P, Hkv, page_size, D] (flashinfer's HND): the write places
    each (token, head) row bit for bit and both decode kernels read it."""
    _, plan = _check_decode(lib, _edge_workload(lengths, ps, Hq, Hkv, D), layout="HND")
    assert plan.kind == kind


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 8), (16, 4)])
def test_decode_large_magnitudes(lib, Hq, Hkv):
    """Queries scaled by 8: logits spread over many octaves."""
    rng = np.random.default_rng(12)
    lengths = np.array([400, 260], dtype=np.int32)
    ps = 32 if Hkv == 4 else 16
    bt, P = synth.page_tables(rng, lengths, ps)
    q = synth.bf16_round(synth.bf16_normal(rng, (2, Hq, 128)) * 8.0)
    wl = synth.DecodeWorkload(seed=12, B=2, Hq=Hq, Hkv=Hkv, D=128, page_size=ps, lengths=lengths,
                              block_table=bt, num_pages=P, q=q, scale=1.0 / np.sqrt(128.0),
                              workload_id=8)
    _check_decode(lib, wl)


@pytest.mark.parametrize("Hq,Hkv,ps", [(32, 8, 16), (16, 4, 32), (8, 2, 16)])
def test_decode_running_max_jumps(lib, Hq, Hkv, ps):
    """Keys grow 6x from token 100 on, inside the first work item: later
    tiles beat the running maximum by far more than 2^8, so the kernels
    must rescale what they have already accumulated."""
    rng = np.random.default_rng(14)
    lengths = np.array([700, 300], dtype=np.int32)
    bt, P = synth.page_tables(rng, lengths, ps)
    wl = synth.DecodeWorkload(seed=14, B=2, Hq=Hq, Hkv=Hkv, D=128, page_size=ps,
                              lengths=lengths, block_table=bt, num_pages=P,
                              q=synth.bf16_normal(rng, (2, Hq, 128)), scale=1.0 / np.sqrt(128.0),
                              workload_id=6)
    k, v = wl.kv_all()
    first = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    grow = np.zeros(k.shape[0], dtype=bool)
    for b, L in enumerate(lengths):
        grow[first[b] + 100:first[b] + L] = True
    k = k.copy()
    k[grow] = synth.bf16_round(k[grow] * 6.0)
    _check_decode(lib, wl, kv=(k, v))


def test_decode_bad_page_sets_error_word(lib):
    rng = np.random.default_rng(13)
    lengths = np.array([100, 50], dtype=np.int32)
    bt, P = synth.page_tables(rng, lengths, 16)
    wl = synth.DecodeWorkload(seed=13, B=2, Hq=4, Hkv=1, D=128, page_size=16, lengths=lengths,
                              block_table=bt, num_pages=P, q=synth.bf16_normal(rng, (2, 4, 128)),
                              scale=0.1, workload_id=7)
    k, v = wl.kv_all()
    d = _dev_inputs(lib, wl, k, v)
    bad = d["bt"].clone()
    bad[1, 0] = P + 5                                     # outside the pool
    plan = lib.DecodePlan(wl.lengths, 4, 1, 16, 128)
    q = torch.from_numpy(wl.q).cuda().to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = plan.run(q, d["k_pool"], d["v_pool"], d["ks"], d["vs"], bad, wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEV_ERR_BAD_PAGE
    # request 0 never touches the bad entry and is still right
    kp, vp, ksp, vsp, obt, _ = _oracle_cache(wl, k, v, [0])
    want, _ = oatt.paged_decode_fp8(wl.q[[0]], kp, vp, ksp, vsp, obt, wl.lengths[[0]], wl.scale)
    assert_attention_close(bf16_to_f64(out)[[0]], want, tight=DECODE_TIGHT)


def test_decode_full_batch_sampled(lib):
    """B=64, L ~ U{512..8192}, 32/8 heads, D=128, page 16: the benchmark's
    launch configuration; the oracle checks the shortest, the longest and
    two other requests (all heads) and their cache bytes."""
    wl = synth.batched_decode(0)
    order = np.argsort(wl.lengths)
    reqs = sorted({int(order[0]), int(order[-1]), 5, 40})
    _check_decode(lib, wl, reqs=reqs)


def test_decode_steps_with_side_stream_replan_and_growing_lengths(lib):
    """Three decode steps as a server runs them: append one token per
    request, re-plan on a side stream for the grown lengths (crossing a
    256-token chunk boundary), attend, merge; every step against the oracle."""
    rng = np.random.default_rng(41)
    B, Hq, Hkv, D, ps = 3, 32, 8, 128, 16
    L0 = np.array([254, 255, 90], np.int32)
    steps = 3
    Lmax = L0 + steps
    bt, P = synth.page_tables(rng, Lmax, ps)
    k_all = [synth.bf16_normal(rng, (int(Lmax[b]), Hkv, D)) for b in range(B)]
    v_all = [synth.bf16_normal(rng, (int(Lmax[b]), Hkv, D)) for b in range(B)]
    qv = synth.bf16_normal(rng, (B, Hq, D))
    dev = "cuda"
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    k_pool = torch.zeros((P, ps, Hkv, D), dtype=torch.uint8, device=dev)
    v_pool = torch.zeros_like(k_pool)
    ks = torch.zeros((P, ps, Hkv), dtype=torch.float32, device=dev)
    vs = torch.zeros_like(ks)
    btd = tt(bt)
    # the cache before the first step: L0 - 1 tokens of each request
    prev = L0 - 1
    lib.write_cache_fp8(tt(np.concatenate([k_all[b][:prev[b]] for b in range(B)])).bfloat16(),
                        tt(np.concatenate([v_all[b][:prev[b]] for b in range(B)])).bfloat16(),
                        tt(np.cumsum(prev).astype(np.int32)), btd, k_pool, v_pool, ks, vs)
    plan = lib.DecodePlan(Lmax, Hq, Hkv, ps, D)     # workspaces sized for the longest step
    side = torch.cuda.Stream()
    q = tt(qv).bfloat16()
    outs = []
    for step in range(steps):
        L = L0 + step
        plan.replan(seqlens_kv=L, stream=side)
        newk = tt(np.stack([k_all[b][L[b] - 1] for b in range(B)])).bfloat16()
        newv = tt(np.stack([v_all[b][L[b] - 1] for b in range(B)])).bfloat16()
        lib.write_cache_fp8(newk, newv, tt(np.arange(1, B + 1, dtype=np.int32)), btd, k_pool, v_pool,
                            ks, vs, start_pos=tt((L - 1).astype(np.int32)))
        plan.attend(q, k_pool, v_pool, ks, vs, btd, 1.0 / np.sqrt(D))
        out = torch.empty_like(q)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        plan.merge(out, lse)
        outs.append((L.copy(), out, lse))
    torch.cuda.synchronize()
    lib.check_errors()
    for L, out, lse in outs:
        kk = np.concatenate([k_all[b][:L[b]] for b in range(B)])
        vv = np.concatenate([v_all[b][:L[b]] for b in range(B)])
        z8 = np.zeros((P, ps, Hkv, D), np.uint8)
        zs = np.zeros((P, ps, Hkv), np.float32)
        kp, vp, ksp, vsp, _, _ = ocache.write_fp8_token_head(
            kk, vv, np.cumsum(L), np.zeros(B, np.int64), bt, ps, z8, z8, zs, zs)
        want_o, want_lse = oatt.paged_decode_fp8(qv, kp, vp, ksp, vsp, bt, L, 1.0 / np.sqrt(D))
        assert_attention_close(bf16_to_f64(out), want_o, tight=DECODE_TIGHT)
        assert_lse_close(lse.cpu().numpy(), want_lse)
