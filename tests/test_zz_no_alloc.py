"""The allocation-free decode entry point (qpkv_decode_static), for callers
that cannot allocate device memory: its output must match the planned
decode (qpkv_decode_plan + qpkv_decode_run) and the CPU oracle on the same
inputs, on two calls in a row (the fixed scratch keeps the previous call's
contents), the second call must leave the device's free memory and torch's
allocation count unchanged, a call on a capturing stream must be refused
with nothing recorded, and oversized batches must be rejected on the host.

This file sorts last so that a run stopping at the first failure has
already run every other test."""
import ctypes
import gc

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import cache as ocache
from quantized_paged_kv_varlen_gb300 import synth
from tests.gpu_util import DECODE_TIGHT, assert_attention_close, assert_lse_close, bf16_to_f64

UNSUPPORTED = 2
STATIC_LIMIT = 7


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(lib, wl, lens, q, d, out, lse, err, num_sms):
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib.qpkv_decode_static(
        lens.ctypes.data, wl.B, wl.Hq, wl.Hkv, wl.page_size, wl.D, num_sms, _ptr(q),
        _ptr(d["k_pool"]), _ptr(d["v_pool"]), _ptr(d["ks"]), _ptr(d["vs"]), d["k_pool"].shape[0],
        _ptr(d["bt"]), d["bt"].shape[1], ctypes.c_float(wl.scale), _ptr(out), _ptr(lse), _ptr(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _cache(q, wl):
    dev = "cuda"
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    d = dict(k_pool=torch.zeros((P, ps, H, D), dtype=torch.uint8, device=dev))
    d["v_pool"] = torch.zeros_like(d["k_pool"])
    d["ks"] = torch.zeros((P, ps, H), dtype=torch.float32, device=dev)
    d["vs"] = torch.zeros_like(d["ks"])
    d["bt"] = torch.from_numpy(wl.block_table).to(dev)
    cu = torch.from_numpy(np.cumsum(wl.lengths).astype(np.int32)).to(dev)
    q.write_cache_fp8(torch.from_numpy(k).to(dev).bfloat16(), torch.from_numpy(v).to(dev).bfloat16(),
                      cu, d["bt"], d["k_pool"], d["v_pool"], d["ks"], d["vs"])
    return d


def _mid_workload():
    rng = np.random.default_rng(21)
    lengths = rng.integers(100, 3000, size=16).astype(np.int32)
    bt, P = synth.page_tables(rng, lengths, 16)
    return synth.DecodeWorkload(seed=21, B=16, Hq=32, Hkv=8, D=128, page_size=16,
                                lengths=lengths, block_table=bt, num_pages=P,
                                q=synth.bf16_normal(rng, (16, 32, 128)),
                                scale=1.0 / np.sqrt(128.0), workload_id=6)


@pytest.mark.gpu
@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_static_decode_matches_planned_decode_twice(lib, which):
    wl = synth.tiny_decode(0) if which == "tiny" else _mid_workload()
    d = _cache(lib, wl)
    q = torch.from_numpy(wl.q).cuda().bfloat16()
    ref_lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
    plan = lib.DecodePlan(wl.lengths, wl.Hq, wl.Hkv, wl.page_size, wl.D)
    ref = plan.run(q, d["k_pool"], d["v_pool"], d["ks"], d["vs"], d["bt"], wl.scale, lse=ref_lse)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    raw = lib.load()
    # the oracle on the same cache bytes (written by the oracle's own quantiser)
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    z8 = np.zeros((P, ps, H, D), np.uint8)
    zs = np.zeros((P, ps, H), np.float32)
    kp, vp, ks, vs, _, _ = ocache.write_fp8_token_head(
        k, v, np.cumsum(wl.lengths), np.zeros(wl.B, np.int64), wl.block_table, ps, z8, z8, zs, zs)
    want_o, want_lse = oatt.paged_decode_fp8(wl.q, kp, vp, ks, vs, wl.block_table, wl.lengths,
                                             wl.scale)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((wl.B, wl.Hq), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        # collect first and keep the collector off across the call, so that
        # tensors of earlier tests freed meanwhile do not move the counters
        gc.collect()
        torch.cuda.synchronize()
        gc.disable()
        try:
            free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            status = _call_static(raw, wl, wl.lengths, q, d, out, lse, err, sms)
            torch.cuda.synchronize()
            free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        finally:
            gc.enable()
        assert status == 0
        if call == 1:
            # nothing allocated by the call itself (the first call may load modules)
            assert free1 == free0
            assert alloc1 == alloc0
        assert int(err.item()) == 0
        assert_attention_close(bf16_to_f64(out), bf16_to_f64(ref))
        assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy())
        assert_attention_close(bf16_to_f64(out), want_o, tight=DECODE_TIGHT)
        assert_lse_close(lse.cpu().numpy(), want_lse)


@pytest.mark.gpu
def test_static_decode_refuses_a_capturing_stream(lib):
    """Begin a capture, make the call, end the capture: the call returns
    QPKV_ERR_UNSUPPORTED and records nothing."""
    wl = synth.tiny_decode(0)
    d = _cache(lib, wl)
    q = torch.from_numpy(wl.q).cuda().bfloat16()
    out = torch.zeros_like(q)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    raw = lib.load()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        st = _call_static(raw, wl, wl.lengths, q, d, out, None, None, sms)
        g.capture_end()
    torch.cuda.synchronize()
    assert st == UNSUPPORTED


def test_static_decode_rejects_batches_beyond_its_scratch():
    """Host-side check, no GPU needed: 8192 requests of 8192 tokens need far
    more than the fixed partial-result array."""
    import quantized_paged_kv_varlen_gb300 as q
    from quantized_paged_kv_varlen_gb300 import build
    import os
    if not os.path.exists(q.LIB_PATH):
        build.build()
    raw = q.load()
    lens = np.full(8192, 8192, dtype=np.int32)
    fake = ctypes.c_void_p(0x100000)
    st = raw.qpkv_decode_static(lens.ctypes.data, len(lens), 32, 8, 16, 128, 148, fake, fake, fake,
                                fake, fake, 10, fake, 512, ctypes.c_float(0.1), fake, None, None,
                                None)
    assert st == STATIC_LIMIT
    assert raw.qpkv_status_string(STATIC_LIMIT).startswith(b"problem exceeds")
