"""GPU: the device error surface.  A bad page id with no caller error word
is reported through the library's own word and qpkv_error_check; the
bounded mbarrier wait every pipeline uses gives up, reports
QPKV_DEV_ERR_TIMEOUT and returns, leaving the context usable."""
import time

import numpy as np
import pytest
import torch

from quantized_paged_kv_varlen_gb300 import synth

pytestmark = pytest.mark.gpu


def _fp8_cache(lib, wl):
    dev = "cuda"
    k, v = wl.kv_all()
    P, ps, H, D = wl.num_pages, wl.page_size, wl.Hkv, wl.D
    k_pool = torch.zeros((P, ps, H, D), dtype=torch.uint8, device=dev)
    v_pool = torch.zeros_like(k_pool)
    ks = torch.zeros((P, ps, H), dtype=torch.float32, device=dev)
    vs = torch.zeros_like(ks)
    bt = torch.from_numpy(wl.block_table).to(dev)
    cu = torch.from_numpy(wl.cu_seqlens).to(dev)
    lib.write_cache_fp8(torch.from_numpy(k).to(dev).bfloat16(),
                        torch.from_numpy(v).to(dev).bfloat16(), cu, bt, k_pool, v_pool, ks, vs)
    return k_pool, v_pool, ks, vs, bt


def test_library_word_reports_a_bad_page_without_a_caller_word(lib):
    lib.check_errors()                                  # start clean (raises if not)
    wl = synth.tiny_decode(0)
    k_pool, v_pool, ks, vs, bt = _fp8_cache(lib, wl)
    assert lib.check_errors() == 0                      # the write set nothing
    bad = bt.clone()
    bad[1, 0] = wl.num_pages + 5
    plan = lib.DecodePlan(wl.lengths, wl.Hq, wl.Hkv, wl.page_size, wl.D)
    q = torch.from_numpy(wl.q).cuda().bfloat16()
    plan.run(q, k_pool, v_pool, ks, vs, bad, wl.scale)
    with pytest.raises(lib.QpkvError) as ei:
        lib.check_errors()
    assert ei.value.status == lib.ERR_DEVICE
    assert lib.check_errors() == 0                      # the check cleared it
    # with the right table nothing is reported
    plan.run(q, k_pool, v_pool, ks, vs, bt, wl.scale)
    assert lib.check_errors() == 0
    raw = lib.load()
    assert raw.qpkv_error_status(lib.DEV_ERR_BAD_PAGE) == lib.ERR_DEVICE
    assert raw.qpkv_error_status(lib.DEV_ERR_TIMEOUT | lib.DEV_ERR_BAD_PAGE) == lib.ERR_TIMEOUT
    assert raw.qpkv_error_status(0) == 0


def test_bounded_wait_runs_out_and_returns(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lib.selftest_wait_timeout(100_000, err)            # ~50 us at 2 GHz
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) == lib.DEV_ERR_TIMEOUT
    assert dt < 5.0
    # the library's word, read through the check call
    lib.selftest_wait_timeout(100_000)
    assert lib.check_errors(raise_on_error=False) == lib.DEV_ERR_TIMEOUT
    assert lib.check_errors() == 0
    # the context still runs work
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == float(np.arange(1024).sum())


def test_selftest_rejects_limits_outside_its_range(lib):
    raw = lib.load()
    s = torch.cuda.current_stream().cuda_stream
    assert raw.qpkv_selftest_wait_timeout(10, None, s) == 1
    assert raw.qpkv_selftest_wait_timeout(10 ** 10, None, s) == 1
