"""GPU parity: dense FP8 attention forward (FA-v3 descale API) against the
CPU oracle, through the C ABI.  P enters the PV product as E4M3, so the
output bound is relative L2 <= 2e-2 with the elementwise max-abs 1e-2 of
every attention path; the lse is checked to 1e-3."""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import quant as oquant
from quantized_paged_kv_varlen_gb300 import synth
from tests.gpu_util import REL_L2_FP8_P, assert_attention_close, assert_lse_close, bf16_to_f64

pytestmark = pytest.mark.gpu


def _quantize_bsnd(x):
    """float32 [B, S, H, D] -> E4M3 codes and one descale per (b, h)."""
    amax = np.abs(x).max(axis=(1, 3))                        # [B, H]
    scale = oquant.absmax_scale(amax, oquant.FP8_QMAX)       # [B, H]
    codes = oquant.quant_fp8(x, scale[:, None, :, None])
    return codes, scale


def _inputs(seed, B, Sq, Sk, Hq, Hkv, D=128, k_grow=None):
    rng = np.random.default_rng((seed, 41))
    q = rng.standard_normal((B, Sq, Hq, D), dtype=np.float32)
    k = rng.standard_normal((B, Sk, Hkv, D), dtype=np.float32)
    v = rng.standard_normal((B, Sk, Hkv, D), dtype=np.float32)
    if k_grow is not None:      # keys from token k_grow on are 6x larger
        k[:, k_grow:] *= 6.0
    q8, qd = _quantize_bsnd(q)
    k8, kd = _quantize_bsnd(k)
    v8, vd = _quantize_bsnd(v)
    return q8, k8, v8, qd, kd, vd


def _run(lib, q8, k8, v8, qd, kd, vd, scale, causal):
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    B, Sq, Hq, D = q8.shape
    lse = torch.full((B, Sq, Hq), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = lib.fp8_attn_fwd(t(q8), t(k8), t(v8), t(qd), t(kd), t(vd), softmax_scale=scale,
                           causal=causal, lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def _check(got_o, got_lse, want_o, want_lse):
    assert_attention_close(got_o, want_o, rel=REL_L2_FP8_P)
    assert_lse_close(got_lse, want_lse)


@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,causal", [
    (1, 128, 128, 1, 1, True),       # one tile, diagonal mask
    (2, 300, 300, 4, 2, True),       # ragged tail, GQA 2:1, paired q tiles
    (1, 200, 457, 2, 2, True),       # Sq < Sk: every row sees Sk - Sq + i + 1 keys
    (1, 457, 200, 2, 1, True),       # Sq > Sk: the first 257 rows see no key
    (1, 130, 390, 2, 2, False),      # no mask, ragged key tail
    (2, 640, 640, 2, 2, True),       # five q tiles: pairs (0,4) (1,3) (2)
])
def test_fp8_attn_shapes(lib, B, Sq, Sk, Hq, Hkv, causal):
    q8, k8, v8, qd, kd, vd = _inputs(B * 1000 + Sq, B, Sq, Sk, Hq, Hkv)
    scale = 1.0 / np.sqrt(128.0)
    got_o, got_lse = _run(lib, q8, k8, v8, qd, kd, vd, scale, causal)
    want_o, want_lse = oatt.dense_fp8(q8, k8, v8, qd, kd, vd, scale, causal)
    _check(got_o, got_lse, want_o, want_lse)
    if causal and Sq > Sk:
        none = np.arange(Sq) + Sk - Sq < 0
        assert np.all(got_o[:, none] == 0.0)
        assert np.all(np.isneginf(got_lse[:, none]))


def test_fp8_attn_running_max_jumps(lib):
    """Keys 6x larger from token 300 on: later tiles beat the running
    maximum by far more than 2^8 and the accumulated O rows are rescaled."""
    q8, k8, v8, qd, kd, vd = _inputs(7, 1, 768, 768, 2, 2, k_grow=300)
    scale = 1.0 / np.sqrt(128.0)
    got_o, got_lse = _run(lib, q8, k8, v8, qd, kd, vd, scale, True)
    want_o, want_lse = oatt.dense_fp8(q8, k8, v8, qd, kd, vd, scale, True)
    _check(got_o, got_lse, want_o, want_lse)


def test_fp8_attn_full_size_sampled(lib):
    """B=4, S=8192, H=32, D=128, causal: the benchmark's launch; the oracle
    checks sampled rows of a few (batch, head) pairs."""
    B, S, H, D = 4, 8192, 32, 128
    q8, k8, v8, qd, kd, vd = synth.dense_fp8_device(0, B, S, H, D, "cuda")
    lse = torch.empty((B, S, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(128.0)
    out = lib.fp8_attn_fwd(q8, k8, v8, qd, kd, vd, softmax_scale=scale, causal=True, lse=lse,
                           error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = [0, 1, 127, 128, 129, 2047, 4096, 6143, 8190, 8191]
    for b, h in [(0, 0), (1, 17), (3, 31)]:
        sl = lambda t, hh: t[b:b + 1, :, hh:hh + 1].cpu().numpy()
        want_o, want_lse = oatt.dense_fp8(
            sl(q8, h), sl(k8, h), sl(v8, h), qd[b:b + 1, h:h + 1].cpu().numpy(),
            kd[b:b + 1, h:h + 1].cpu().numpy(), vd[b:b + 1, h:h + 1].cpu().numpy(), scale, True,
            rows=[(0, s, 0) for s in rows])
        got_o = bf16_to_f64(out[b, rows, h])
        got_lse = lse[b, rows, h].cpu().numpy().astype(np.float64)
        assert_attention_close(got_o, want_o[0, rows, 0], rel=REL_L2_FP8_P, what=f"O(b={b}, h={h})")
        assert_lse_close(got_lse, want_lse[0, rows, 0])
