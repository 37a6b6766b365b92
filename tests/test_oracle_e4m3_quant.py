"""Pins for the oracle's E4M3 codec and absmax quantizers (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3, quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_decode_anchors():
    for code, value in _rows("e4m3_anchors.txt"):
        got = e4m3.decode(np.array([int(code, 16)], dtype=np.uint8))[0]
        assert got == float(value)
        assert np.signbit(got) == value.startswith("-")
    assert np.isnan(e4m3.decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    finite = e4m3.DECODE_TABLE[np.isfinite(e4m3.DECODE_TABLE)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert np.sum(np.isnan(e4m3.DECODE_TABLE)) == 2


def test_encode_hand_worked_rounding():
    for value, code, *_ in _rows("e4m3_rounding.txt"):
        got = e4m3.encode_rne_satfinite(np.array([float(value)], dtype=np.float32))[0]
        assert got == int(code, 16), value


def test_encode_decode_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    finite = np.isfinite(e4m3.DECODE_TABLE)
    back = e4m3.encode_rne_satfinite(e4m3.DECODE_TABLE[finite].astype(np.float32))
    assert np.array_equal(back, codes[finite])


def test_encode_matches_torch_cast_exhaustively_on_midpoints():
    """torch's float8_e4m3fn cast (a library routine) on values pre-clamped to
    +-448, including every midpoint between neighbouring codes and random
    float32 values across the whole range."""
    pos = np.unique(e4m3.DECODE_TABLE[np.isfinite(e4m3.DECODE_TABLE)])
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(7)
    rand = rng.uniform(-448, 448, 200000)
    tiny = rng.uniform(-2 ** -5, 2 ** -5, 50000)
    nudged = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                             np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    x = np.concatenate([pos, -pos, mids, -mids, rand, tiny, nudged, -nudged]).astype(np.float32)
    x = np.clip(x, -448, 448)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3.encode_rne_satfinite(x)
    assert np.array_equal(got, want)


def test_fp8_quant_absmax_maps_to_448_and_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 8, 128)).astype(np.float32)
    codes, scale = quant.quant_fp8_last_axis(x)
    assert scale.dtype == np.float32
    assert np.array_equal(scale, (np.abs(x).max(-1) / np.float32(448)).astype(np.float32))
    arg = np.abs(x).argmax(-1)
    top = np.take_along_axis(codes, arg[..., None], -1)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    deq = quant.dequant_fp8(codes, scale[..., None])
    y = x.astype(np.float64) / scale[..., None]
    # half an E4M3 quantum at the value (2^-10 absolute in the subnormal range)
    q = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 1e-30))), -6) - 3)
    assert np.all(np.abs(deq / scale[..., None] - y) <= q / 2 * (1 + 1e-6))
    # idempotent: re-quantising the dequantised value with the same scale
    again = quant.quant_fp8(deq.astype(np.float32), scale[..., None])
    assert np.array_equal(again, codes)


def test_int8_quant_hand_worked_and_bounds():
    x = np.array([[127.0, -63.5, 0.5, 1.5, -2.5, 0.0]], dtype=np.float32)
    codes, scale = quant.quant_int8_last_axis(x)
    assert scale[0] == np.float32(1.0)
    # ties to even: -63.5 -> -64, 0.5 -> 0, 1.5 -> 2, -2.5 -> -2
    assert codes[0].tolist() == [127, -64, 0, 2, -2, 0]
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 100, (500, 1))).astype(np.float32)
    codes, scale = quant.quant_int8_last_axis(x)
    assert codes.min() >= -127 and codes.max() <= 127
    assert np.all(np.abs(codes).max(-1) == 127)
    deq = quant.dequant_int8(codes, scale[:, None])
    assert np.all(np.abs(deq - x) <= scale[:, None].astype(np.float64) * 0.5 * (1 + 1e-5))
    again = quant.quant_int8(deq.astype(np.float32), scale[:, None])
    assert np.array_equal(again, codes)


def test_zero_rows_give_zero_scale_and_codes():
    x = np.zeros((3, 16), dtype=np.float32)
    c8, s8 = quant.quant_fp8_last_axis(x)
    ci, si = quant.quant_int8_last_axis(x)
    assert np.all(s8 == 0) and np.all(c8 == 0) and np.all(si == 0) and np.all(ci == 0)


def _encode_ties_away(x):
    """A plausible wrong encoder: ties rounded away from zero."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.maximum(a, 1e-30))), -6)
    qn = np.exp2(e - 3)
    v = np.floor(a / qn + 0.5) * qn
    return e4m3.encode_rne_satfinite((np.sign(x) * v).astype(np.float32))


def test_planted_mistakes_are_caught():
    """Plausible quantizer bugs, planted in copies here, fail the pins above."""
    ties = [(float(v), int(c, 16)) for v, c, *_ in _rows("e4m3_rounding.txt")]
    xs = np.array([v for v, _ in ties], dtype=np.float32)
    want = np.array([c for _, c in ties], dtype=np.uint8)
    assert not np.array_equal(_encode_ties_away(xs), want)
    x = np.array([[3.0, 1.1, -0.7, 0.3]], dtype=np.float32)
    codes, _ = quant.quant_fp8_last_axis(x)
    bad_scale = (np.abs(x).max(-1) / np.float32(127)).astype(np.float32)
    assert not np.array_equal(quant.quant_fp8(x, bad_scale[:, None]), codes)
