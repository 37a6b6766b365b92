"""Symmetric absmax quantizers with fp32 scales, in IEEE float32 arithmetic.

Test infrastructure only (see oracle/__init__.py).

The pages fix the granularities, not the rounding:
* per (token, head) FP8 E4M3 scale -- "KvQuantSparseFlashAttention" README,
  功能说明 (Per-Token-Head quantisation) and the key/value dtype FLOAT8_E4M3;
* per (128-token block, head) INT8 scale for Sage-style Q/K -- "[Feature]
  Sage Attention Support Varlen & write kv cache BF16/FP16", Description
  item 2 (quant kernels made varlen-aware, so a block never crosses a
  sequence boundary);
* per (token, 128-wide D tile) INT8 scale for the MLA row -- README,
  参数说明 rows key_quant_mode / value_quant_mode = 2 (per_tile) and
  tile_size = 128.

Readings taken where the pages are silent:
  scale = float32(absmax) / float32(QMAX), QMAX = 448 (E4M3) or 127 (INT8);
  code  = round(float32(x) / scale) with IEEE float32 division;
  E4M3 rounding is nearest-even with saturation to +-448;
  INT8 rounding is nearest-even, clipped to the symmetric range [-127, 127];
  absmax == 0 stores scale 0.0 and all-zero codes;
  dequant(code, scale) = code * scale, evaluated in float64.
"""
import numpy as np

from . import e4m3

F32 = np.float32
FP8_QMAX = F32(448.0)
INT8_QMAX = F32(127.0)


def absmax_scale(absmax: np.ndarray, qmax: np.float32) -> np.ndarray:
    """fp32 scale = absmax / qmax (IEEE round-to-nearest division)."""
    return (np.asarray(absmax, dtype=F32) / qmax).astype(F32)


def _divide(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x / scale in float32; entries with scale 0 give 0 (their x is all 0)."""
    x = np.asarray(x, dtype=F32)
    scale = np.asarray(scale, dtype=F32)
    safe = np.where(scale == 0, F32(1.0), scale).astype(F32)
    y = (x / safe).astype(F32)
    return np.where(scale == 0, F32(0.0), y).astype(F32)


def quant_fp8(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """E4M3 codes of x / scale (scale broadcast against x)."""
    return e4m3.encode_rne_satfinite(_divide(x, scale))


def quant_int8(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """INT8 codes of x / scale, nearest-even, clipped to [-127, 127]."""
    y = _divide(x, scale).astype(np.float64)
    return np.clip(np.rint(y), -127, 127).astype(np.int8)


def quant_fp8_last_axis(x: np.ndarray):
    """Per-row (last axis) E4M3 quantisation: returns (codes u8, scale f32).

    Used for the per-(token, head) FP8 cache: one scale per D-vector.
    """
    x = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x), axis=-1)
    scale = absmax_scale(amax, FP8_QMAX)
    return quant_fp8(x, scale[..., None]), scale


def quant_int8_last_axis(x: np.ndarray):
    """Per-row (last axis) INT8 quantisation: returns (codes i8, scale f32)."""
    x = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x), axis=-1)
    scale = absmax_scale(amax, INT8_QMAX)
    return quant_int8(x, scale[..., None]), scale


def dequant_fp8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """float64 values codes * scale (scale broadcast)."""
    return e4m3.decode(codes) * np.asarray(scale, dtype=np.float64)


def dequant_int8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)
