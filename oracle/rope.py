"""Rotary position embedding applied on the cache-write path.

Test infrastructure only (see oracle/__init__.py).

"[Feature] Sage Attention Support Varlen & write kv cache BF16/FP16",
Description item 1, fuses RoPE into the KV-cache write; flashinfer's
"[Refactor] Unify JIT/Customization/AOT mode" interfaces carry the
``rope_theta`` / ``rope_scale`` parameters.  Neither page spells the rotation
out, so the plainest (Llama / NeoX "rotate-half") reading is taken:

    inv_freq_i = theta^(-2i/D),            i < D/2, float64
    angle      = (pos / rope_scale) * inv_freq_i, float64
    c, s       = float32(cos(angle)), float32(sin(angle))
    x'_i       = x_i * c - x_{i+D/2} * s
    x'_{i+D/2} = x_{i+D/2} * c + x_i * s

Each product and each sum is rounded to float32 separately (no fused
multiply-add), so the rotated values are reproducible bit for bit.
"""
import numpy as np

F32 = np.float32


def cos_sin_table(max_pos: int, dim: int, theta: float, rope_scale: float = 1.0):
    """float32 cos/sin tables of shape [max_pos, dim // 2]."""
    half = dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.power(np.float64(theta), -2.0 * i / np.float64(dim))
    pos = np.arange(max_pos, dtype=np.float64) / np.float64(rope_scale)
    angle = pos[:, None] * inv_freq[None, :]
    return np.cos(angle).astype(F32), np.sin(angle).astype(F32)


def rotate(x: np.ndarray, pos: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate rows x[..., D] (float32 values) at integer positions pos[...]."""
    x = np.asarray(x, dtype=F32)
    half = x.shape[-1] // 2
    c = cos[pos].astype(F32)
    s = sin[pos].astype(F32)
    # broadcast tables over any head axis between the token axis and D
    while c.ndim < x.ndim:
        c = c[..., None, :]
        s = s[..., None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    a = (x1 * c).astype(F32)
    b = (x2 * s).astype(F32)
    y1 = (a - b).astype(F32)
    a2 = (x2 * c).astype(F32)
    b2 = (x1 * s).astype(F32)
    y2 = (a2 + b2).astype(F32)
    return np.concatenate([y1, y2], axis=-1).astype(F32)
