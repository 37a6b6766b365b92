"""Seeded synthetic inputs shaped like the five paged-attention workloads.

This module draws random numbers and lays them out; it holds none of the
attention, quantisation or RoPE arithmetic (those live in the CUDA library
and, independently, in the CPU oracle).  Both sides are fed from here.

Every array is numpy.  Values meant to be bf16 are float32 arrays whose
entries are bf16-representable (N(0,1) draws rounded to nearest-even bf16),
so ``torch.from_numpy(x).to(torch.bfloat16)`` is exact.  Each request's
K/V (and each (batch, head) slice of the dense workload) comes from its own
generator ``default_rng((seed, workload, index))``, so a test can regenerate
the slices it samples without drawing the whole workload.
"""
from dataclasses import dataclass, field

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest-even bf16 value."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    u = ((u + rounding) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_round(rng.standard_normal(shape, dtype=np.float32))


def page_tables(rng, lengths, page_size, extra_pages=0, fill=-1):
    """Random page assignment: a pool of exactly sum(ceil(L/ps)) (+extra)
    pages, randomly permuted and handed out in request order.
    Returns (block_table int32 [B, W], num_pages); unused entries = fill."""
    n_pages = [(int(L) + page_size - 1) // page_size for L in lengths]
    total = int(sum(n_pages)) + int(extra_pages)
    perm = rng.permutation(total).astype(np.int32)
    W = max(1, max(n_pages) if n_pages else 1)
    bt = np.full((len(lengths), W), fill, dtype=np.int32)
    off = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, total


def inclusive_prefix(lengths):
    return np.cumsum(np.asarray(lengths, dtype=np.int64)).astype(np.int32)


# --------------------------------------------------------------- paged decode

@dataclass
class DecodeWorkload:
    """One query token per request over an FP8 paged cache holding L_b tokens.

    q [B, Hq, D]; kv(b) -> (k, v) float32 [L_b, Hkv, D] for request b.
    """
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    lengths: np.ndarray
    block_table: np.ndarray
    num_pages: int
    q: np.ndarray
    scale: float
    workload_id: int = 2

    def kv(self, b: int):
        rng = np.random.default_rng((self.seed, self.workload_id, 1000 + b))
        L = int(self.lengths[b])
        k = bf16_normal(rng, (L, self.Hkv, self.D))
        v = bf16_normal(rng, (L, self.Hkv, self.D))
        return k, v

    def kv_all(self):
        """TND concatenation of every request's K and V (prefix order)."""
        ks, vs = zip(*(self.kv(b) for b in range(self.B)))
        return np.concatenate(ks), np.concatenate(vs)

    @property
    def cu_seqlens(self):
        return inclusive_prefix(self.lengths)


def tiny_decode(seed: int = 0) -> DecodeWorkload:
    """B=2, L={37,100}, Hq=4, Hkv=1 (GQA 4:1), D=64, page 16, 10 pages."""
    rng = np.random.default_rng((seed, 1))
    lengths = np.array([37, 100], dtype=np.int32)
    bt, P = page_tables(rng, lengths, 16)
    q = bf16_normal(rng, (2, 4, 64))
    return DecodeWorkload(seed, 2, 4, 1, 64, 16, lengths, bt, P, q,
                          1.0 / np.sqrt(64.0), workload_id=1)


def batched_decode(seed: int = 0, B: int = 64, lo: int = 512, hi: int = 8192,
                   Hq: int = 32, Hkv: int = 8, D: int = 128,
                   page_size: int = 16) -> DecodeWorkload:
    """Llama-3-8B-shaped heads: B requests, L ~ U{lo..hi}, page 16."""
    rng = np.random.default_rng((seed, 2))
    lengths = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    bt, P = page_tables(rng, lengths, page_size)
    q = bf16_normal(rng, (B, Hq, D))
    return DecodeWorkload(seed, B, Hq, Hkv, D, page_size, lengths, bt, P, q,
                          1.0 / np.sqrt(float(D)), workload_id=2)


# ------------------------------------------------------ varlen INT8 prefill

@dataclass
class PrefillWorkload:
    """Packed TND sequences, causal, K/V written into a page-64 cache."""
    seed: int
    lengths: np.ndarray
    H: int
    D: int
    page_size: int
    block_table: np.ndarray
    num_pages: int
    theta: float
    scale: float
    q: np.ndarray = field(repr=False)
    k: np.ndarray = field(repr=False)
    v: np.ndarray = field(repr=False)

    @property
    def cu_seqlens(self):
        return inclusive_prefix(self.lengths)

    @property
    def num_blocks(self):
        return int((int(np.max(self.lengths)) + 127) // 128)


def varlen_prefill(seed: int = 0, B: int = 8, lo: int = 256, hi: int = 4096,
                   H: int = 32, D: int = 128, page_size: int = 64,
                   lengths=None) -> PrefillWorkload:
    rng = np.random.default_rng((seed, 3))
    if lengths is None:
        lengths = rng.integers(lo, hi + 1, size=B)
    lengths = np.asarray(lengths, dtype=np.int32)
    bt, P = page_tables(rng, lengths, page_size)
    T = int(lengths.sum())
    q = bf16_normal(rng, (T, H, D))
    k = bf16_normal(rng, (T, H, D))
    v = bf16_normal(rng, (T, H, D))
    return PrefillWorkload(seed, lengths, H, D, page_size, bt, P, 1.0e4,
                           1.0 / np.sqrt(float(D)), q, k, v)


# ------------------------------------------------------------ dense FP8

@dataclass
class DenseWorkload:
    """BSND N(0,1) draws for Q, K, V; quantised to E4M3 per (b, h) by the user."""
    seed: int
    B: int
    S: int
    H: int
    D: int
    scale: float

    def slice(self, which: str, b: int, h: int) -> np.ndarray:
        """float32 [S, D] draws of tensor which in {'q','k','v'} at (b, h)."""
        tag = {"q": 0, "k": 1, "v": 2}[which]
        rng = np.random.default_rng((self.seed, 4, tag, b, h))
        return rng.standard_normal((self.S, self.D), dtype=np.float32)

    def tensor(self, which: str) -> np.ndarray:
        out = np.empty((self.B, self.S, self.H, self.D), dtype=np.float32)
        for b in range(self.B):
            for h in range(self.H):
                out[b, :, h] = self.slice(which, b, h)
        return out


def dense_fp8(seed: int = 0, B: int = 4, S: int = 8192, H: int = 32,
              D: int = 128) -> DenseWorkload:
    return DenseWorkload(seed, B, S, H, D, 1.0 / np.sqrt(float(D)))


def dense_fp8_device(seed: int, B: int, S: int, H: int, D: int, device):
    """Full-size FP8 inputs made on the GPU: for q, k and v in turn, N(0,1)
    float32 draws [B, S, H, D] from a seeded device generator, one fp32
    descale per (b, h) = absmax / 448, codes = torch's float8_e4m3fn cast of
    x / descale (round to nearest even) viewed as uint8.
    Returns q8, k8, v8, q_descale, k_descale, v_descale."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for _ in range(3):
        x = torch.randn((B, S, H, D), generator=g, device=device, dtype=torch.float32)
        scale = x.abs().amax(dim=(1, 3)) / 448.0
        codes = (x / scale[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        out.append((codes.contiguous(), scale.contiguous()))
        del x
    (q8, qd), (k8, kd), (v8, vd) = out
    return q8, k8, v8, qd, kd, vd


# ------------------------------------------------------ MLA sparse decode

@dataclass
class MlaWorkload:
    """q [B, QN, 576]; kv(b) -> [L_b, 576] draws (nope || rope);
    sparse_indices [B, 1, S] distinct ids of request b, -1 padded."""
    seed: int
    B: int
    QN: int
    lengths: np.ndarray
    block_size: int
    block_table: np.ndarray
    num_pages: int
    q: np.ndarray
    sparse_indices: np.ndarray
    scale: float

    def kv(self, b: int) -> np.ndarray:
        rng = np.random.default_rng((self.seed, 5, 1000 + b))
        return bf16_normal(rng, (int(self.lengths[b]), 576))

    @property
    def cu_seqlens_q(self):
        return np.arange(1, self.B + 1, dtype=np.int32)


def mla_sparse(seed: int = 0, B: int = 32, QN: int = 128, lo: int = 32768,
               hi: int = 65536, block_size: int = 64, topk: int = 2048,
               sparse_size: int = 2048, lengths=None) -> MlaWorkload:
    rng = np.random.default_rng((seed, 5))
    if lengths is None:
        lengths = rng.integers(lo, hi + 1, size=B)
    lengths = np.asarray(lengths, dtype=np.int32)
    bt, P = page_tables(rng, lengths, block_size)
    q = bf16_normal(rng, (B, QN, 576))
    idx = np.full((B, 1, sparse_size), -1, dtype=np.int32)
    for b in range(B):
        n = min(topk, int(lengths[b]), sparse_size)
        idx[b, 0, :n] = rng.permutation(int(lengths[b]))[:n]
    return MlaWorkload(seed, B, QN, lengths, block_size, bt, P, q, idx,
                       1.0 / np.sqrt(576.0))


def mla_sparse_device(seed: int, device, B: int = 32, QN: int = 128, lo: int = 32768,
                      hi: int = 65536, block_size: int = 64, topk: int = 2048,
                      sparse_size: int = 2048):
    """Full-size MLA inputs with the bulk made on the GPU: lengths, the page
    permutation and the sparse ids from numpy (seed, 6); q [B, QN, 576] and
    the cache rows' values kv [sum L, 576] as N(0,1) draws of a seeded torch
    device generator, rounded to bf16.  Returns a dict of device tensors
    (and the host lengths / block table)."""
    import torch
    rng = np.random.default_rng((seed, 6))
    lengths = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    bt, P = page_tables(rng, lengths, block_size)
    idx = np.full((B, 1, sparse_size), -1, dtype=np.int32)
    for b in range(B):
        n = min(topk, int(lengths[b]), sparse_size)
        idx[b, 0, :n] = rng.permutation(int(lengths[b]))[:n]
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 6)
    q = torch.randn((B, QN, 576), generator=g, device=device).to(torch.bfloat16)
    kv = torch.randn((int(lengths.sum()), 576), generator=g, device=device).to(torch.bfloat16)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return dict(lengths=lengths, block_table=bt, num_pages=P, block_size=block_size, q=q, kv=kv,
                idx=dev(idx), bt=dev(bt), lk=dev(lengths), cu_kv=dev(inclusive_prefix(lengths)),
                cu_q=dev(np.arange(1, B + 1, dtype=np.int32)), scale=1.0 / np.sqrt(576.0))
