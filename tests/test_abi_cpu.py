"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol include/qpkv.h declares, mirrors its structs, plans on the host,
and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qpkv.h")


@pytest.fixture(scope="module")
def qlib():
    import quantized_paged_kv_varlen_gb300 as q
    from quantized_paged_kv_varlen_gb300 import build
    if not os.path.exists(q.LIB_PATH):
        build.build()
    return q, q.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qpkv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(qlib):
    _, lib = qlib
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_struct_mirror_and_strings(qlib):
    q, lib = qlib
    assert lib.qpkv_struct_size(0) == ctypes.sizeof(q.WriteParams)
    assert lib.qpkv_struct_size(1) == ctypes.sizeof(q.PrefillParams)
    assert lib.qpkv_struct_size(2) == ctypes.sizeof(q.MlaParams)
    assert lib.qpkv_struct_size(99) == 0
    assert lib.qpkv_status_string(0) == b"ok"
    assert lib.qpkv_status_string(3) == b"workspace too small"
    assert lib.qpkv_version() >= 100


PLAN_LEN = 24   # QPKV_PLAN_INFO_LEN


def test_plan_info_length_matches_header():
    import re
    from pathlib import Path
    import quantized_paged_kv_varlen_gb300 as q
    hdr = (Path(__file__).resolve().parent.parent / "include" / "qpkv.h").read_text()
    n = int(re.search(r"#define QPKV_PLAN_INFO_LEN (\d+)", hdr).group(1))
    assert n == PLAN_LEN == q.PLAN_INFO_LEN


def _plan(lib, lens, Hq=32, Hkv=8, ps=16, D=128, sms=148):
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    ib, fb = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib.qpkv_decode_workspace_sizes(lens.ctypes.data, len(lens), Hq, Hkv, D, sms,
                                         ctypes.byref(ib), ctypes.byref(fb))
    assert st == 0
    host = np.zeros(ib.value, dtype=np.uint8)
    info = (ctypes.c_int64 * PLAN_LEN)()
    st = lib.qpkv_decode_plan_host(lens.ctypes.data, len(lens), Hq, Hkv, ps, D, sms,
                                   host.ctypes.data, host.nbytes, info)
    assert st == 0
    n_items, chunk, total_splits, items_off, split_off_off = (info[i] for i in range(5))
    int_bytes, float_bytes, kind, counter_off = info[5], info[6], info[13], info[14]
    assert int_bytes <= ib.value and float_bytes <= fb.value
    items = host[items_off:items_off + 32 * n_items].view(np.int32).reshape(n_items, 8)
    split_off = host[split_off_off:split_off_off + 4 * (len(lens) + 1)].view(np.int32)
    counters = host[counter_off:counter_off + 8].view(np.int32) if kind == 1 else None
    return dict(info=list(info), items=items, split_off=split_off, chunk=chunk, kind=kind,
                total_splits=total_splits, float_bytes=fb.value, counters=counters)


@pytest.mark.parametrize("Hq,Hkv,kind", [(64, 8, 0), (8, 2, 0), (16, 4, 1), (32, 8, 1)])
def test_decode_plan_covers_every_token_once(qlib, Hq, Hkv, kind):
    _, lib = qlib
    rng = np.random.default_rng(0)
    lens = rng.integers(0, 3000, 40)
    lens[[3, 7]] = 0
    lens[5] = 256
    lens[6] = 257
    p = _plan(lib, lens, Hq=Hq, Hkv=Hkv, ps=32)
    assert p["kind"] == kind
    chunk = p["chunk"]
    heads = Hkv if kind == 0 else 1
    cover = {}
    for b, h, t0, t1, slot, *_ in p["items"].tolist():
        assert 0 <= t0 < t1 <= lens[b] and t1 - t0 <= chunk and t0 % chunk == 0
        assert slot == p["split_off"][b] + t0 // chunk
        assert 0 <= h < heads
        cover.setdefault((b, h), []).append((t0, t1))
    for b, L in enumerate(lens):
        for h in range(heads):
            spans = sorted(cover.get((b, h), []))
            assert sum(t1 - t0 for t0, t1 in spans) == L
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
    splits = [(L + chunk - 1) // chunk for L in lens]
    assert p["split_off"].tolist() == np.concatenate([[0], np.cumsum(splits)]).tolist()
    assert p["total_splits"] == sum(splits)
    it = p["items"]
    if kind == 0:
        # items of one token range are adjacent across kv heads
        assert np.all(it[0::Hkv, 1] == 0) and np.all(it[1::Hkv, 1] == 1)
        assert np.array_equal(it[0::Hkv, [0, 2]], it[1::Hkv, [0, 2]])
    else:
        # one item per token range, handed out largest first, counters armed
        sizes = it[:, 3] - it[:, 2]
        assert np.all(np.diff(sizes) <= 0)
        assert p["counters"].tolist() == [0, 0]
    assert p["float_bytes"] >= sum(splits) * Hq * 129 * 4


def test_small_batches_use_smaller_items(qlib):
    _, lib = qlib
    assert _plan(lib, [37, 100], Hq=4, Hkv=1, D=64)["chunk"] == 128
    assert _plan(lib, [4000] * 64)["chunk"] == 256              # all heads: 16 tiles of 16 tokens
    assert _plan(lib, [4000] * 64, Hq=64)["chunk"] == 512       # per kv head
    assert _plan(lib, [300] * 64, Hq=64, sms=148)["chunk"] == 256


@pytest.mark.parametrize("args,want", [
    (dict(B=0), 1), (dict(lens=[5, -1]), 1), (dict(D=96), 2), (dict(Hq=64, Hkv=4), 2),
    (dict(Hq=12, Hkv=8), 1)])
def test_decode_sizes_rejects_bad_arguments(qlib, args, want):
    _, lib = qlib
    lens = np.ascontiguousarray(args.get("lens", [5, 6]), dtype=np.int32)
    B = args.get("B", len(lens))
    ib, fb = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib.qpkv_decode_workspace_sizes(lens.ctypes.data, B, args.get("Hq", 32),
                                         args.get("Hkv", 8), args.get("D", 128), 148,
                                         ctypes.byref(ib), ctypes.byref(fb))
    assert st == want


def test_plan_rejects_page_size_and_small_buffers(qlib):
    _, lib = qlib
    lens = np.ascontiguousarray([100, 200], dtype=np.int32)
    host = np.zeros(1 << 16, dtype=np.uint8)
    info = (ctypes.c_int64 * PLAN_LEN)()
    assert lib.qpkv_decode_plan_host(lens.ctypes.data, 2, 32, 8, 24, 128, 148,
                                     host.ctypes.data, host.nbytes, info) == 2
    assert lib.qpkv_decode_plan_host(lens.ctypes.data, 2, 32, 8, 16, 128, 148,
                                     host.ctypes.data, 8, info) == 3


def test_run_rejects_foreign_plan_and_null_pointers(qlib):
    _, lib = qlib
    bogus = (ctypes.c_int64 * PLAN_LEN)(*([7] * PLAN_LEN))
    fake = ctypes.c_void_p(0x100000)
    st = lib.qpkv_decode_run(bogus, fake, 1 << 20, fake, fake, fake, fake, fake, fake, 10, 16,
                             fake, 4, ctypes.c_float(0.1), fake, None, None, None)
    assert st == 1
    p = _plan(lib, [100, 200])
    info = (ctypes.c_int64 * PLAN_LEN)(*p["info"])
    st = lib.qpkv_decode_run(info, None, 1 << 20, fake, fake, fake, fake, fake, fake, 10, 16,
                             fake, 4, ctypes.c_float(0.1), fake, None, None, None)
    assert st == 1
    st = lib.qpkv_decode_run(info, fake, 16, fake, fake, fake, fake, fake, fake, 10, 16,
                             fake, 16, ctypes.c_float(0.1), fake, None, None, None)
    assert st == 3
    assert lib.qpkv_decode_plan_set_kv_layout(info, 2) == 1          # unknown layout
    assert lib.qpkv_decode_plan_set_kv_layout(bogus, 1) == 1         # not a plan
    assert lib.qpkv_decode_plan_set_kv_layout(info, 1) == 0 and info[15] == 1
    misaligned = ctypes.c_void_p(0x100004)
    st = lib.qpkv_decode_run(info, fake, 1 << 30, fake, misaligned, fake, fake, fake, fake, 10,
                             16, fake, 16, ctypes.c_float(0.1), fake, None, None, None)
    assert st == 1
    # 200 tokens in pages of 16 need 13 block_table entries per row
    st = lib.qpkv_decode_run(info, fake, 1 << 30, fake, fake, fake, fake, fake, fake, 10, 16,
                             fake, 12, ctypes.c_float(0.1), fake, None, None, None)
    assert st == 1


def test_write_cache_rejects_before_launch(qlib):
    q, lib = qlib
    assert lib.qpkv_write_cache(None, None) == 1
    p = q.WriteParams()
    fake = 0x100000
    for n in ("cu_seqlens_q", "block_table", "k", "v", "k_pool", "v_pool", "k_scale_pool",
              "v_scale_pool", "q", "q_out", "k_block_scale", "q_block_scale"):
        setattr(p, n, fake)
    p.num_seqs, p.num_tokens, p.num_heads_kv, p.head_dim = 2, 10, 1, 128
    p.page_size, p.num_pages, p.bt_stride = 16, 4, 2
    p.mode = 7
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 2
    p.mode = 0
    p.page_size = 24
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 2
    p.page_size = 16
    p.head_dim = 96
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 2
    p.head_dim = 128
    p.k = fake + 4
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.k = fake
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1   # FP8 mode: q without RoPE tables
    p.rope_cos = fake
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1   # ... or with one table only
    p.rope_cos = None
    p.mode = 1                       # INT8 mode: start_pos must be NULL, tables present
    p.num_heads_q = 1
    p.start_pos = fake
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.start_pos = None
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1   # no RoPE tables
    p.rope_cos, p.rope_sin, p.rope_max_pos, p.max_seqlen, p.num_blocks = fake, fake, 64, 10, 1
    p.flags = 2                      # unknown flag
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 2
    p.flags = 1                      # K smoothing: needs k_mean and scratch
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.k_mean, p.workspace, p.workspace_bytes = fake, fake, 8
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 3
    assert lib.qpkv_smooth_workspace_bytes(2, 1, 1) == 2 * 128 * (8 + 4)
    p.flags, p.k_mean = 4, None      # FP8 V: needs the channel-scale output
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.v_channel_scale = fake         # ... and the scratch
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 3
    p.v_channel_scale = None
    p.flags = 0
    p.rope_cos, p.rope_sin, p.rope_max_pos = None, None, 0
    p.mode = 2                       # MLA needs head_dim 576
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 2
    p.head_dim = 576                 # MLA: rotating q needs the RoPE tables
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.rope_cos = fake                # ... both of them, with rows
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1
    p.rope_sin, p.rope_max_pos = fake, 64
    p.q = fake + 8                   # misaligned query rows
    assert lib.qpkv_write_cache(ctypes.byref(p), None) == 1



def test_prefill_rejects_before_launch(qlib):
    q, lib = qlib
    assert lib.qpkv_prefill_paged(None, None) == 1
    assert lib.qpkv_prefill_workspace_bytes(8, 1000, 4) >= 4 * (1 + 5 * 8) + 32 * 4 * (4 + 8)
    assert lib.qpkv_prefill_workspace_bytes(-1, 10, 4) == 0
    p = q.PrefillParams()
    fake = 0x100000
    for n in ("cu_seqlens_q", "seqlens_kv", "block_table", "q", "q_block_scale", "k_pool",
              "k_block_scale", "v_pool", "o", "workspace"):
        setattr(p, n, fake)
    p.num_seqs, p.num_tokens, p.num_heads_q, p.num_heads_kv = 2, 300, 4, 2
    p.head_dim, p.page_size, p.num_pages, p.bt_stride, p.num_blocks = 128, 64, 10, 5, 3
    p.causal = 1
    p.workspace_bytes = lib.qpkv_prefill_workspace_bytes(2, 300, 4)
    p.head_dim = 64
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 2
    p.head_dim = 128
    for ps in (24, 48, 192, 32768):   # not a multiple of 16 dividing 128 or of 128, or too long
        p.page_size = ps
        assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 2
    p.page_size = 64
    p.num_heads_q = 65536          # the head index is packed into 16 bits
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 2
    p.num_heads_q = 4
    p.num_heads_kv = 3             # 4 q heads do not group over 3 kv heads
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 2
    p.num_heads_kv = 2
    p.v_pool = fake + 8
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 1
    p.v_pool = fake
    p.workspace_bytes = 8
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 3
    p.workspace_bytes = lib.qpkv_prefill_workspace_bytes(2, 300, 4)
    p.num_blocks = 0
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 1
    p.num_blocks = 3
    p.num_tokens = 0               # nothing to do: OK without touching memory
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 0


def test_mla_rejects_before_launch(qlib):
    q, lib = qlib
    assert lib.qpkv_mla_sparse_decode(None, None) == 1
    assert lib.qpkv_mla_workspace_bytes(32, 2048) >= 32 * 128 * 2048 * 2 + 32 * 2048 * 4
    assert lib.qpkv_mla_workspace_bytes(-1, 2048) == 0
    p = q.MlaParams()
    fake = 0x100000
    for n in ("cu_seqlens_q", "seqlens_kv", "block_table", "q", "kv_pool", "sparse_indices", "o",
              "workspace"):
        setattr(p, n, fake)
    p.num_seqs, p.num_tokens, p.num_heads_q, p.head_dim_qk, p.head_dim_v = 2, 2, 128, 576, 512
    p.block_size, p.num_blocks, p.bt_stride, p.sparse_size = 64, 10, 5, 256
    p.workspace_bytes = lib.qpkv_mla_workspace_bytes(2, 256)
    p.head_dim_qk = 192
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 2
    p.head_dim_qk = 576
    p.num_heads_q = 256            # more heads than one MMA tile
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 2
    p.num_heads_q = 128
    p.sparse_mode = 1
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 2
    p.sparse_mode = 3
    p.kv_pool = fake + 4
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 1
    p.kv_pool = fake
    p.workspace_bytes = 64
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 3
    p.workspace_bytes = lib.qpkv_mla_workspace_bytes(2, 256)
    p.sparse_size = 0
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 1
    p.sparse_size = 256
    p.sparse_block_size = 129      # block-wise lists: at most 128 tokens per id
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 2
    p.sparse_block_size = 4        # the workspace then covers 4x the keys
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 3
    p.sparse_block_size = 0
    p.num_tokens = 0
    assert lib.qpkv_mla_sparse_decode(ctypes.byref(p), None) == 0


def test_csr_to_block_table(qlib):
    """flashinfer's CSR page description -> block_table rows and lengths."""
    q, lib = qlib
    indptr = np.array([0, 3, 3, 5], np.int32)
    indices = np.array([7, 2, 9, 4, 1], np.int32)
    last = np.array([16, 5, 1], np.int32)
    bt, lens = q.csr_to_block_table(indptr, indices, last, 16, bt_stride=4)
    assert bt.tolist() == [[7, 2, 9, -1], [-1, -1, -1, -1], [4, 1, -1, -1]]
    assert lens.tolist() == [48, 0, 17]
    # round trip from a random block table
    rng = np.random.default_rng(4)
    L = rng.integers(0, 400, 20).astype(np.int32)
    n = (L + 15) // 16
    ptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    ids = rng.permutation(int(ptr[-1])).astype(np.int32)
    lastp = np.where(n > 0, L - (n - 1) * 16, 1).astype(np.int32)
    bt2, lens2 = q.csr_to_block_table(ptr, ids, lastp, 16)
    assert np.array_equal(lens2, L)
    for b in range(20):
        assert np.array_equal(bt2[b, :n[b]], ids[ptr[b]:ptr[b + 1]])
        assert np.all(bt2[b, n[b]:] == -1)
    # rejected descriptions
    def bad(ip, ix, lp, stride=4):
        arrs = [np.ascontiguousarray(x, np.int32) for x in (ip, ix, lp)]
        outs = [np.zeros((len(ip) - 1) * stride, np.int32), np.zeros(len(ip) - 1, np.int32)]
        return lib.qpkv_csr_to_block_table(arrs[0].ctypes.data, arrs[1].ctypes.data,
                                           arrs[2].ctypes.data, len(ip) - 1, 16, stride,
                                           outs[0].ctypes.data, outs[1].ctypes.data)
    assert bad([0, 2], [1, 2], [0]) == 1          # last page holds no token
    assert bad([0, 2], [1, 2], [17]) == 1         # more than a page
    assert bad([0, 3, 2], [1, 2, 3], [1, 1]) == 1 # decreasing indptr
    assert bad([1, 3], [1, 2, 3], [1]) == 1       # indptr not starting at 0
    assert bad([0, 5], [1, 2, 3, 4, 5], [1]) == 1  # more pages than the row holds
    assert bad([0, 2], [1, 2], [3]) == 0


def test_prefill_ragged_rejects_before_launch(qlib):
    q, lib = qlib
    p = q.PrefillParams()
    fake = 0x100000
    for n in ("cu_seqlens_q", "cu_seqlens_kv", "q", "q_block_scale", "k_pool", "k_block_scale",
              "v_pool", "o", "workspace"):
        setattr(p, n, fake)
    p.num_seqs, p.num_tokens, p.num_heads_q, p.num_heads_kv = 2, 300, 4, 2
    p.head_dim, p.num_blocks, p.num_kv_tokens, p.causal = 128, 3, 500, 1
    p.workspace_bytes = lib.qpkv_prefill_workspace_bytes(2, 300, 4)
    p.page_size = 24                # ignored with ragged K/V
    p.num_kv_tokens = -1
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 1
    p.num_kv_tokens = 500
    p.k_pool = None
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 1
    p.k_pool = fake
    p.num_tokens = 0
    assert lib.qpkv_prefill_paged(ctypes.byref(p), None) == 0

def test_binding_raises_without_library(tmp_path):
    import quantized_paged_kv_varlen_gb300 as q
    saved = q._lib
    q._lib = None
    try:
        with pytest.raises(ImportError):
            q.load(str(tmp_path / "missing.so"))
    finally:
        q._lib = saved
