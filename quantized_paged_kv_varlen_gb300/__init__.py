"""Python binding of the qpkv C-ABI library (quantized paged-KV varlen
attention on GB300).

Argument marshalling only: tensors are checked for dtype / shape /
contiguity, their device pointers and the current CUDA stream are passed to
``libqpkv.so``, and every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory (including the workspaces the
library asks for) and streams.  There is no CPU or PyTorch fallback: a
missing library raises.

The submodule ``synth`` (seeded synthetic inputs) is importable without the
library.
"""
import ctypes
import os

__all__ = [
    "QpkvError", "load", "check_errors", "selftest_wait_timeout", "rope_table", "write_cache_fp8", "write_cache_int8_block128_rope",
    "write_cache_mla", "DecodePlan", "PAGE_ROW_MLA",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqpkv.so")
PAGE_ROW_MLA = 656

WRITE_FP8_TOKEN_HEAD = 0
WRITE_INT8_BLOCK128_ROPE = 1
WRITE_MLA_ROW = 2
WRITE_SMOOTH_K = 1          # qpkv_write_params.flags
WRITE_HND = 2
WRITE_V_FP8 = 4
PLAN_INFO_LEN = 24
KV_LAYOUTS = {"NHD": 0, "HND": 1}   # K/V pool layouts of the FP8 decode path

DEV_ERR_TIMEOUT = 1
DEV_ERR_BAD_PAGE = 2
DEV_ERR_BAD_INDEX = 4
DEV_ERR_BAD_LENGTH = 8

ERR_UNSUPPORTED = 2
ERR_CUDA = 4
ERR_DEVICE = 5
ERR_TIMEOUT = 6

_lib = None


class QpkvError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: qpkv status {status} ({_status_text(status)})")


def _status_text(status):
    if _lib is None:
        return "?"
    return _lib.qpkv_status_string(status).decode()


_i32 = ctypes.c_int32
_p = ctypes.c_void_p


class WriteParams(ctypes.Structure):
    """Mirror of ``qpkv_write_params`` (include/qpkv.h)."""
    _fields_ = [(n, _i32) for n in (
        "mode", "num_seqs", "num_tokens", "max_seqlen", "num_heads_q", "num_heads_kv",
        "head_dim", "page_size", "num_pages", "bt_stride", "num_blocks", "rope_max_pos")] + [
        (n, _p) for n in (
            "cu_seqlens_q", "start_pos", "block_table", "q", "k", "v", "rope_cos", "rope_sin",
            "k_pool", "v_pool", "k_scale_pool", "v_scale_pool", "k_block_scale", "q_out",
            "q_block_scale", "slot_mapping", "error_word")] + [
        ("flags", _i32), ("pad0", _i32), ("k_mean", _p), ("workspace", _p),
        ("workspace_bytes", ctypes.c_size_t), ("v_channel_scale", _p)]



class PrefillParams(ctypes.Structure):
    """Mirror of ``qpkv_prefill_params`` (include/qpkv.h)."""
    _fields_ = [(n, _i32) for n in (
        "num_seqs", "num_tokens", "num_heads_q", "num_heads_kv", "head_dim", "page_size",
        "num_pages", "bt_stride", "num_blocks", "causal")] + [
        ("sm_scale", ctypes.c_float), ("num_kv_tokens", _i32)] + [
        (n, _p) for n in (
            "cu_seqlens_q", "seqlens_kv", "cu_seqlens_kv", "block_table", "q", "q_block_scale", "k_pool",
            "k_block_scale", "v_pool", "o", "lse", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t), ("error_word", _p), ("v_scale", _p)]


class MlaParams(ctypes.Structure):
    """Mirror of ``qpkv_mla_params`` (include/qpkv.h)."""
    _fields_ = [(n, _i32) for n in (
        "num_seqs", "num_tokens", "num_heads_q", "head_dim_qk", "head_dim_v", "block_size",
        "num_blocks", "bt_stride", "sparse_size", "sparse_mode")] + [
        ("scale", ctypes.c_float), ("sparse_block_size", _i32)] + [
        (n, _p) for n in (
            "cu_seqlens_q", "seqlens_kv", "block_table", "q", "kv_pool", "sparse_indices", "o",
            "lse", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t), ("error_word", _p)]

def _declare(lib):
    S = ctypes.c_size_t
    P64 = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "qpkv_status_string": (ctypes.c_char_p, [_i32]),
        "qpkv_version": (_i32, []),
        "qpkv_struct_size": (S, [_i32]),
        "qpkv_rope_table": (_i32, [ctypes.c_float, ctypes.c_float, _i32, _i32, _p, _p, _p]),
        "qpkv_write_cache": (_i32, [ctypes.POINTER(WriteParams), _p]),
        "qpkv_decode_workspace_sizes": (_i32, [_p, _i32, _i32, _i32, _i32, _i32,
                                               ctypes.POINTER(S), ctypes.POINTER(S)]),
        "qpkv_decode_plan_host": (_i32, [_p, _i32, _i32, _i32, _i32, _i32, _i32, _p, S, P64]),
        "qpkv_decode_plan": (_i32, [_p, _i32, _i32, _i32, _i32, _i32, _i32, _p, S, _p, S,
                                    P64, _p]),
        "qpkv_decode_run": (_i32, [P64, _p, S, _p, _p, _p, _p, _p, _p, _i32, _i32, _p, _i32,
                                   ctypes.c_float, _p, _p, _p, _p]),
        "qpkv_decode_attend": (_i32, [P64, _p, S, _p, _p, _p, _p, _p, _p, _i32, _i32, _p,
                                      _i32, ctypes.c_float, _p, _p]),
        "qpkv_decode_merge": (_i32, [P64, _p, S, _p, _p, _p, _p]),
        "qpkv_decode_plan_set_kv_layout": (_i32, [P64, _i32]),
        "qpkv_decode_static": (_i32, [_p, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                      _i32, _p, _i32, ctypes.c_float, _p, _p, _p, _p]),
        "qpkv_fp8_attn_fwd": (_i32, [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p,
                                     ctypes.c_float, _i32, _p, _p, _p, _p]),
        "qpkv_prefill_workspace_bytes": (S, [_i32, _i32, _i32]),
        "qpkv_prefill_paged": (_i32, [ctypes.POINTER(PrefillParams), _p]),
        "qpkv_csr_to_block_table": (_i32, [_p, _p, _p, _i32, _i32, _i32, _p, _p]),
        "qpkv_mla_workspace_bytes": (S, [_i32, _i32]),
        "qpkv_smooth_workspace_bytes": (S, [_i32, _i32, _i32]),
        "qpkv_mla_sparse_decode": (_i32, [ctypes.POINTER(MlaParams), _p]),
        "qpkv_error_status": (_i32, [_i32]),
        "qpkv_error_check": (_i32, [_p, ctypes.POINTER(_i32)]),
        "qpkv_selftest_wait_timeout": (_i32, [ctypes.c_int64, _p, _p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def load(path: str = LIB_PATH):
    """Load libqpkv.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"qpkv CUDA library not built: {path} is missing "
                              "(run quantized_paged_kv_varlen_gb300.build.build())")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def _check(status, where):
    if status != 0:
        raise QpkvError(status, where)


# ------------------------------------------------------------------ helpers

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, name, dtype=None, ndim=None, device=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must live on the GPU")
    return t


def rope_table(theta, max_pos, rot_dim, rope_scale=1.0, device="cuda"):
    """(cos, sin) float32 [max_pos, rot_dim // 2] computed by the library."""
    torch = _torch()
    lib = load()
    cos = torch.empty(max_pos, rot_dim // 2, dtype=torch.float32, device=device)
    sin = torch.empty_like(cos)
    _check(lib.qpkv_rope_table(float(theta), float(rope_scale), int(max_pos), int(rot_dim),
                               _ptr(cos), _ptr(sin), _stream()), "qpkv_rope_table")
    return cos, sin


def check_errors(raise_on_error=True):
    """Read and clear the library's device error word of the current GPU
    (the word kernels use when a call passed no ``error_word``); waits for
    the current stream.  Returns the QPKV_DEV_ERR_* bits, or raises
    QpkvError (status QPKV_ERR_DEVICE / QPKV_ERR_TIMEOUT) when a bit is set
    and ``raise_on_error``."""
    lib = load()
    bits = _i32(0)
    st = lib.qpkv_error_check(_stream(), ctypes.byref(bits))
    if st != 0 and (raise_on_error or st == ERR_CUDA):
        raise QpkvError(st, f"qpkv_error_check (bits {bits.value:#x})")
    return bits.value


def selftest_wait_timeout(limit_cycles, error_word=None):
    """Launch the one-CTA self-test whose mbarrier wait never completes: it
    gives up after ``limit_cycles`` SM cycles and sets DEV_ERR_TIMEOUT in
    ``error_word`` (or the library's word)."""
    _check(load().qpkv_selftest_wait_timeout(int(limit_cycles), _ptr(error_word), _stream()),
           "qpkv_selftest_wait_timeout")


def _base_params(mode, cu_seqlens, block_table, page_size, num_pages, num_tokens, max_seqlen):
    torch = _torch()
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    p = WriteParams()
    p.mode = mode
    p.num_seqs = cu_seqlens.shape[0]
    p.num_tokens = num_tokens
    p.max_seqlen = max_seqlen
    p.page_size = page_size
    p.num_pages = num_pages
    p.bt_stride = block_table.shape[1]
    p.cu_seqlens_q = _ptr(cu_seqlens)
    p.block_table = _ptr(block_table)
    return p


def write_cache_fp8(k, v, cu_seqlens, block_table, k_pool, v_pool, k_scale_pool, v_scale_pool,
                    start_pos=None, slot_mapping=None, error_word=None, kv_layout="NHD",
                    rope_cos=None, rope_sin=None, q=None, q_out=None):
    """FP8 per-(token, head) cache write.  k, v: bf16 [T, Hkv, D]; pools u8
    [P, page_size, Hkv, D] (kv_layout "HND": [P, Hkv, page_size, D]); scale
    pools float32 [P, page_size, Hkv] in both layouts.  With rope_cos /
    rope_sin (fp32 [max_pos, D/2], ``rope_table(theta, max_pos, D)``) k is
    rotated at each token's position before it is quantised; with q (bf16
    [T, Hq, D]) the rotated queries go to q_out (bf16, allocated when None,
    may be q itself), which is returned."""
    torch = _torch()
    lib = load()
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.uint8, 4)
    _need(v_pool, "v_pool", torch.uint8, 4)
    _need(k_scale_pool, "k_scale_pool", torch.float32, 3)
    _need(v_scale_pool, "v_scale_pool", torch.float32, 3)
    if kv_layout == "HND":
        P, H, ps, D = k_pool.shape
    else:
        P, ps, H, D = k_pool.shape
    p = _base_params(WRITE_FP8_TOKEN_HEAD, cu_seqlens, block_table, ps, P, k.shape[0], 0)
    p.flags = WRITE_HND if kv_layout == "HND" else 0
    p.num_heads_kv = H
    p.head_dim = D
    p.k, p.v = _ptr(k), _ptr(v)
    p.k_pool, p.v_pool = _ptr(k_pool), _ptr(v_pool)
    p.k_scale_pool, p.v_scale_pool = _ptr(k_scale_pool), _ptr(v_scale_pool)
    if rope_cos is not None:
        _need(rope_cos, "rope_cos", torch.float32, 2)
        _need(rope_sin, "rope_sin", torch.float32, 2)
        if rope_cos.shape[1] != D // 2 or tuple(rope_sin.shape) != tuple(rope_cos.shape):
            raise ValueError("RoPE tables must be [max_pos, D/2]")
        p.rope_max_pos = rope_cos.shape[0]
        p.rope_cos, p.rope_sin = _ptr(rope_cos), _ptr(rope_sin)
    if q is not None:
        if rope_cos is None:
            raise ValueError("rotating q needs the RoPE tables")
        _need(q, "q", torch.bfloat16, 3)
        if q.shape[0] != k.shape[0] or q.shape[2] != D:
            raise ValueError("q must be [T, Hq, D]")
        if q_out is None:
            q_out = torch.empty_like(q)
        _need(q_out, "q_out", torch.bfloat16, 3)
        p.num_heads_q = q.shape[1]
        p.q, p.q_out = _ptr(q), _ptr(q_out)
    p.start_pos = _ptr(start_pos)
    p.slot_mapping = _ptr(slot_mapping)
    p.error_word = _ptr(error_word)
    _check(lib.qpkv_write_cache(ctypes.byref(p), _stream()), "qpkv_write_cache(fp8)")
    return q_out


def smooth_workspace(num_seqs, num_blocks, num_heads_kv, device="cuda"):
    """Scratch for a K-smoothing INT8 write."""
    torch = _torch()
    n = int(load().qpkv_smooth_workspace_bytes(int(num_seqs), int(num_blocks), int(num_heads_kv)))
    return torch.empty(((n + 15) // 16) * 16, dtype=torch.uint8, device=device)


def write_cache_int8_block128_rope(q, k, v, cu_seqlens, block_table, max_seqlen, rope_cos,
                                   rope_sin, k_pool, v_pool, k_block_scale, q_out,
                                   q_block_scale, slot_mapping=None, error_word=None,
                                   k_mean=None, workspace=None, v_channel_scale=None):
    """Sage-style prefill write: RoPE(q, k), INT8 per-(sequence, 128-token
    block, head) Q and K, bf16 V into pages.  q/k/v bf16 [T, H, 128];
    k_pool int8 [P, ps, Hkv, 128]; v_pool bf16 [P, ps, Hkv, 128];
    k_block_scale [B, nb, Hkv]; q_out int8 [T, Hq, 128]; q_block_scale [B, nb, Hq].
    With k_mean (fp32 [B, Hkv, 128], filled) the keys are smoothed: their
    per-(sequence, head) mean is subtracted before quantising.  With
    v_channel_scale (fp32 [B, Hkv, 128], filled) V is stored as E4M3 codes
    (v_pool uint8) with one scale per (sequence, head, channel)."""
    torch = _torch()
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.int8, 4)
    _need(v_pool, "v_pool", torch.uint8 if v_channel_scale is not None else torch.bfloat16, 4)
    _need(q_out, "q_out", torch.int8, 3)
    _need(k_block_scale, "k_block_scale", torch.float32, 3)
    _need(q_block_scale, "q_block_scale", torch.float32, 3)
    _need(rope_cos, "rope_cos", torch.float32, 2)
    _need(rope_sin, "rope_sin", torch.float32, 2)
    P, ps, Hkv, D = k_pool.shape
    p = _base_params(WRITE_INT8_BLOCK128_ROPE, cu_seqlens, block_table, ps, P, k.shape[0],
                     int(max_seqlen))
    p.num_heads_q = q.shape[1]
    p.num_heads_kv = Hkv
    p.head_dim = D
    p.num_blocks = k_block_scale.shape[1]
    p.rope_max_pos = rope_cos.shape[0]
    p.q, p.k, p.v = _ptr(q), _ptr(k), _ptr(v)
    p.rope_cos, p.rope_sin = _ptr(rope_cos), _ptr(rope_sin)
    p.k_pool, p.v_pool = _ptr(k_pool), _ptr(v_pool)
    p.k_block_scale, p.q_out, p.q_block_scale = _ptr(k_block_scale), _ptr(q_out), _ptr(q_block_scale)
    p.slot_mapping = _ptr(slot_mapping)
    p.error_word = _ptr(error_word)
    for name, t in (("k_mean", k_mean), ("v_channel_scale", v_channel_scale)):
        if t is not None:
            _need(t, name, torch.float32, 3)
            if tuple(t.shape) != (p.num_seqs, Hkv, D):
                raise ValueError(f"{name} must be [B, Hkv, 128]")
    if k_mean is not None or v_channel_scale is not None:
        if workspace is None:
            workspace = smooth_workspace(p.num_seqs, p.num_blocks, Hkv, k.device)
        p.flags = (WRITE_SMOOTH_K if k_mean is not None else 0) | (
            WRITE_V_FP8 if v_channel_scale is not None else 0)
        p.k_mean, p.v_channel_scale = _ptr(k_mean), _ptr(v_channel_scale)
        p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(lib.qpkv_write_cache(ctypes.byref(p), _stream()), "qpkv_write_cache(int8)")


def write_cache_mla(kv, cu_seqlens, block_table, pool, start_pos=None, slot_mapping=None,
                    error_word=None, rope_cos=None, rope_sin=None, q=None, q_out=None):
    """MLA combined-row write: kv bf16 [T, 576] -> pool u8 [P, bs, 1, 656].

    With rope_cos / rope_sin (fp32 [max_pos, 32], ``rope_table(theta, max_pos,
    64)``) the 64-wide rope part is rotated at each token's position first;
    with q (bf16 [T, Hq, 576]) the rotated queries go to q_out (allocated
    when None, may be q itself), which is returned."""
    torch = _torch()
    lib = load()
    _need(kv, "kv", torch.bfloat16, 2)
    _need(pool, "pool", torch.uint8, 4)
    P, bs, one, W = pool.shape
    if one != 1 or W != PAGE_ROW_MLA or kv.shape[1] != 576:
        raise ValueError("MLA pool must be [P, bs, 1, 656] and kv [T, 576]")
    p = _base_params(WRITE_MLA_ROW, cu_seqlens, block_table, bs, P, kv.shape[0], 0)
    p.num_heads_kv = 1
    p.head_dim = 576
    p.k = _ptr(kv)
    p.k_pool = _ptr(pool)
    if rope_cos is not None:
        _need(rope_cos, "rope_cos", torch.float32, 2)
        _need(rope_sin, "rope_sin", torch.float32, 2)
        if rope_cos.shape[1] != 32 or tuple(rope_sin.shape) != tuple(rope_cos.shape):
            raise ValueError("MLA RoPE tables must be [max_pos, 32]")
        p.rope_max_pos = rope_cos.shape[0]
        p.rope_cos, p.rope_sin = _ptr(rope_cos), _ptr(rope_sin)
    if q is not None:
        if rope_cos is None:
            raise ValueError("rotating q needs the RoPE tables")
        _need(q, "q", torch.bfloat16, 3)
        if q.shape[0] != kv.shape[0] or q.shape[2] != 576:
            raise ValueError("q must be [T, Hq, 576]")
        if q_out is None:
            q_out = torch.empty_like(q)
        _need(q_out, "q_out", torch.bfloat16, 3)
        p.num_heads_q = q.shape[1]
        p.q, p.q_out = _ptr(q), _ptr(q_out)
    p.start_pos = _ptr(start_pos)
    p.slot_mapping = _ptr(slot_mapping)
    p.error_word = _ptr(error_word)
    _check(lib.qpkv_write_cache(ctypes.byref(p), _stream()), "qpkv_write_cache(mla)")
    return q_out


class DecodePlan:
    """Plan/run split for paged FP8 decode (one query token per request).

    ``DecodePlan(seqlens_kv, Hq, Hkv, page_size, head_dim)`` sizes and
    allocates the workspaces (torch device memory plus page-locked host
    buffers) and runs the library's host planner, which copies the work list
    to the device.  ``run`` launches the split-KV kernel and the log-sum-exp
    merge (``attend`` and ``merge`` launch them one at a time).

    The work list lives in one of two device buffers that alternate between
    plans, so the copy of a new plan never waits for, nor overwrites, the
    list that the previous run's kernels are still reading.
    """

    def __init__(self, seqlens_kv, num_qo_heads, num_kv_heads, page_size, head_dim,
                 device="cuda", num_sms=None, kv_layout="NHD"):
        torch = _torch()
        import numpy as np
        lib = load()
        lens = np.ascontiguousarray(np.asarray(seqlens_kv, dtype=np.int32))
        self.lens = lens
        self.B = int(lens.shape[0])
        self.Hq, self.Hkv, self.D, self.page_size = num_qo_heads, num_kv_heads, head_dim, page_size
        if kv_layout not in KV_LAYOUTS:
            raise ValueError("kv_layout must be 'NHD' or 'HND'")
        self.kv_layout = kv_layout
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.num_sms = int(num_sms)
        ib, fb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib.qpkv_decode_workspace_sizes(lens.ctypes.data, self.B, self.Hq, self.Hkv,
                                               self.D, self.num_sms, ctypes.byref(ib),
                                               ctypes.byref(fb)), "qpkv_decode_workspace_sizes")
        self.int_bytes, self.float_bytes = ib.value, fb.value
        n = max(self.int_bytes, 256)
        self._int_ws = [torch.empty(n, dtype=torch.uint8, device=device) for _ in range(2)]
        self.float_ws = torch.empty(max(self.float_bytes, 256), dtype=torch.uint8, device=device)
        # per buffer i: the page-locked staging of its plan (rewritten only
        # after the copy out of it is done), the plan_info, the event behind
        # that copy, and the event behind the last launch that read it
        self._pinned = [torch.empty(n, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self._info = [(ctypes.c_int64 * PLAN_INFO_LEN)() for _ in range(2)]
        self._copied = [None, None]
        self._released = [None, None]
        self._ready = None        # a side-stream copy the next launch must wait for
        self._cur = 1
        self.replan()

    @property
    def plan_info(self):
        return self._info[self._cur]

    @property
    def int_ws(self):
        return self._int_ws[self._cur]

    def replan(self, seqlens_kv=None, stream=None):
        """Run the host planner again (for new per-request lengths when
        ``seqlens_kv`` is given; they must fit the workspaces sized at
        construction) and copy the work list into the other device buffer
        (the per-step cost of the plan/run split).  The copy runs on the
        current stream, or on ``stream`` (a torch.cuda.Stream), where it
        overlaps other work on the current stream: it waits only for the
        launches that read that buffer two plans ago, and the next attend /
        merge / run waits for it."""
        torch = _torch()
        import numpy as np
        lib = load()
        if seqlens_kv is not None:
            lens = np.ascontiguousarray(np.asarray(seqlens_kv, dtype=np.int32))
            if lens.shape != self.lens.shape:
                raise ValueError("seqlens_kv must keep the batch size")
            ib, fb = ctypes.c_size_t(), ctypes.c_size_t()
            _check(lib.qpkv_decode_workspace_sizes(lens.ctypes.data, self.B, self.Hq, self.Hkv,
                                                   self.D, self.num_sms, ctypes.byref(ib),
                                                   ctypes.byref(fb)), "qpkv_decode_workspace_sizes")
            if ib.value > self._int_ws[0].numel() or fb.value > self.float_ws.numel():
                raise ValueError("new lengths need larger workspaces than this plan holds")
            self.lens = lens
        i = self._cur ^ 1
        if self._copied[i] is not None:
            self._copied[i].synchronize()       # the host may rewrite pinned[i]
        s = stream if stream is not None else torch.cuda.current_stream()
        if self._released[i] is not None:
            s.wait_event(self._released[i])     # the readers of int_ws[i] are done
        buf, info = self._pinned[i], self._info[i]
        _check(lib.qpkv_decode_plan(self.lens.ctypes.data, self.B, self.Hq, self.Hkv,
                                    self.page_size, self.D, self.num_sms,
                                    ctypes.c_void_p(buf.data_ptr()), buf.numel(),
                                    _ptr(self._int_ws[i]), self._int_ws[i].numel(), info,
                                    ctypes.c_void_p(s.cuda_stream)), "qpkv_decode_plan")
        _check(lib.qpkv_decode_plan_set_kv_layout(info, KV_LAYOUTS[self.kv_layout]),
               "qpkv_decode_plan_set_kv_layout")
        ev = torch.cuda.Event()
        ev.record(s)
        self._copied[i] = ev
        self._ready = ev if stream is not None else None
        self._cur = i

    def wait_ready(self):
        """Make the current stream wait for a pending side-stream plan copy
        (attend, merge and run do this themselves)."""
        if self._ready is not None:
            _torch().cuda.current_stream().wait_event(self._ready)
            self._ready = None

    def _after_run(self):
        ev = _torch().cuda.Event()
        ev.record()
        self._released[self._cur] = ev

    @property
    def num_items(self):
        return int(self.plan_info[0])

    @property
    def chunk(self):
        return int(self.plan_info[1])

    @property
    def total_splits(self):
        return int(self.plan_info[2])

    @property
    def kind(self):
        """0: one kv head per work item, 1: all kv heads of a token range."""
        return int(self.plan_info[13])

    def _check_run(self, q, k_pool, v_pool, k_scale_pool, v_scale_pool, block_table):
        torch = _torch()
        _need(q, "q", torch.bfloat16, 3)
        _need(k_pool, "k_pool", torch.uint8, 4)
        _need(v_pool, "v_pool", torch.uint8, 4)
        _need(k_scale_pool, "k_scale_pool", torch.float32, 3)
        _need(v_scale_pool, "v_scale_pool", torch.float32, 3)
        _need(block_table, "block_table", torch.int32, 2)
        if tuple(q.shape) != (self.B, self.Hq, self.D):
            raise ValueError(f"q must be [{self.B}, {self.Hq}, {self.D}]")
        ps_dim, h_dim = (2, 1) if self.kv_layout == "HND" else (1, 2)
        if k_pool.shape[ps_dim] != self.page_size or k_pool.shape[h_dim] != self.Hkv:
            raise ValueError("pool shape does not match the plan")

    def run(self, q, k_pool, v_pool, k_scale_pool, v_scale_pool, block_table, sm_scale,
            out=None, lse=None, error_word=None):
        torch = _torch()
        lib = load()
        self._check_run(q, k_pool, v_pool, k_scale_pool, v_scale_pool, block_table)
        if out is None:
            out = torch.empty_like(q)
        self.wait_ready()
        _check(lib.qpkv_decode_run(self.plan_info, _ptr(self.float_ws), self.float_ws.numel(),
                                   _ptr(self.int_ws), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                   _ptr(k_scale_pool), _ptr(v_scale_pool), k_pool.shape[0],
                                   self.page_size, _ptr(block_table), block_table.shape[1],
                                   float(sm_scale), _ptr(out), _ptr(lse), _ptr(error_word),
                                   _stream()), "qpkv_decode_run")
        self._after_run()
        return out

    def attend(self, q, k_pool, v_pool, k_scale_pool, v_scale_pool, block_table, sm_scale,
               error_word=None):
        lib = load()
        self._check_run(q, k_pool, v_pool, k_scale_pool, v_scale_pool, block_table)
        self.wait_ready()
        _check(lib.qpkv_decode_attend(self.plan_info, _ptr(self.float_ws), self.float_ws.numel(),
                                      _ptr(self.int_ws), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                      _ptr(k_scale_pool), _ptr(v_scale_pool), k_pool.shape[0],
                                      self.page_size, _ptr(block_table), block_table.shape[1],
                                      float(sm_scale), _ptr(error_word), _stream()),
               "qpkv_decode_attend")
        self._after_run()

    def merge(self, out, lse=None):
        lib = load()
        self.wait_ready()
        _check(lib.qpkv_decode_merge(self.plan_info, _ptr(self.float_ws), self.float_ws.numel(),
                                     _ptr(self.int_ws), _ptr(out), _ptr(lse), _stream()),
               "qpkv_decode_merge")
        self._after_run()
        return out


def fp8_attn_fwd(q, k, v, q_descale, k_descale, v_descale, softmax_scale=None, causal=False,
                 out=None, lse=None, error_word=None):
    """Dense FP8 attention (BSND E4M3 codes as uint8 tensors): returns bf16 O
    [B, Sq, Hq, D]; ``lse`` (fp32 [B, Sq, Hq]) is filled when given."""
    torch = _torch()
    lib = load()
    _need(q, "q", torch.uint8, 4)
    _need(k, "k", torch.uint8, 4)
    _need(v, "v", torch.uint8, 4)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Sk, Hkv, D] matching q")
    for t, n, h in ((q_descale, "q_descale", Hq), (k_descale, "k_descale", Hkv),
                    (v_descale, "v_descale", Hkv)):
        _need(t, n, torch.float32, 2)
        if tuple(t.shape) != (B, h):
            raise ValueError(f"{n} must be [{B}, {h}]")
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    _check(lib.qpkv_fp8_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Sq, Sk, Hq, Hkv, D,
                                 _ptr(q_descale), _ptr(k_descale), _ptr(v_descale),
                                 float(softmax_scale) if softmax_scale else 0.0,
                                 1 if causal else 0, _ptr(out), _ptr(lse), _ptr(error_word),
                                 _stream()), "qpkv_fp8_attn_fwd")
    return out


def prefill_workspace(num_seqs, num_tokens, num_heads_q, device="cuda"):
    """A device workspace large enough for ``prefill_paged`` on num_seqs
    sequences of num_tokens query rows and num_heads_q heads."""
    torch = _torch()
    n = int(load().qpkv_prefill_workspace_bytes(int(num_seqs), int(num_tokens), int(num_heads_q)))
    return torch.empty(((n + 15) // 16) * 16, dtype=torch.uint8, device=device)


def prefill_paged(q8, q_block_scale, k_pool, k_block_scale, v_pool, block_table, cu_seqlens_q,
                  seqlens_kv, sm_scale=None, causal=True, out=None, lse=None, workspace=None,
                  error_word=None, cu_seqlens_kv=None, v_scale=None):
    """Varlen prefill with INT8 Q/K (block-128 scales) and bf16 V: q8 int8
    [T, Hq, 128]; a paged cache k_pool int8 / v_pool bf16 [P, ps, Hkv, 128]
    with block_table and seqlens_kv, or (cu_seqlens_kv given) ragged K/V
    [T_kv, Hkv, 128] with inclusive prefix sums of the kv lengths; scales
    fp32 [B, NB, H]; returns bf16 O [T, Hq, 128] (``lse`` fp32 [T, Hq]
    filled when given).  With v_scale (fp32 [B, Hkv, 128]) v_pool holds
    E4M3 codes (uint8) and P.V runs in FP8."""
    torch = _torch()
    lib = load()
    ragged = cu_seqlens_kv is not None
    _need(q8, "q8", torch.int8, 3)
    _need(k_pool, "k_pool", torch.int8, 3 if ragged else 4)
    _need(v_pool, "v_pool", torch.uint8 if v_scale is not None else torch.bfloat16,
          3 if ragged else 4)
    _need(q_block_scale, "q_block_scale", torch.float32, 3)
    _need(k_block_scale, "k_block_scale", torch.float32, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    T, Hq, D = q8.shape
    B = cu_seqlens_q.shape[0]
    if tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("v_pool must match k_pool's shape")
    prm = PrefillParams()
    if ragged:
        _need(cu_seqlens_kv, "cu_seqlens_kv", torch.int32, 1)
        if cu_seqlens_kv.shape[0] != B:
            raise ValueError("cu_seqlens_kv must have one entry per sequence")
        T_kv, Hkv, _ = k_pool.shape
        prm.num_kv_tokens = T_kv
        prm.cu_seqlens_kv = _ptr(cu_seqlens_kv)
        prm.page_size, prm.num_pages, prm.bt_stride = 128, 1, 1
    else:
        _need(block_table, "block_table", torch.int32, 2)
        _need(seqlens_kv, "seqlens_kv", torch.int32, 1)
        P, ps, Hkv, _ = k_pool.shape
        if seqlens_kv.shape[0] != B or block_table.shape[0] != B:
            raise ValueError("seqlens_kv / block_table must have one row per sequence")
        prm.page_size, prm.num_pages, prm.bt_stride = ps, P, block_table.shape[1]
        prm.seqlens_kv, prm.block_table = _ptr(seqlens_kv), _ptr(block_table)
    NB = q_block_scale.shape[1]
    if tuple(q_block_scale.shape) != (B, NB, Hq) or tuple(k_block_scale.shape) != (B, NB, Hkv):
        raise ValueError("block scales must be [B, NB, Hq] and [B, NB, Hkv]")
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q8.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        workspace = prefill_workspace(B, T, Hq, q8.device)
    prm.num_seqs, prm.num_tokens, prm.num_heads_q, prm.num_heads_kv = B, T, Hq, Hkv
    prm.head_dim = D
    prm.num_blocks = NB
    prm.causal = 1 if causal else 0
    prm.sm_scale = float(sm_scale) if sm_scale else 0.0
    prm.cu_seqlens_q = _ptr(cu_seqlens_q)
    prm.q, prm.q_block_scale = _ptr(q8), _ptr(q_block_scale)
    prm.k_pool, prm.k_block_scale, prm.v_pool = _ptr(k_pool), _ptr(k_block_scale), _ptr(v_pool)
    prm.o, prm.lse = _ptr(out), _ptr(lse)
    prm.workspace, prm.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    prm.error_word = _ptr(error_word)
    if v_scale is not None:
        _need(v_scale, "v_scale", torch.float32, 3)
        if tuple(v_scale.shape) != (B, Hkv, D):
            raise ValueError("v_scale must be [B, Hkv, 128]")
        prm.v_scale = _ptr(v_scale)
    _check(lib.qpkv_prefill_paged(ctypes.byref(prm), _stream()), "qpkv_prefill_paged")
    return out


def csr_to_block_table(indptr, indices, last_page_len, page_size, bt_stride=None):
    """flashinfer's CSR page description (numpy int32 arrays) -> (block_table
    int32 [B, bt_stride], seqlens int32 [B]), computed by the library."""
    import numpy as np
    lib = load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    last = np.ascontiguousarray(last_page_len, dtype=np.int32)
    B = len(indptr) - 1
    if bt_stride is None:
        bt_stride = max(1, int(np.max(np.diff(indptr))) if B > 0 else 1)
    bt = np.empty((B, bt_stride), dtype=np.int32)
    lens = np.empty(B, dtype=np.int32)
    st = lib.qpkv_csr_to_block_table(indptr.ctypes.data, indices.ctypes.data if indices.size else None,
                                     last.ctypes.data, B, int(page_size), int(bt_stride),
                                     bt.ctypes.data, lens.ctypes.data)
    _check(st, "qpkv_csr_to_block_table")
    return bt, lens


def mla_workspace(num_tokens, sparse_size, device="cuda", sparse_block_size=1):
    """A device workspace large enough for ``mla_sparse_decode``."""
    torch = _torch()
    n = int(load().qpkv_mla_workspace_bytes(int(num_tokens),
                                            int(sparse_size) * max(1, int(sparse_block_size))))
    return torch.empty(((n + 15) // 16) * 16, dtype=torch.uint8, device=device)


def mla_sparse_decode(q, kv_pool, sparse_indices, block_table, seqlens_kv, cu_seqlens_q,
                      scale=None, sparse_mode=0, out=None, lse=None, workspace=None,
                      error_word=None, sparse_block_size=1):
    """MLA-absorb sparse decode: q bf16 [T, Hq, 576]; kv_pool u8 [P, bs, 1, 656];
    sparse_indices int32 [T, 1, S] (token ids, or with sparse_block_size n > 1
    ids of n-token blocks); returns bf16 O [T, Hq, 512] (``lse`` fp32 [T, Hq]
    filled when given)."""
    torch = _torch()
    lib = load()
    _need(q, "q", torch.bfloat16, 3)
    _need(kv_pool, "kv_pool", torch.uint8, 4)
    _need(sparse_indices, "sparse_indices", torch.int32, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens_kv, "seqlens_kv", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    T, Hq, Dqk = q.shape
    P, bs, one, W = kv_pool.shape
    if one != 1 or W != PAGE_ROW_MLA or Dqk != 576:
        raise ValueError("kv_pool must be [P, bs, 1, 656] and q [T, Hq, 576]")
    S = sparse_indices.shape[2]
    if sparse_indices.shape[0] != T:
        raise ValueError("sparse_indices must be [T, 1, S]")
    if out is None:
        out = torch.empty((T, Hq, 512), dtype=torch.bfloat16, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        workspace = mla_workspace(T, S, q.device, sparse_block_size)
    prm = MlaParams()
    prm.num_seqs, prm.num_tokens, prm.num_heads_q = cu_seqlens_q.shape[0], T, Hq
    prm.head_dim_qk, prm.head_dim_v, prm.block_size, prm.num_blocks = 576, 512, bs, P
    prm.bt_stride, prm.sparse_size, prm.sparse_mode = block_table.shape[1], S, int(sparse_mode)
    prm.scale = float(scale) if scale else 0.0
    prm.sparse_block_size = int(sparse_block_size)
    prm.cu_seqlens_q, prm.seqlens_kv, prm.block_table = (
        _ptr(cu_seqlens_q), _ptr(seqlens_kv), _ptr(block_table))
    prm.q, prm.kv_pool, prm.sparse_indices = _ptr(q), _ptr(kv_pool), _ptr(sparse_indices)
    prm.o, prm.lse = _ptr(out), _ptr(lse)
    prm.workspace, prm.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    prm.error_word = _ptr(error_word)
    _check(lib.qpkv_mla_sparse_decode(ctypes.byref(prm), _stream()), "qpkv_mla_sparse_decode")
    return out
