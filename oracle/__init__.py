"""CPU oracle for quantized paged-KV varlen attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or link anything here; only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
use it.  The oracle shares no code, tables or constants with the CUDA path.

It is plain numpy: float64 for attention arithmetic, IEEE float32 where the
method fixes fp32 rounding (the quantizers and RoPE, whose bytes must match
the GPU bit for bit).  Every function cites the passage of the source pages
it follows:

* "KvQuantSparseFlashAttention" README (ops-transformer): 计算公式 (the
  formula softmax(Q·Dequant(K)^T/sqrt(d_k))·Dequant(V)), the
  Per-Token-Head-Tile-128 quantisation named under 功能说明, and the
  参数说明 table (PA_BSND layout, block_table, actual_seq_lengths_*,
  sparse_indices, sparse_mode 0/3, scale_value, MLA-absorb row layout).
* "[Feature] Sage Attention Support Varlen & write kv cache BF16/FP16"
  (PaddleNLP PR 10360), Description items 1-2: RoPE fused into the
  KV-cache write, varlen quantisation per sequence.
* "[Refactor] Unify JIT/Customization/AOT mode" (flashinfer PR 748),
  "Batch Decode/Prefill Attention Kernels": plan/run split, maybe_lse.
* "[Triton] FP8 with FA v3 API" (ROCm aiter PR 917), the flash_attn_func
  usage: FP8 q/k/v with per-(batch, head) q/k/v descales.

Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``):
  e4m3.py      exhaustive comparison with torch's float8_e4m3fn cast,
               format anchors (448, 2^-9, 1.0, NaN codes), ties-to-even.
  quant.py     round-trip bounds, idempotence, absmax -> +-127 / +-448,
               zero blocks, closed-form scale values.
  rope.py      position 0 is the identity, pair norms kept, q_m.k_n depends
               only on m-n, table against closed-form angles.
  cache.py     slot mapping against a brute-force page walk; permuted pages.
  attention.py brute force vs torch SDPA (fp64), single visible key, equal
               keys -> mean of V, permuted page table, sparse covering,
               shift invariance, split + LSE merge, GQA == repeated MHA.
  mla.py       row pack/unpack round trip, reduction to dense attention
               with unit scales and zero rope part.
No function is "parity unpinned".
"""
