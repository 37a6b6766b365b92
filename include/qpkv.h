/*
 * qpkv: quantized paged-KV varlen attention for NVIDIA GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels.  Every pointer argument named
 * "device" is a raw device pointer the caller allocated and owns; "host"
 * pointers are ordinary host memory.  The library never allocates, frees or
 * synchronises: each call enqueues work on the caller's CUDA stream (passed
 * as `void*`, i.e. a cudaStream_t; NULL is the legacy default stream) and
 * returns.  No C++ exception crosses this boundary; every call returns a
 * qpkv_status.  Argument checks that need no device memory run on the host
 * before anything is launched; contents of device arrays (page ids, sparse
 * indices) are checked by the kernels, which skip a bad entry and set a bit
 * in a device error word: the caller's `error_word` (int32), or, when the
 * caller passes NULL, a word the library keeps per GPU, which
 * qpkv_error_check reads and clears (see "device error word" below).
 *
 * Strides are in elements.  All layouts are row-major and contiguous unless
 * a stride argument says otherwise.  Names follow the source pages:
 *  - "KvQuantSparseFlashAttention" README (ops-transformer): the formula
 *    softmax(Q . Dequant(K)^T / sqrt(d_k)) . Dequant(V) (计算公式), the
 *    PA_BSND page layout [block_num, block_size, KV_N, KV_D], block_table,
 *    actual_seq_lengths_query / _kv, sparse_indices, sparse_mode 0 / 3,
 *    scale_value, the MLA-absorb combined row (参数说明 table);
 *  - "[Refactor] Unify JIT/Customization/AOT mode" (flashinfer): the decode
 *    plan / run split with float / int / page-locked workspaces, maybe_lse,
 *    the cuda_stream argument ("Batch Decode/Prefill Attention Kernels");
 *  - "[Feature] Sage Attention Support Varlen & write kv cache BF16/FP16"
 *    (PaddleNLP): RoPE fused into the cache write, varlen grids that exit
 *    past each sequence's end, varlen INT8 quantisation of Q/K (Description);
 *  - "[Triton] FP8 with FA v3 API" (ROCm aiter): FP8 q/k/v with
 *    q_descale / k_descale / v_descale, softmax_scale, causal.
 */
#ifndef QPKV_H_
#define QPKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
typedef int32_t qpkv_status;
#define QPKV_OK 0
#define QPKV_ERR_INVALID_ARG 1         /* null pointer, bad size, misaligned pointer */
#define QPKV_ERR_UNSUPPORTED 2         /* head_dim, page_size, head ratio, dtype, mode */
#define QPKV_ERR_WORKSPACE_TOO_SMALL 3 /* a caller workspace is smaller than required */
#define QPKV_ERR_CUDA 4                /* a CUDA runtime/driver call or launch failed */
#define QPKV_ERR_DEVICE 5              /* a kernel set a bit of the device error word */
#define QPKV_ERR_TIMEOUT 6             /* a kernel's pipeline wait ran out (QPKV_DEV_ERR_TIMEOUT) */
#define QPKV_ERR_STATIC_LIMIT 7        /* problem too large for qpkv_decode_static's fixed scratch */

/* bits a kernel ORs into the device error word */
#define QPKV_DEV_ERR_TIMEOUT 1   /* an internal pipeline wait gave up after ~2 s */
#define QPKV_DEV_ERR_BAD_PAGE 2  /* a block_table entry outside [0, num_pages) was skipped */
#define QPKV_DEV_ERR_BAD_INDEX 4 /* a sparse index outside [0, L_kv) was skipped */
#define QPKV_DEV_ERR_BAD_LENGTH 8 /* a sequence length does not fit the arrays described; skipped */

/* Text of a status code (static storage, never NULL). */
const char* qpkv_status_string(qpkv_status status);

/* ------------------------------------------------------ device error word
 * Kernels report what they cannot return (a skipped bad page id or sparse
 * index, a pipeline wait that ran out) by OR-ing QPKV_DEV_ERR_* bits into a
 * device int32.  Every entry point that takes an `error_word` uses the
 * caller's word when one is given and otherwise a word owned by the library
 * (one per GPU, a file-scope __device__ variable; the first call on a
 * device looks up its address with that device current).  The outputs of a
 * call that set QPKV_DEV_ERR_TIMEOUT are undefined.
 *
 * qpkv_error_status maps a word's bits to a status: QPKV_ERR_TIMEOUT when
 * the timeout bit is set, else QPKV_ERR_DEVICE for any other bit, else
 * QPKV_OK.
 *
 * qpkv_error_check takes the library's word of the current device (an
 * atomic exchange with 0, in a one-thread kernel on `stream`), copies it to
 * the host and synchronises `stream` (the only call of this library that
 * waits); *bits_out (may be NULL) receives the bits and the return value is
 * qpkv_error_status(bits), or QPKV_ERR_CUDA when a CUDA call fails.  Bits
 * set by work on other streams that has not finished are reported by a
 * later check. */
qpkv_status qpkv_error_status(int32_t bits);
qpkv_status qpkv_error_check(void* stream, int32_t* bits_out);

/* Self-test of the bounded wait that every pipeline wait of the library's
 * kernels uses: a one-CTA kernel waits on an mbarrier whose arrival never
 * comes, gives up after limit_cycles SM cycles (1000 .. 4e9; the kernels use
 * 4e9, about 2 s) and sets QPKV_DEV_ERR_TIMEOUT in error_word (the
 * library's word when NULL).  The kernel then returns normally and the
 * context stays usable.  INVALID_ARG for a limit outside the range. */
qpkv_status qpkv_selftest_wait_timeout(int64_t limit_cycles, int32_t* error_word, void* stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t qpkv_version(void);

/* sizeof of the parameter structs below, so that bindings in other
 * languages can check their mirror of the layout:
 * which = 0 -> qpkv_write_params, 1 -> qpkv_prefill_params,
 * 2 -> qpkv_mla_params.  Unknown `which` returns 0. */
size_t qpkv_struct_size(int32_t which);

/* -------------------------------------------------------------- RoPE table
 * cos/sin tables for the rotate-half RoPE of the cache write ("[Feature]
 * Sage Attention ... write kv cache BF16/FP16", Description item 1; the
 * rope_theta / rope_scale parameters of flashinfer's interfaces):
 *   inv_freq_i = theta^(-2i/rot_dim), angle = (pos / rope_scale) * inv_freq_i,
 * evaluated in double precision on the device and rounded to float.
 * cos_out, sin_out: device float [max_pos, rot_dim/2] (caller-allocated).
 * Errors: INVALID_ARG for null outputs, max_pos < 1, odd or non-positive
 * rot_dim, theta <= 0 or rope_scale <= 0; CUDA on launch failure. */
qpkv_status qpkv_rope_table(float theta, float rope_scale, int32_t max_pos, int32_t rot_dim,
                            float* cos_out, float* sin_out, void* stream);

/* -------------------------------------------------------------- cache write
 * RoPE + quantise + page-append of new tokens ("[Feature] Sage Attention
 * ... write kv cache BF16/FP16", Description items 1-2; README 参数说明 rows
 * key / block_table / actual_seq_lengths_query).  New token t of sequence b
 * has position p = start_pos[b] + (t - begin_b) and goes to pool row
 * ("slot") block_table[b * bt_stride + p / page_size] * page_size + p % page_size.
 *
 * Modes:
 *  QPKV_WRITE_FP8_TOKEN_HEAD  k, v bf16 [T, Hkv, D] -> E4M3 pools
 *     [P, page_size, Hkv, D] + float scale pools [P, page_size, Hkv];
 *     scale = absmax_D / 448, code = RNE_satfinite(x / scale) (IEEE fp32
 *     division), absmax 0 -> scale 0 and zero codes.  D in {64, 128}.
 *     With rope_cos / rope_sin (float [rope_max_pos, D/2], qpkv_rope_table
 *     with rot_dim D) k is rotated first (rotate-half, pairs (i, i + D/2),
 *     each product and sum rounded to float32) at the token's position and
 *     the float32 result quantised; v never is.  With q as well (bf16
 *     [T, Hq, D], Hq = num_heads_q) the rotated queries are rounded to bf16
 *     (nearest-even) into q_out (bf16, same shape; may alias q).  A position
 *     outside the tables leaves the token unwritten and sets
 *     QPKV_DEV_ERR_BAD_LENGTH.
 *  QPKV_WRITE_INT8_BLOCK128_ROPE  q, k, v bf16 [T, H, D]: RoPE (rotate-half,
 *     pairs (i, i + D/2), tables from qpkv_rope_table) on q and k, then one
 *     scale per (sequence, 128-token block, head): scale = absmax / 127,
 *     code = clamp(RNE(x / scale), -127, 127).  K codes go to the int8
 *     k_pool, V is copied unchanged into the bf16 v_pool, Q codes go to
 *     q_out (int8 [T, Hq, D], TND), scales to k_block_scale [B, num_blocks,
 *     Hkv] and q_block_scale [B, num_blocks, Hq].  Whole sequences only
 *     (start_pos must be NULL: every sequence starts at position 0).  D = 128.
 *     With flags & QPKV_WRITE_SMOOTH_K (K smoothing, the role of the Sage
 *     varlen page's segment_mean kernel) the keys quantised are k_rot - m,
 *     m[b, h] = float32(float64(S) / (n_b * 2^24)) with S the exact int64 sum
 *     over the sequence's n_b tokens of RNE(clamp(k_rot, -2^15, 2^15) * 2^24);
 *     m goes to k_mean (float [B, Hkv, 128]) and workspace holds int64
 *     partial sums [B, num_blocks, Hkv, 128] (qpkv_smooth_workspace_bytes).
 *     Attention over the smoothed cache is unchanged (every logit of a query
 *     row moves by scale * q . m); its lse moves by the same amount.
 *     With flags & QPKV_WRITE_V_FP8 (Sage-style FP8 V, for an FP8 P.V
 *     product) v_pool holds E4M3 codes (u8 [P, page_size, Hkv, 128]) of
 *     v / s, s[b, h, c] = absmax over sequence b of channel c of head h / 448
 *     (float32 division; s = 0 gives zero codes), and s goes to
 *     v_channel_scale (float [B, Hkv, 128]).  Both options use workspace.
 *  QPKV_WRITE_MLA_ROW  k = kv bf16 [T, 576] (512 nope || 64 rope), Hkv = 1:
 *     each token becomes one 656-byte row of the pool [P, page_size, 1, 656]:
 *     bytes [0, 512) INT8 nope codes (tile i = dims 128i..128i+127 has scale
 *     absmax/127), [512, 640) the bf16 rope values, [640, 656) the 4 fp32
 *     tile scales, little-endian ("512+64*2+4*4", README row key).
 *     With rope_cos / rope_sin (float [rope_max_pos, 32], from
 *     qpkv_rope_table with rot_dim 64) the rope part is first rotated
 *     (rotate-half, pairs (i, i + 32)) at the token's position and the
 *     float32 result rounded to bf16 (nearest-even); a position outside the
 *     tables leaves the row unwritten and sets QPKV_DEV_ERR_BAD_LENGTH.
 *     With q (bf16 [T, Hq, 576], Hq = num_heads_q) the query rows are written
 *     to q_out (bf16, same shape; may alias q) with their rope part rotated
 *     the same way and the nope part copied; q requires the tables.
 *
 * Device arrays: cu_seqlens_q int32 [B] inclusive prefix sums (batch b spans
 * [cu[b-1], cu[b]), cu[-1] = 0); start_pos int32 [B] or NULL (all zero);
 * block_table int32 [B, bt_stride]; slot_mapping int32 [T] out or NULL.
 * Every pointer must be 16-byte aligned.  Pool rows of tokens not written
 * are left untouched.
 * Errors: INVALID_ARG (null required pointer, non-positive sizes, misaligned
 * pointer, start_pos given in INT8 mode), UNSUPPORTED (mode, D, page_size
 * not a multiple of 16, Hq % Hkv != 0), CUDA.  Page ids outside
 * [0, num_pages) are skipped with QPKV_DEV_ERR_BAD_PAGE. */
#define QPKV_WRITE_FP8_TOKEN_HEAD 0
#define QPKV_WRITE_INT8_BLOCK128_ROPE 1
#define QPKV_WRITE_MLA_ROW 2

/* qpkv_write_params.flags */
#define QPKV_WRITE_SMOOTH_K 1   /* INT8 mode: subtract the per-(sequence, head) key mean */
#define QPKV_WRITE_HND 2        /* FP8 mode: K/V pools [P, Hkv, page_size, D] (scales unchanged) */
#define QPKV_WRITE_V_FP8 4      /* INT8 mode: V as E4M3 with one scale per (sequence, head, channel) */

typedef struct qpkv_write_params {
  int32_t mode;
  int32_t num_seqs;       /* B */
  int32_t num_tokens;     /* T, number of new tokens */
  int32_t max_seqlen;     /* host upper bound of any sequence's new-token count */
  int32_t num_heads_q;    /* Hq (INT8 mode), else ignored */
  int32_t num_heads_kv;   /* Hkv (1 for MLA) */
  int32_t head_dim;       /* D (576 for MLA: input width) */
  int32_t page_size;
  int32_t num_pages;      /* P, pool size, for page-id checks */
  int32_t bt_stride;      /* row stride of block_table */
  int32_t num_blocks;     /* INT8 mode: dim 1 of the block-scale arrays */
  int32_t rope_max_pos;   /* rows of the RoPE tables (INT8 and MLA modes) */
  const int32_t* cu_seqlens_q;
  const int32_t* start_pos;
  const int32_t* block_table;
  const void* q;          /* bf16 [T, Hq, D] (INT8 mode; MLA: [T, Hq, 576] or NULL) */
  const void* k;          /* bf16 [T, Hkv, D] ([T, 576] for MLA) */
  const void* v;          /* bf16 [T, Hkv, D] (not used for MLA) */
  const float* rope_cos;  /* [rope_max_pos, D/2] (INT8 mode; MLA: [rope_max_pos, 32] or NULL) */
  const float* rope_sin;
  void* k_pool;           /* u8 E4M3 / int8 / MLA rows */
  void* v_pool;           /* u8 E4M3 (FP8 mode) / bf16 (INT8 mode) */
  float* k_scale_pool;    /* FP8 mode [P, page_size, Hkv] */
  float* v_scale_pool;
  float* k_block_scale;   /* INT8 mode [B, num_blocks, Hkv] */
  void* q_out;            /* INT8 mode: int8 [T, Hq, D]; MLA: bf16 [T, Hq, 576] */
  float* q_block_scale;   /* INT8 mode [B, num_blocks, Hq] */
  int32_t* slot_mapping;  /* [T] or NULL */
  int32_t* error_word;    /* device int32, or NULL for the library's word */
  int32_t flags;          /* QPKV_WRITE_SMOOTH_K (INT8 mode) or 0 */
  int32_t pad0;
  float* k_mean;          /* INT8 + SMOOTH_K: out float [B, Hkv, 128] */
  void* workspace;        /* INT8 + SMOOTH_K or V_FP8: scratch, 16-byte aligned */
  size_t workspace_bytes;
  float* v_channel_scale; /* INT8 + V_FP8: out float [B, Hkv, 128] */
} qpkv_write_params;

/* Scratch bytes of an INT8 write with QPKV_WRITE_SMOOTH_K and / or
 * QPKV_WRITE_V_FP8 (0 for negative sizes). */
size_t qpkv_smooth_workspace_bytes(int32_t num_seqs, int32_t num_blocks, int32_t num_heads_kv);

qpkv_status qpkv_write_cache(const qpkv_write_params* params, void* stream);

/* ----------------------------------------------------------- decode: plan
 * Paged FP8 decode, one query token per request (flashinfer "Batch Decode
 * Attention Kernels": BatchDecodeWithPagedKVCachePlan / ...Run; aiter's
 * flash_attn_with_kvcache with page_table and cache_seqlens).
 *
 * qpkv_decode_plan splits every (request, kv head) into work items of at
 * most `chunk` (128 or 256) tokens so that the items fill the GPU, writes
 * the work list into the caller's page-locked host buffer and copies it
 * (one cudaMemcpyAsync on `stream`) into the caller's device int workspace.
 * seqlens_kv_host: host int32 [B], tokens in each request's cache (>= 0).
 * num_sms: SM count of the device (used to pick the chunk).
 * plan_info: host int64 [QPKV_PLAN_INFO_LEN] out, passed to qpkv_decode_run.
 * Required sizes come from qpkv_decode_workspace_sizes.  The pinned buffer
 * must stay untouched until the copy has run (stream order).
 * Errors: INVALID_ARG (null pointers, B < 1, negative length, Hq % Hkv),
 * UNSUPPORTED (head_dim not in {64, 128}, Hq/Hkv not in {1, 2, 4, 8},
 * page_size not a multiple of 16 dividing 256 or a multiple of 256),
 * WORKSPACE_TOO_SMALL, CUDA. */
#define QPKV_PLAN_INFO_LEN 24

/* K/V pool layouts of the FP8 decode path (flashinfer's kv_layout_code in
 * "[Refactor] Unify JIT/Customization/AOT mode", BatchDecodeWithPagedKVCacheRun):
 * NHD = [P, page_size, Hkv, D] (the default), HND = [P, Hkv, page_size, D].
 * The per-(token, head) scale pools stay [P, page_size, Hkv] in both. */
#define QPKV_KV_LAYOUT_NHD 0
#define QPKV_KV_LAYOUT_HND 1

/* Switch a plan (from qpkv_decode_plan / qpkv_decode_plan_host) to the K/V
 * pool layout of the pools later passed to qpkv_decode_run / _attend; a new
 * plan starts as NHD.  Errors: INVALID_ARG (not a plan, unknown layout). */
qpkv_status qpkv_decode_plan_set_kv_layout(int64_t* plan_info, int32_t kv_layout);

qpkv_status qpkv_decode_workspace_sizes(const int32_t* seqlens_kv_host, int32_t batch_size,
                                        int32_t num_qo_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t num_sms, size_t* int_ws_bytes,
                                        size_t* float_ws_bytes);

/* Host-only part of the plan (no CUDA call): fills host_int_ws and plan_info.
 * qpkv_decode_plan = this + the async copy to the device int workspace. */
qpkv_status qpkv_decode_plan_host(const int32_t* seqlens_kv_host, int32_t batch_size,
                                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t page_size,
                                  int32_t head_dim, int32_t num_sms, void* host_int_ws,
                                  size_t host_int_bytes, int64_t* plan_info);

qpkv_status qpkv_decode_plan(const int32_t* seqlens_kv_host, int32_t batch_size,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t page_size,
                             int32_t head_dim, int32_t num_sms, void* pinned_int_ws,
                             size_t pinned_bytes, void* int_ws, size_t int_ws_bytes,
                             int64_t* plan_info, void* stream);

/* ------------------------------------------------------------ decode: run
 * O[b, h, :] = softmax(sm_scale * q[b, h] . Dequant(K_b)^T) . Dequant(V_b)
 * over the L_b cached tokens of request b, kv head h / (Hq / Hkv), with
 * Dequant(x)[t] = e4m3(x[t]) * scale_pool[t] (README 计算公式; per-token-head
 * FP8).  q: device bf16 [B, Hq, D]; k_pool / v_pool: device u8
 * [num_pages, page_size, Hkv, D]; k_scale_pool / v_scale_pool: device float
 * [num_pages, page_size, Hkv]; block_table: device int32 [B, bt_stride];
 * o: device bf16 [B, Hq, D]; lse: device float [B, Hq] (natural log of the
 * softmax denominator of the scaled logits) or NULL.
 * float_ws / int_ws: the workspaces given to qpkv_decode_plan (device).  The
 * run also writes the int workspace: when the plan takes all kv heads per
 * work item it holds two work counters that the attend kernel advances and
 * re-arms before it finishes (so the same plan can be run repeatedly, in
 * stream order).
 * A request with L_b = 0 gets O = 0 and lse = -inf.
 * qpkv_decode_run = qpkv_decode_attend (split-KV partials) followed by
 * qpkv_decode_merge (log-sum-exp merge), both on `stream`.
 * block_table rows must hold at least ceil(max_b L_b / page_size) entries.
 * Errors: INVALID_ARG (null / misaligned pointers, plan_info not from
 * qpkv_decode_plan, bt_stride too small for the longest request),
 * WORKSPACE_TOO_SMALL, CUDA. */
qpkv_status qpkv_decode_run(const int64_t* plan_info, void* float_ws, size_t float_ws_bytes,
                            void* int_ws, const void* q, const void* k_pool,
                            const void* v_pool, const float* k_scale_pool,
                            const float* v_scale_pool, int32_t num_pages, int32_t page_size,
                            const int32_t* block_table, int32_t bt_stride, float sm_scale,
                            void* o, float* lse, int32_t* error_word, void* stream);

/* Split-KV step alone: writes per-split partial O (float) and lse into
 * float_ws.  Same arguments as qpkv_decode_run without o / lse. */
qpkv_status qpkv_decode_attend(const int64_t* plan_info, void* float_ws, size_t float_ws_bytes,
                               void* int_ws, const void* q, const void* k_pool,
                               const void* v_pool, const float* k_scale_pool,
                               const float* v_scale_pool, int32_t num_pages, int32_t page_size,
                               const int32_t* block_table, int32_t bt_stride, float sm_scale,
                               int32_t* error_word, void* stream);

/* Merge step alone: O = sum_s exp(lse_s - M) O_s / sum_s exp(lse_s - M),
 * lse = M + ln sum_s exp(lse_s - M), M = max_s lse_s, per (request, head). */
qpkv_status qpkv_decode_merge(const int64_t* plan_info, const void* float_ws,
                              size_t float_ws_bytes, const void* int_ws, void* o, float* lse,
                              void* stream);

/* ------------------------------------------ decode without any allocation
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: code running where cudaMalloc is not
 * allowed or not wanted (an embedding runtime that owns all device memory,
 * a plugin with no allocator handle, a hard real-time loop that must not
 * hit the allocator).  It runs the same paged FP8 decode as
 * qpkv_decode_plan + qpkv_decode_run, with the same arguments minus the
 * workspaces: the work list and the split-KV partials live in fixed arrays
 * compiled into the library (QPKV_STATIC_INT_BYTES + QPKV_STATIC_FLOAT_BYTES
 * of device memory per GPU, held from the first call until the process
 * exits), and the plan is staged through a fixed host buffer.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on each device looks up the arrays' device addresses
 * (cudaGetSymbolAddress) with that device current.  The work list goes
 * through one shared host buffer by a pageable copy, so a call made while
 * its stream is capturing returns QPKV_ERR_UNSUPPORTED and enqueues
 * nothing.  Every call reuses the same arrays: calls
 * whose work overlaps on the GPU (different streams, or different host
 * threads without ordering) race and corrupt each other's results; nothing
 * in the arrays needs to start at zero (each call rewrites what it reads).
 * Errors: as qpkv_decode_plan / qpkv_decode_run, plus QPKV_ERR_STATIC_LIMIT
 * when the batch needs more work-list or partial-result space than the
 * fixed arrays hold (checked on the host before any CUDA call). */
#define QPKV_STATIC_INT_BYTES (2u << 20)    /* 2 MiB work list */
#define QPKV_STATIC_FLOAT_BYTES (32u << 20) /* 32 MiB split-KV partials */

qpkv_status qpkv_decode_static(const int32_t* seqlens_kv_host, int32_t batch_size,
                               int32_t num_qo_heads, int32_t num_kv_heads, int32_t page_size,
                               int32_t head_dim, int32_t num_sms, const void* q,
                               const void* k_pool, const void* v_pool, const float* k_scale_pool,
                               const float* v_scale_pool, int32_t num_pages,
                               const int32_t* block_table, int32_t bt_stride, float sm_scale,
                               void* o, float* lse, int32_t* error_word, void* stream);

/* ------------------------------------------ dense FP8 attention forward
 * "[Triton] FP8 with FA v3 API" (flash_attn_func with q/k/v in FP8 and
 * their descale values):
 *   O = softmax(softmax_scale * qd[b,h] * kd[b,hk] * Q8 . K8^T + mask)
 *       . V8 * vd[b,hk]
 * Q8/K8/V8 are E4M3 codes; a code times its descale is the value.
 *   q          device, E4M3 [B, Sq, Hq, D] (BSND, contiguous)
 *   k, v       device, E4M3 [B, Sk, Hkv, D]
 *   q_descale  device fp32 [B, Hq]; k_descale, v_descale fp32 [B, Hkv]
 *   softmax_scale  <= 0 selects 1/sqrt(D)
 *   causal     0: every key visible; 1: bottom-right aligned, key j visible
 *              to query i iff j <= i + Sk - Sq
 *   o          device bf16 [B, Sq, Hq, D]; rows that see no key are 0
 *   lse        device fp32 [B, Sq, Hq] or NULL: natural log of the sum of
 *              exp(scaled logits); -inf for rows that see no key
 *   error_word device int32 (NULL: the library's word): QPKV_DEV_ERR_* bits set by the kernel
 * kv head of q head h: h / (Hq / Hkv).  Supported: D = 128, Hq % Hkv == 0;
 * every pointer 16-byte aligned.  P enters the PV product as two E4M3
 * terms (hi + lo, about 8 significant bits).  The caller owns all
 * memory; nothing is allocated.  Errors: QPKV_ERR_INVALID_ARG (null or
 * misaligned pointers, negative sizes), QPKV_ERR_UNSUPPORTED (D, head
 * grouping), QPKV_ERR_CUDA (launch). */
qpkv_status qpkv_fp8_attn_fwd(const void* q, const void* k, const void* v, int32_t batch,
                              int32_t seqlen_q, int32_t seqlen_k, int32_t num_qo_heads,
                              int32_t num_kv_heads, int32_t head_dim, const float* q_descale,
                              const float* k_descale, const float* v_descale,
                              float softmax_scale, int32_t causal, void* o, float* lse,
                              int32_t* error_word, void* stream);

/* ------------------------------------------------- varlen prefill (INT8 QK)
 * Causal varlen prefill over a paged cache in the layout QPKV_WRITE_INT8_
 * BLOCK128_ROPE writes ("[Feature] Sage Attention Support Varlen & write kv
 * cache BF16/FP16", Description items 1-3; "KvQuantSparseFlashAttention"
 * README 计算公式, 参数说明 rows actual_seq_lengths_query /
 * actual_seq_lengths_kv / block_table / sparse_mode):
 *   logit(i, j) = sm_scale * sq[b, i/128, h] * sk[b, j/128, hk] * (q8_i . k8_j)
 *   o_i = sum_j softmax_j(logit(i, .)) * v_j       (v bf16, no scale)
 *   lse_i = ln sum_j exp(logit(i, j))
 * Query i of sequence b (0-based, L_q = its row count) sees key j iff
 * j < L_kv[b] and, when causal, j <= i + L_kv[b] - L_q (bottom-right).  The
 * kv head of q head h is h / (Hq / Hkv).  Rows that see no key get o = 0
 * and lse = -inf.
 *
 * Arrays (device; the caller owns all memory):
 *   cu_seqlens_q  int32 [B] inclusive prefix sums; sequence b owns q/o rows
 *                 [cu[b-1], cu[b]) (cu[-1] = 0), cu[B-1] <= num_tokens
 *   seqlens_kv    int32 [B] tokens in the cache per sequence (L_kv)
 *   block_table   int32 [B, bt_stride]: key j lives at pool row
 *                 block_table[b][j / page_size] * page_size + j % page_size;
 *                 entries past L_kv are never read
 *   q             int8 [T, Hq, 128] codes (TND), q_block_scale fp32 [B,
 *                 num_blocks, Hq] (query block of row i is i / 128)
 *   k_pool        int8 [P, page_size, Hkv, 128], k_block_scale fp32
 *                 [B, num_blocks, Hkv] (key block of key j is j / 128)
 *   v_pool        bf16 [P, page_size, Hkv, 128]; or, with v_scale set
 *                 (Sage-style FP8 V, written with QPKV_WRITE_V_FP8), E4M3
 *                 codes u8 of the same shape and v_scale fp32 [B, Hkv, 128]:
 *                 v_j = code * v_scale[b, hk, channel], P enters P.V as two
 *                 E4M3 terms (relative L2 error of o within 2e-2)
 *   o             bf16 [T, Hq, 128]; lse fp32 [T, Hq] or NULL
 *   workspace     qpkv_prefill_workspace_bytes(B, T, Hq) bytes of device
 *                 memory, overwritten by every call (the call's work order)
 *   error_word    int32 (NULL: the library's word): QPKV_DEV_ERR_BAD_PAGE (a block_table entry
 *                 outside [0, P) read as zeros), QPKV_DEV_ERR_BAD_LENGTH (a
 *                 sequence whose lengths exceed num_blocks * 128, the
 *                 block_table row or num_tokens: its rows are zeroed),
 *                 QPKV_DEV_ERR_TIMEOUT.
 * Ragged K/V (flashinfer's BatchPrefillWithRaggedKVCache layout, "[Refactor]
 * Unify JIT/Customization/AOT mode", Batch Prefill): with cu_seqlens_kv set,
 * k_pool is int8 [num_kv_tokens, Hkv, 128] and v_pool bf16 [num_kv_tokens,
 * Hkv, 128], sequence b's keys are rows [cu_kv[b-1], cu_kv[b]) and L_kv[b]
 * = cu_kv[b] - cu_kv[b-1]; block_table, seqlens_kv, page_size and
 * num_pages are not used (block_table and seqlens_kv may be NULL).
 * Supported: head_dim 128, page_size a multiple of 16 that divides 128 or
 * is a multiple of 128 up to 16384, Hq <= 32768, Hq % Hkv == 0.  q, k_pool, v_pool, o 16-byte
 * aligned.  sm_scale <= 0 selects 1/sqrt(128).
 * Errors: INVALID_ARG (null required pointer, negative or zero sizes,
 * misaligned pointer), UNSUPPORTED (head_dim, page_size, head grouping),
 * WORKSPACE_TOO_SMALL, CUDA (launch). */
typedef struct qpkv_prefill_params {
  int32_t num_seqs;      /* B */
  int32_t num_tokens;    /* T: rows of q, o, lse */
  int32_t num_heads_q;   /* Hq */
  int32_t num_heads_kv;  /* Hkv */
  int32_t head_dim;      /* 128 */
  int32_t page_size;
  int32_t num_pages;     /* P */
  int32_t bt_stride;     /* row stride of block_table */
  int32_t num_blocks;    /* dim 1 of q_block_scale / k_block_scale */
  int32_t causal;
  float sm_scale;
  int32_t num_kv_tokens;  /* ragged K/V only: rows of k_pool / v_pool */
  const int32_t* cu_seqlens_q;
  const int32_t* seqlens_kv;
  const int32_t* cu_seqlens_kv;  /* NULL: paged K/V; else ragged, inclusive prefix sums [B] */
  const int32_t* block_table;
  const void* q;
  const float* q_block_scale;
  const void* k_pool;
  const float* k_block_scale;
  const void* v_pool;
  void* o;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  int32_t* error_word;
  const float* v_scale;   /* NULL: v_pool is bf16.  Else v_pool holds E4M3 codes (u8, shaped
                             like k_pool) and v_scale [B, Hkv, 128] the per-(sequence, head,
                             channel) scales of QPKV_WRITE_V_FP8; P.V is then an FP8 product
                             with P as two E4M3 terms (hi + lo, about 8 significant bits) */
} qpkv_prefill_params;

/* Device workspace bytes qpkv_prefill_paged needs for num_seqs sequences of
 * num_tokens query rows in total and num_heads_q query heads (0 for a
 * negative argument). */
size_t qpkv_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens, int32_t num_heads_q);

qpkv_status qpkv_prefill_paged(const qpkv_prefill_params* params, void* stream);

/* ------------------------------------------------------ CSR page description
 * flashinfer's CSR description of a paged cache ("[Refactor] Unify
 * JIT/Customization/AOT mode", Batch Decode/Prefill: paged_kv_indptr,
 * paged_kv_indices, paged_kv_last_page_len) -> this library's block_table
 * rows and per-request lengths, on the host:
 *   block_table[b][i] = indices[indptr[b] + i] for i < n_b = indptr[b+1] - indptr[b]
 *   seqlens[b] = (n_b - 1) * page_size + last_page_len[b]   (0 when n_b = 0)
 * Entries of block_table past n_b are set to -1.  Host arrays: indptr [B+1],
 * indices [indptr[B]], last_page_len [B], block_table_out [B, bt_stride],
 * seqlens_out [B] (caller-allocated).
 * Errors: INVALID_ARG (null pointer, B < 0, page_size < 1, indptr not
 * starting at 0 or decreasing, n_b > bt_stride, last_page_len[b] outside
 * [1, page_size] for n_b > 0, a length above INT32_MAX). */
qpkv_status qpkv_csr_to_block_table(const int32_t* indptr, const int32_t* indices,
                                    const int32_t* last_page_len, int32_t batch,
                                    int32_t page_size, int32_t bt_stride,
                                    int32_t* block_table_out, int32_t* seqlens_out);

/* ------------------------------------------------ MLA-absorb sparse decode
 * ("KvQuantSparseFlashAttention" README, 计算公式; 参数说明 rows query, key,
 * value, sparse_indices, block_table, actual_seq_lengths_query,
 * actual_seq_lengths_kv, sparse_mode, scale_value; attention_mode 2 with
 * the combined cache row, quant_scale_repo_mode 1):
 *   for query token t (sequence b, row i of its L_q rows) and q head h the
 *   keys are the entries of sparse_indices[t, 0, :] before the first -1,
 *   logical token positions of sequence b mapped through block_table
 *   (pool row block_table[b][id / block_size] * block_size + id % block_size);
 *   sparse_mode 3 also drops ids above i + L_kv - L_q.  With
 *   sparse_block_size n > 1 (block-wise sparsity, README row
 *   sparse_block_size) an entry id names the n tokens [id * n, id * n + n)
 *   of the sequence, which share the decision; tokens of the block at or
 *   past L_kv are not keys, and an id with id * n >= L_kv is out of range.
 *   A cache row is 656
 *   bytes: 512 INT8 nope codes, 64 bf16 rope values, 4 fp32 scales (nope
 *   tile k = dims 128k..128k+127), the layout QPKV_WRITE_MLA_ROW writes.
 *   K = [code * scale || rope] (576), V = code * scale (512);
 *   o[t, h] = softmax(scale_value * q[t, h] . K^T) . V (bf16 [T, Hq, 512]),
 *   lse[t, h] = ln sum exp(logits); no visible key: o = 0, lse = -inf.
 * The nope is dequantised to bf16 (code * scale rounded once) for both
 * products; the logits and the softmax are fp32, P enters PV as bf16.
 *
 * Arrays (device): q bf16 [T, Hq, 576]; kv_pool u8 [P, block_size, 1, 656];
 * sparse_indices int32 [T, 1, sparse_size]; block_table int32 [B,
 * bt_stride]; seqlens_kv int32 [B]; cu_seqlens_q int32 [B] inclusive prefix
 * sums; o bf16 [T, Hq, 512]; lse fp32 [T, Hq] or NULL; workspace of
 * qpkv_mla_workspace_bytes(T, sparse_size * sparse_block_size) bytes
 * (overwritten).
 * error_word bits: QPKV_DEV_ERR_BAD_INDEX (an id outside [0, L_kv) before
 * the first -1, skipped), QPKV_DEV_ERR_BAD_PAGE, QPKV_DEV_ERR_TIMEOUT.
 * Supported: 1 <= Hq <= 128, head_dim_qk 576, head_dim_v 512, sparse_mode
 * 0 or 3, 1 <= sparse_block_size <= 128 (0 reads as 1), sparse_size *
 * sparse_block_size <= 2^24.  q, kv_pool, o, workspace 16-byte aligned.
 * scale <= 0 selects 1/sqrt(576).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
typedef struct qpkv_mla_params {
  int32_t num_seqs;      /* B */
  int32_t num_tokens;    /* T: query tokens (rows of q, o, lse) */
  int32_t num_heads_q;   /* Hq, at most 128 */
  int32_t head_dim_qk;   /* 576 */
  int32_t head_dim_v;    /* 512 */
  int32_t block_size;    /* tokens per cache block */
  int32_t num_blocks;    /* P */
  int32_t bt_stride;
  int32_t sparse_size;   /* entries per sparse_indices row */
  int32_t sparse_mode;   /* 0 or 3 */
  float scale;
  int32_t sparse_block_size;   /* tokens per listed id: 1 (token-wise) .. 128; 0 = 1 */
  const int32_t* cu_seqlens_q;
  const int32_t* seqlens_kv;
  const int32_t* block_table;
  const void* q;
  const void* kv_pool;
  const int32_t* sparse_indices;
  void* o;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  int32_t* error_word;
} qpkv_mla_params;

/* Device workspace bytes qpkv_mla_sparse_decode needs (0 for negative sizes). */
size_t qpkv_mla_workspace_bytes(int32_t num_tokens, int32_t sparse_size);

qpkv_status qpkv_mla_sparse_decode(const qpkv_mla_params* params, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QPKV_H_ */
