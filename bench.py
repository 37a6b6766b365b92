"""Benchmark: paged FP8 decode step on the Llama-3-8B-shaped batch.

Workload (one step = one pass of the decode hot path over one batch):
  B = 64 requests, kv lengths ~ U{512..8192}, 32 query / 8 kv heads,
  head_dim 128, page 16, pages randomly permuted in the pool, FP8 E4M3 K/V
  with fp32 per-(token, head) scales.  Each step appends one new token per
  request through the cache-write kernel, re-plans the split-KV work list
  (host planner + one async copy), runs the split-KV attention kernel and the
  log-sum-exp merge.  Inputs are resident in HBM (the cache is ~589 MB per
  step of reads, larger than the 129 MB L2, so no flush is needed).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(test infrastructure) on a bounded sample of the same workload instead.
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
collective on the data path); time = max over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode HBM GB/s & tokens/s; FP8 prefill TFLOP/s (% of GB300 roofline)"
WORKLOAD = ("Llama-3-8B-shaped paged FP8 decode: B=64, q_len=1, kv lengths ~U{512..8192}, "
            "32 qo / 8 kv heads, head_dim 128, page 16, permuted page pool, E4M3 K/V with "
            "fp32 per-(token, head) scales")
B, HQ, HKV, D, PS, LO, HI = 64, 32, 8, 128, 16, 512, 8192
L2_BYTES = 129 * 2 ** 20
ATT_EVERY = 8   # timed steps between two samples of the attend kernel's duration
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_heads_llama8b_b64.txt")
KERNEL_SOURCE = os.path.join(ROOT, "quantized_paged_kv_varlen_gb300", "csrc", "decode_heads.cu")


def algorithmic_bytes(lengths):
    """Bytes the decode step must move at minimum (per request batch)."""
    import numpy as np
    lengths = np.asarray(lengths, dtype=np.int64)
    kv = int(lengths.sum()) * HKV * D * 2                # E4M3 K and V
    scales = int(lengths.sum()) * HKV * 4 * 2            # fp32 k/v scales
    bt = int(((lengths + PS - 1) // PS).sum()) * 4       # block table entries
    q = len(lengths) * HQ * D * 2                        # bf16 query
    o = len(lengths) * HQ * (D * 2 + 4)                  # bf16 output + lse
    new = len(lengths) * HKV * (D * 2 * 2 + (D + 4) * 2)  # new token: bf16 in, fp8+scale out
    attend = kv + scales + bt + q
    return attend + o + new, attend


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) while the GPU is loaded."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if len(r) >= 9]
        inside = [r for t, r in self.rows if t0 <= t <= t1 and len(r) >= 9]
        window = "timed region"
        if not inside:   # region shorter than the sampling interval: nearest samples
            inside = [r for t, r in self.rows if t0 - 0.2 <= t <= t1 + 0.2 and len(r) >= 9]
            window = "timed region +- 200 ms"
        use = inside if inside else rows
        if not inside:
            window = "whole run"
        n_inside = len([1 for t, r in self.rows if t0 <= t <= t1 and len(r) >= 9])
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(use[0][2]), "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": n_inside, "window": window,
                "power_w_max": max((num(r[3]) or 0.0) for r in use)}


# ------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- workload

class DecodeBench:
    """Device-resident decode workload for one rank (seed = base + rank)."""

    def __init__(self, seed, device):
        import numpy as np
        import torch
        import quantized_paged_kv_varlen_gb300 as q
        from quantized_paged_kv_varlen_gb300 import synth
        self.q, self.torch, self.device = q, torch, device
        rng = np.random.default_rng((seed, 2))
        self.lengths = rng.integers(LO, HI + 1, size=B).astype(np.int32)
        bt, P = synth.page_tables(rng, self.lengths, PS)
        self.P = P
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        dev = device
        # cache holds L_b - 1 tokens; each step appends token L_b - 1 and decodes L_b tokens
        prev = self.lengths - 1
        T0 = int(prev.sum())
        self.k_pool = torch.zeros((P, PS, HKV, D), dtype=torch.uint8, device=dev)
        self.v_pool = torch.zeros_like(self.k_pool)
        self.ks = torch.zeros((P, PS, HKV), dtype=torch.float32, device=dev)
        self.vs = torch.zeros_like(self.ks)
        self.bt = torch.from_numpy(bt).to(dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        chunk = 1 << 22
        cu_prev = torch.from_numpy(np.cumsum(prev).astype(np.int32)).to(dev)
        k_all = torch.empty((T0, HKV, D), dtype=torch.bfloat16, device=dev)
        v_all = torch.empty_like(k_all)
        for t in range(0, T0, chunk):
            n = min(chunk, T0 - t)
            k_all[t:t + n] = torch.randn((n, HKV, D), generator=g, device=dev).to(torch.bfloat16)
            v_all[t:t + n] = torch.randn((n, HKV, D), generator=g, device=dev).to(torch.bfloat16)
        q.write_cache_fp8(k_all, v_all, cu_prev, self.bt, self.k_pool, self.v_pool, self.ks,
                          self.vs, error_word=self.err)
        del k_all, v_all
        # per-step inputs: one new token per request, the query
        self.k_new = torch.randn((B, HKV, D), generator=g, device=dev).to(torch.bfloat16)
        self.v_new = torch.randn((B, HKV, D), generator=g, device=dev).to(torch.bfloat16)
        self.qry = torch.randn((B, HQ, D), generator=g, device=dev).to(torch.bfloat16)
        self.cu_new = torch.arange(1, B + 1, dtype=torch.int32, device=dev)
        self.start_pos = torch.from_numpy(prev.astype(np.int32)).to(dev)
        self.out = torch.empty((B, HQ, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, HQ), dtype=torch.float32, device=dev)
        self.scale = 1.0 / float(np.sqrt(D))
        self.plan = q.DecodePlan(self.lengths, HQ, HKV, PS, D, device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)   # the plan copy overlaps the write
        torch.cuda.synchronize()
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error word {int(self.err.item())} during setup")
        self.total_bytes, self.attend_bytes = algorithmic_bytes(self.lengths)

    def step(self, ev_attend=None):
        """One decode step: append each request's new token, attend with the
        plan copied during the previous step, merge; then plan the next step
        (the host planner runs now and its copy to the other device buffer
        overlaps this step's kernels on a side stream: the plan/run split)."""
        q = self.q
        # the stream waits for the plan copy (issued a step ago, long done)
        # ahead of the write, so that nothing stands between the write, attend
        # and merge launches, which overlap their starts with the kernel before
        self.plan.wait_ready()
        q.write_cache_fp8(self.k_new, self.v_new, self.cu_new, self.bt, self.k_pool, self.v_pool,
                          self.ks, self.vs, start_pos=self.start_pos, error_word=self.err)
        if ev_attend is not None:
            ev_attend[0].record()
        self.plan.attend(self.qry, self.k_pool, self.v_pool, self.ks, self.vs, self.bt,
                         self.scale, error_word=self.err)
        if ev_attend is not None:
            ev_attend[1].record()
        self.plan.merge(self.out, self.lse)
        self.plan.replan(stream=self.copy_stream)


def kernel_source_hash(source=KERNEL_SOURCE):
    with open(source, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(summary=PROFILE_SUMMARY, source=KERNEL_SOURCE):
    """DRAM bytes (read + write) per launch from a committed ncu summary, or
    None when the kernel source changed since that capture."""
    if not os.path.exists(summary):
        return None
    vals = {}
    for line in open(summary):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(source):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _extra_traffic(profile, source):
    return profiled_traffic(os.path.join(ROOT, "profiles", profile),
                            os.path.join(ROOT, "quantized_paged_kv_varlen_gb300", "csrc", source))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def peaks_all():
    """hbm_gbs and bf16_tflops from MEASURED_PEAKS.json, else the fallbacks."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        out["hbm_gbs"] = float(p.get("hbm_gbs", out["hbm_gbs"]))
        out["bf16_tflops"] = float(p.get("bf16_tflops", out["bf16_tflops"]))
        out["source"] = "measured"
    return out


# ------------------------------------------------------------ CPU baseline

def cpu_worker(seconds, n_req):
    """Runs in a child process with one BLAS/OpenMP thread: times the oracle's
    paged decode on n_req requests of the workload (repeated for `seconds`)."""
    import numpy as np
    from quantized_paged_kv_varlen_gb300 import synth
    from oracle import attention as oatt
    from oracle import cache as ocache
    wl = synth.batched_decode(0)
    order = np.argsort(wl.lengths)
    reqs = [int(order[len(order) * (i + 1) // (n_req + 1)]) for i in range(n_req)]
    prepared = []
    for b in reqs:
        k, v = wl.kv(b)
        L = k.shape[0]
        n = (L + PS - 1) // PS
        bt = np.arange(n, dtype=np.int32)[None]
        z8 = np.zeros((n, PS, HKV, D), np.uint8)
        zs = np.zeros((n, PS, HKV), np.float32)
        kp, vp, ksp, vsp, _, _ = ocache.write_fp8_token_head(
            k, v, np.array([L]), np.array([0]), bt, PS, z8, z8, zs, zs)
        prepared.append((b, L, kp, vp, ksp, vsp, bt))
    lens = [p[1] for p in prepared]
    total, _ = algorithmic_bytes(lens)
    t0 = time.perf_counter()
    passes = 0
    while True:
        for b, L, kp, vp, ksp, vsp, bt in prepared:
            oatt.paged_decode_fp8(wl.q[[b]], kp, vp, ksp, vsp, bt, np.array([L]), wl.scale)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return {"value": total * passes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_req} requests of the workload (lengths {lens}), all 32 heads, "
                      f"{passes} passes in {dt:.1f} s, one thread",
            "seconds_per_pass": dt / passes, "tokens_per_s": len(lens) * passes / dt}


def cpu_worker_extras(seconds):
    """Child process, one thread: the oracle on bounded samples of the three
    other workloads, each for about `seconds`, in the units of their lines
    (useful causal FLOP of the sampled rows per second)."""
    import numpy as np
    from quantized_paged_kv_varlen_gb300 import synth
    from oracle import attention as oatt
    from oracle import cache as ocache
    from oracle import mla as omla
    from oracle import quant as oquant
    from oracle import rope as orope
    out = {}

    def timed(fn):
        t0 = time.perf_counter()
        n = 0
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= seconds:
                return n, dt

    # dense FP8 causal: rows of one (batch, head) slice of the workload
    dw = synth.dense_fp8(0)
    S, Dd = dw.S, dw.D
    codes, desc = [], []
    for which in ("q", "k", "v"):
        x = dw.slice(which, 0, 0)[None, :, None, :]
        s = oquant.absmax_scale(np.abs(x).max(axis=(1, 3)), oquant.FP8_QMAX)
        codes.append(oquant.quant_fp8(x, s[:, None, :, None]))
        desc.append(s)
    rows = list(range(0, S, S // 64))
    flops = float(sum(4.0 * Dd * (i + 1) for i in rows))
    n, dt = timed(lambda: oatt.dense_fp8(*codes, *desc, dw.scale, True,
                                         rows=[(0, i, 0) for i in rows]))
    out["fp8_attn_causal"] = {"value": flops * n / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "kind": "oracle",
                              "sample": f"{len(rows)} query rows (every {S // 64}th) of one "
                                        f"(batch, head) slice, S={S}, {n} passes in {dt:.1f} s"}
    # INT8 varlen prefill: one sequence of the workload, two heads, all rows
    pw = synth.varlen_prefill(0)
    b = int(np.argsort(pw.lengths)[len(pw.lengths) // 2])
    L = int(pw.lengths[b])
    beg = int(np.sum(pw.lengths[:b]))
    H2 = 2
    sl = lambda a: a[beg:beg + L, :H2]
    cos, sin = orope.cos_sin_table(L, pw.D, pw.theta)
    nbk = (L + 127) // 128
    P = (L + pw.page_size - 1) // pw.page_size
    bt = np.arange(P, dtype=np.int32)[None]
    kp0 = np.zeros((P, pw.page_size, H2, pw.D), np.int8)
    vp0 = np.zeros((P, pw.page_size, H2, pw.D), np.uint16)
    kp, vp, ksc, q8, qsc, _ = ocache.write_int8_block128_rope(
        sl(pw.q), sl(pw.k), sl(pw.v), np.array([L]), bt, pw.page_size, cos, sin, nbk, kp0, vp0)
    flops = 4.0 * pw.D * H2 * L * (L + 1) / 2
    n, dt = timed(lambda: oatt.paged_prefill_int8(q8, qsc, kp, ksc, vp, bt, np.array([L]),
                                                   np.array([L]), pw.scale, causal=True))
    out["int8_prefill_varlen"] = {"value": flops * n / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
                                  "kind": "oracle",
                                  "sample": f"sequence {b} (L={L}) of the workload, {H2} of 32 "
                                            f"heads, all rows, {n} passes in {dt:.1f} s"}
    # MLA sparse decode: two query tokens of the workload, all 128 heads
    mw = synth.mla_sparse(0, B=2, QN=128, lengths=[32768, 40000])
    pool = np.zeros((mw.num_pages, mw.block_size, 1, 656), np.uint8)
    for bb in range(mw.B):
        pool, _ = ocache.write_mla_rows(mw.kv(bb), np.array([mw.lengths[bb]]), np.array([0]),
                                        mw.block_table[bb:bb + 1], mw.block_size, pool)
    flops = 2 * 128.0 * 2048 * 2 * (576 + 512)
    n, dt = timed(lambda: omla.mla_sparse_decode(mw.q, pool, mw.sparse_indices, mw.block_table,
                                                 mw.lengths, mw.cu_seqlens_q, mw.scale))
    out["mla_sparse_decode"] = {"value": flops * n / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"2 query tokens (L = 32768, 40000), 128 heads, 2048 "
                                          f"ids each, {n} passes in {dt:.1f} s"}
    return out


def run_cpu_baseline_extras(seconds):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker-extras", str(seconds)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        why = (r.stderr.strip().splitlines() or ["?"])[-1][:200]
        return {k: {"value": None, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                    "sample": "failed: " + why}
                for k in ("fp8_attn_causal", "int8_prefill_varlen", "mla_sparse_decode")}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_cpu_baseline(seconds, n_req):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", str(seconds), str(n_req)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "failed: " + r.stderr.strip().splitlines()[-1][:200]}
    return json.loads(r.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------- arms

def run_reference(args):
    """The oracle as the reference arm: K timed steps, each the oracle's
    decode of a bounded sample (2 requests) of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    from quantized_paged_kv_varlen_gb300 import synth
    from oracle import attention as oatt
    from oracle import cache as ocache
    wl = synth.batched_decode(0)
    order = np.argsort(wl.lengths)
    reqs = [int(order[len(order) // 3]), int(order[2 * len(order) // 3])]
    prepared = []
    for b in reqs:
        k, v = wl.kv(b)
        L = k.shape[0]
        n = (L + PS - 1) // PS
        bt = np.arange(n, dtype=np.int32)[None]
        z8 = np.zeros((n, PS, HKV, D), np.uint8)
        zs = np.zeros((n, PS, HKV), np.float32)
        kp, vp, ksp, vsp, _, _ = ocache.write_fp8_token_head(
            k, v, np.array([L]), np.array([0]), bt, PS, z8, z8, zs, zs)
        prepared.append((b, L, kp, vp, ksp, vsp, bt))
    lens = [p[1] for p in prepared]
    total, _ = algorithmic_bytes(lens)

    def step():
        for b, L, kp, vp, ksp, vsp, bt in prepared:
            oatt.paged_decode_fp8(wl.q[[b]], kp, vp, ksp, vsp, bt, np.array([L]), wl.scale)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = total * args.steps / dt / 1e9
    sample = f"2 requests (lengths {lens}) of the workload per step, all 32 heads"
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "tokens_per_s": len(lens) * args.steps / dt,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_qpkv(args):
    import numpy as np
    import torch
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import quantized_paged_kv_varlen_gb300 as q
    if not os.path.exists(q.LIB_PATH):
        from quantized_paged_kv_varlen_gb300 import build
        if rank == 0:
            build.build()
        barrier(world, device)
    q.load()
    wb = DecodeBench(seed=rank, device=device)
    sampler = ClockSampler(local)
    sampler.start()
    # warm-up: W steps, and at least ~1 s of work so clocks settle
    t_w = time.time()
    n_w = 0
    while n_w < args.warmup or time.time() - t_w < args.min_warmup_s:
        wb.step()
        n_w += 1
        if n_w % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(world, device)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # the attend kernel's own duration, from events around it on every
    # ATT_EVERY-th step of the timed region (events between the launches cost
    # the step the overlap of consecutive kernels, so not on every step)
    att = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for i in range(0, args.steps, ATT_EVERY)}
    t_region0 = time.time()
    ev0.record()
    for i in range(args.steps):
        wb.step(att.get(i))
    ev1.record()
    torch.cuda.synchronize()
    t_region1 = time.time()
    barrier(world, device)
    ms = ev0.elapsed_time(ev1)
    ms_attend = sum(a.elapsed_time(b) for a, b in att.values()) / len(att)
    ms_max = max_over_ranks(ms, world, device)
    if int(wb.err.item()) != 0:
        raise RuntimeError(f"device error word {int(wb.err.item())}")

    # end to end through the public API with host buffers in the timed region:
    # the step's inputs (query, new K, new V) staged in one page-locked
    # buffer and sent with one copy; the device tensors are views of its
    # device twin
    parts = [wb.qry, wb.k_new, wb.v_new]
    sizes = [t.numel() for t in parts]
    pin_in = torch.cat([t.reshape(-1).cpu() for t in parts]).pin_memory()
    dev_in = torch.empty_like(pin_in, device=device)
    offs = np.cumsum([0] + sizes)
    wb.qry, wb.k_new, wb.v_new = (dev_in[offs[i]:offs[i + 1]].view(parts[i].shape)
                                  for i in range(3))
    pin_o = torch.empty(wb.out.shape, dtype=wb.out.dtype).pin_memory()
    h2d = pin_in.numel() * pin_in.element_size()
    d2h = pin_o.numel() * pin_o.element_size()

    def e2e_step():
        dev_in.copy_(pin_in, non_blocking=True)
        wb.step()
        pin_o.copy_(wb.out, non_blocking=True)
    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world, device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, device)
    sampler.stop()
    clocks = sampler.summary(t_region0, t_region1)

    if rank != 0:
        return
    step_s = ms_max / 1e3 / args.steps
    value = wb.total_bytes * world / step_s / 1e9
    peak, peak_kind = peaks()
    achieved = wb.attend_bytes / (ms_attend / 1e3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.cpu_seconds, 3)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": f"U{{{LO}..{HI}}}",
                   "parallelism": f"replicas x{world} (independent requests, no collective)",
                   "l2": f"no flush: {wb.total_bytes / 1e6:.0f} MB moved per step > "
                         f"{L2_BYTES / 1e6:.0f} MB L2",
                   "step": "write_cache(1 token/request) + split-KV attend + LSE merge + "
                           "host plan of the next step (copy on a side stream)",
                   "sum_kv_tokens": int(wb.lengths.sum())},
        "tokens_per_s": B * world / step_s,
        "algorithmic_bytes_per_step": wb.total_bytes,
        "roofline": {"bound": "hbm", "kernel": "decode_heads_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": profiled_traffic(),
                     "algorithmic_bytes_per_launch": wb.attend_bytes,
                     "ms_per_launch": ms_attend,
                     "ms_per_launch_from": f"CUDA events around the attend launch on every "
                                           f"{ATT_EVERY}th timed step ({len(att)} samples)"},
        "cpu_baseline": cpu,
        "e2e": {"value": wb.total_bytes * world / (ms_e2e / 1e3 / args.steps) / 1e9,
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e / args.steps},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_extras:
        line["also"] = run_extras(device)
        if not args.no_cpu_baseline:
            cpu_x = run_cpu_baseline_extras(args.cpu_seconds / 3)
            for k, v in line["also"].items():
                v["cpu_baseline"] = cpu_x.get(k)
    print(json.dumps(line), flush=True)


def _median_ms(fn, iters, flush=None, reps=1):
    """Median CUDA-event time of fn() on the current stream: L2 flushed
    before each run when `flush` is given, else `reps` calls back to back
    between the events (divided by reps), so the binding's host time per
    call overlaps the kernels instead of idling the GPU inside the timed
    region (used where the inputs are larger than L2)."""
    import torch
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps if flush is None else 1):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / (reps if flush is None else 1))
    ts.sort()
    return ts[len(ts) // 2]


def run_extras(device, iters=10):
    """The other hot paths at their full sizes, timed alone: dense FP8
    causal attention (B=4, S=8192, H=32, D=128), the varlen INT8-QK paged
    prefill (8 sequences, L ~ U{256..4096}, 32 heads, page 64) and the
    MLA-absorb sparse decode (B=32, 128 heads, 2048 ids of L ~ U{32768..65536})."""
    import numpy as np
    import torch
    import quantized_paged_kv_varlen_gb300 as q
    from quantized_paged_kv_varlen_gb300 import synth
    pk = peaks_all()
    bf16, fp8 = pk["bf16_tflops"], 2.0 * pk["bf16_tflops"]
    out = {}
    err = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    # dense FP8, causal
    B4, S4, H4, D4 = 4, 8192, 32, 128
    q8, k8, v8, qd, kd, vd = synth.dense_fp8_device(0, B4, S4, H4, D4, device)
    o4 = torch.empty((B4, S4, H4, D4), dtype=torch.bfloat16, device=device)
    f4 = lambda: q.fp8_attn_fwd(q8, k8, v8, qd, kd, vd, causal=True, out=o4, error_word=err)
    for _ in range(3):
        f4()
    ms = _median_ms(f4, iters, reps=3)
    flops = 2.0 * B4 * H4 * D4 * S4 * (S4 + 1)
    tf = flops / (ms / 1e3) / 1e12
    out["fp8_attn_causal"] = {
        "workload": f"dense FP8 causal B={B4} S={S4} H={H4} D={D4} (BSND e4m3, per-(b,h) descales)",
        "ms": ms, "value": tf, "unit": "TFLOP/s", "flops": flops,
        "timing": "median of 10 CUDA-event samples of 3 back-to-back calls (inputs > L2)",
        "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8, "unit": "TFLOP/s",
                     "frac": tf / fp8, "peak_source": "measured bf16_tflops x 2 (fp8 nominal ratio)",
                     "traffic": _extra_traffic("fp8_attn_causal_b4_s8192_h32.txt", "fp8_attn.cu"),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"}}
    del q8, k8, v8, o4

    # varlen INT8-QK paged prefill (cache written by the library)
    wl = synth.varlen_prefill(0)
    L = wl.lengths
    T, H, D = wl.q.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    cos, sin = q.rope_table(wl.theta, int(L.max()), 128)
    nb = wl.num_blocks
    k_pool = torch.zeros((wl.num_pages, wl.page_size, H, D), dtype=torch.int8, device=device)
    v_pool = torch.zeros((wl.num_pages, wl.page_size, H, D), dtype=torch.bfloat16, device=device)
    ks = torch.zeros((len(L), nb, H), dtype=torch.float32, device=device)
    qs = torch.zeros_like(ks)
    q8p = torch.zeros((T, H, D), dtype=torch.int8, device=device)
    cu, bt, lk = t(synth.inclusive_prefix(L)), t(wl.block_table), t(L)
    qb, kb, vb = (t(x).to(torch.bfloat16) for x in (wl.q, wl.k, wl.v))
    wr = lambda: q.write_cache_int8_block128_rope(qb, kb, vb, cu, bt, int(L.max()), cos, sin,
                                                  k_pool, v_pool, ks, q8p, qs, error_word=err)
    wr()
    op = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
    wsp = q.prefill_workspace(len(L), T, H, device)
    fp = lambda: q.prefill_paged(q8p, qs, k_pool, ks, v_pool, bt, cu, lk, causal=True, out=op,
                                 workspace=wsp, error_word=err)
    for _ in range(3):
        fp()
    ms = _median_ms(fp, iters, reps=3)
    ms_w = _median_ms(wr, iters, reps=5)
    flops = float(sum(4.0 * D * H * int(x) * (int(x) + 1) / 2 for x in L))
    tf = flops / (ms / 1e3) / 1e12
    # the write moves bf16 q, k, v in and int8 q, int8 k, bf16 v out (the
    # per-block scales are a few KB): 10 bytes per (token, head, dim)
    w_bytes = float(T) * H * D * (2 + 2 + 2 + 1 + 1 + 2)
    w_gbs = w_bytes / (ms_w / 1e3) / 1e9
    out["int8_prefill_varlen"] = {
        "workload": f"varlen causal prefill {len(L)} seqs L={L.tolist()} H={H} D={D} page 64, "
                    "INT8 Q/K block-128 scales, bf16 V",
        "ms": ms, "value": tf, "unit": "TFLOP/s", "flops": flops, "write_cache_ms": ms_w,
        "timing": "median of 10 CUDA-event samples of 3 (the write: 5) back-to-back calls "
                  "(inputs > L2)",
        "write_cache_roofline": {
            "bound": "hbm", "bytes": w_bytes, "achieved": w_gbs, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": w_gbs / pk["hbm_gbs"],
            "traffic": _extra_traffic("write_int8_block128_rope_8seqs_h32.txt", "write_cache.cu"),
            "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16, "unit": "TFLOP/s",
                     "frac": tf / bf16, "peak_source": "measured bf16_tflops (f16/bf16 MMAs)",
                     "traffic": _extra_traffic("prefill_int8_8seqs_h32_page64.txt",
                                               "prefill_int8.cu"),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"}}
    # the same prefill over ragged (packed, non-paged) K/V of the same sizes
    gk = torch.Generator(device=device)
    gk.manual_seed(13)
    k_rag = torch.randint(-127, 128, (T, H, D), generator=gk, dtype=torch.int8, device=device)
    v_rag = torch.randn((T, H, D), generator=gk, device=device).to(torch.bfloat16)
    fr = lambda: q.prefill_paged(q8p, qs, k_rag, ks, v_rag, None, cu, None, causal=True, out=op,
                                 workspace=wsp, error_word=err, cu_seqlens_kv=cu)
    for _ in range(3):
        fr()
    ms_r = _median_ms(fr, iters, reps=3)
    out["int8_prefill_varlen"]["ragged_kv_ms"] = ms_r
    out["int8_prefill_varlen"]["ragged_kv_tflops"] = flops / (ms_r / 1e3) / 1e12
    del k_rag, v_rag
    # the same paged prefill with Sage-style FP8 V (per-channel scales) and an
    # FP8 P.V product; the write quantises V with the same call
    v8_pool = torch.zeros((wl.num_pages, wl.page_size, H, D), dtype=torch.uint8, device=device)
    vsc = torch.zeros((len(L), H, D), dtype=torch.float32, device=device)
    wsw = q.smooth_workspace(len(L), nb, H, device)
    wr8 = lambda: q.write_cache_int8_block128_rope(qb, kb, vb, cu, bt, int(L.max()), cos, sin,
                                                   k_pool, v8_pool, ks, q8p, qs, error_word=err,
                                                   v_channel_scale=vsc, workspace=wsw)
    wr8()
    f8 = lambda: q.prefill_paged(q8p, qs, k_pool, ks, v8_pool, bt, cu, lk, causal=True, out=op,
                                 workspace=wsp, error_word=err, v_scale=vsc)
    for _ in range(3):
        f8()
    ms_8 = _median_ms(f8, iters, reps=3)
    out["int8_prefill_varlen"]["fp8_v_ms"] = ms_8
    out["int8_prefill_varlen"]["fp8_v_tflops"] = flops / (ms_8 / 1e3) / 1e12
    out["int8_prefill_varlen"]["fp8_v_write_cache_ms"] = _median_ms(wr8, iters, reps=5)
    del k_pool, v_pool, v8_pool, q8p, qb, kb, vb, op

    # MLA-absorb sparse decode
    d = synth.mla_sparse_device(0, device)
    pool = torch.empty((d["num_pages"], 64, 1, 656), dtype=torch.uint8, device=device)
    q.write_cache_mla(d["kv"], d["cu_kv"], d["bt"], pool, error_word=err)
    om = torch.empty((32, 128, 512), dtype=torch.bfloat16, device=device)
    wsm = q.mla_workspace(32, 2048, device)
    fm = lambda: q.mla_sparse_decode(d["q"], pool, d["idx"], d["bt"], d["lk"], d["cu_q"],
                                     scale=d["scale"], out=om, workspace=wsm, error_word=err)
    for _ in range(3):
        fm()
    ms = _median_ms(fm, iters * 2, flush=flush)
    flops = 32.0 * 128 * 2048 * 2 * (576 + 512)
    row_bytes = 32 * 2048 * 656 + 32 * 128 * 576 * 2 + 32 * 128 * 512 * 2 + 32 * 2048 * 4
    tf = flops / (ms / 1e3) / 1e12
    gbs = row_bytes / (ms / 1e3) / 1e9
    t_qk = _extra_traffic("mla_qk_b32.txt", "mla_sparse.cu")
    t_pv = _extra_traffic("mla_pv_b32.txt", "mla_sparse.cu")
    mla_traffic = t_qk + t_pv if t_qk is not None and t_pv is not None else None
    out["mla_sparse_decode"] = {
        "workload": "MLA-absorb sparse decode B=32 QN=128 D=576/512, 2048 ids of "
                    "L~U{32768..65536}, block 64, INT8 nope + bf16 rope rows",
        "ms": ms, "value": tf, "unit": "TFLOP/s", "flops": flops, "gb_per_s": gbs,
        "l2": "flushed (256 MB write) before each run",
        "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16, "unit": "TFLOP/s",
                     "frac": tf / bf16, "hbm_frac": gbs / pk["hbm_gbs"],
                     "peak_source": "measured bf16_tflops; hbm_frac of measured hbm_gbs",
                     "traffic": mla_traffic,
                     "traffic_unit": "bytes per call (ncu dram read + write of the QK and PV "
                                     "kernels)"}}
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the extra workloads")
    return out


def set_batch(n):
    """Number of requests per rank (the workload's B)."""
    global B, WORKLOAD
    if n != B:
        WORKLOAD = WORKLOAD.replace(f"B={B},", f"B={n},")
        B = n


def main():
    if len(sys.argv) >= 2 and sys.argv[1] == "--cpu-worker":
        print(json.dumps(cpu_worker(float(sys.argv[2]), int(sys.argv[3]))))
        return
    if len(sys.argv) >= 2 and sys.argv[1] == "--cpu-worker-extras":
        print(json.dumps(cpu_worker_extras(float(sys.argv[2]))))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["qpkv", "reference"], default="qpkv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the dense FP8, INT8 prefill and MLA decode measurements")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up for at least this long so clocks settle")
    ap.add_argument("--batch", type=int, default=B,
                    help="requests per rank (64 is the benchmark; smaller batches are for "
                         "profiler captures)")
    args = ap.parse_args()
    set_batch(args.batch)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_qpkv(args)


if __name__ == "__main__":
    main()
