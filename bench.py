#!/usr/bin/env python3
"""Benchmark of the paged-KV GQA hot path on one GB300 (or N replicas).

One step = the whole path over one batch: ensure_append (host, copy-on-append),
per layer append + attend (device: page-table upload, append scatter, split-K
decode, log-sum-exp merge), advance (host), then truncate back to the step's
starting lengths so every step does identical work.

Default workload: continuous-batching decode, M = 256 rows, lengths
log-uniform in [128, 32768], 32 query / 8 kv heads of width 128, block size
16, a shuffled pool of 600 000 blocks (78.6 GB of K+V), f32 N(0, 1) data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
                    [--workload NAME] [--no-cpu-baseline]

Prints ONE JSON line (rank 0).  ``value`` is KV GB/s: the K and V rows each
row attends over, read once per layer (sum of total_k * kv_dim * 8 bytes), per
second of device time, summed over all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attention KV GB/s (fraction of GB300 HBM peak); rows·layers/s"
HBM_FALLBACK_GBS = 6800.0


# --------------------------------------------------------------- helpers ----

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


_CSRC = "paged_kv_gqa_nx_gb300/csrc/"
# the sources a committed ncu summary was taken on, per (kernel, pool element
# type): a summary's sha256 prefix covers these files in this order
KERNEL_SOURCES = {
    ("decode", "f32"): ["pkv_kernels.cu", "pkv_rows.h"],
    ("decode", "bf16"): ["pkv_decode_mma.cu", "pkv_rows.h"],
    ("decode", "fp8"): ["pkv_decode_mma.cu", "pkv_rows.h"],
    ("prefill", "f32"): ["pkv_prefill.cu", "pkv_tcgen05.h"],
    ("prefill", "bf16"): ["pkv_prefill.cu", "pkv_tcgen05.h"],
    ("prefill", "fp8"): ["pkv_prefill.cu", "pkv_tcgen05.h"],
}
PROFILE_FILES = {"decode": "decode_%s.md", "prefill": "prefill_tc_%s.md"}


def measured_bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


_TF32_CACHE = {}


def measured_tf32_tflops(n=8192, reps=10):
    """cuBLAS TF32 dense matmul throughput on this GPU, measured the way the
    bf16 figure in MEASURED_PEAKS.json is: torch.matmul of two n x n f32
    matrices with TF32 tensor cores allowed, 2 n^3 flops, best of `reps`
    launches timed with CUDA events.  Cached per process."""
    if "v" in _TF32_CACHE:
        return _TF32_CACHE["v"]
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e-3)
        del a, b, c
        torch.cuda.empty_cache()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    _TF32_CACHE["v"] = 2.0 * n ** 3 / best / 1e12
    return _TF32_CACHE["v"]


def tensor_peak(kv_dtype="f32"):
    """f32-accurate peak of the prefill contraction: the measured dense f16 /
    bf16 tensor rate (MEASURED_PEAKS.json, cuBLAS bf16; f16 runs at the same
    rate) divided by the f16 products each f32-accurate product takes -- three
    (x0*y0 + x0*y1 + x1*y0) on an f32 pool, two on bf16 / fp8 pools (their K
    and V are single f16 pieces).  The detail also carries the live cuBLAS
    TF32 rate and the issue rates of the kernel's own instruction."""
    f16, kind = measured_bf16_peak()
    products = 3.0 if kv_dtype == "f32" else 2.0
    detail = {"f16_tflops": round(f16, 1), "f16_source": kind + " (MEASURED_PEAKS.json bf16_tflops)",
              "f16_products_per_f32_product": products,
              "tf32_tflops_cublas": round(measured_tf32_tflops(), 1)}
    detail.update(tcgen05_rates())
    return f16 / products, detail


def tcgen05_rates():
    """The issue rate of the prefill kernel's own instruction, measured by the
    library's probe (pkv_probe_f16_mma): tcgen05.mma kind::f16, M = 128, A in
    tensor memory, at N = 64 (its QK^T products) and N = 128 (its PV
    products)."""
    if "probe" in _TF32_CACHE:
        return _TF32_CACHE["probe"]
    import paged_kv_gqa_nx_gb300 as pkv
    out = {}
    for n in (64, 128):
        clk, tf = pkv.pkv_probe_f16_mma(n, True, 4096)
        out["tcgen05_f16_n%d" % n] = {"clk_per_mma": round(clk, 2), "tflops": round(tf, 1)}
    _TF32_CACHE["probe"] = out
    return out


def kernel_source_digest(kernel: str = "decode", kv_dtype: str = "f32"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[(kernel, kv_dtype)]:
        with open(os.path.join(ROOT, _CSRC + name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "decode", kv_dtype: str = "f32"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary for
    this workload and pool element type (f32 summaries carry no suffix), if it
    was taken on the current kernel source; else None."""
    name = workload if kv_dtype == "f32" else "%s_%s" % (workload, kv_dtype)
    path = os.path.join(ROOT, "profiles", PROFILE_FILES[kernel] % name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_digest(kernel, kv_dtype):
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,uuid")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            if self.uuid and self.uuid not in parts[7]:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workloads ----

def get_workload(name):
    from synth import workloads as wl
    table = {
        "continuous_batching_m256": wl.continuous_batching_m256,
        "continuous_batching_small": wl.continuous_batching_small,
        "batched_decode_m64": wl.batched_decode_m64,
        "chunked_prefill": wl.chunked_prefill,
        "shared_prefix_forks": wl.shared_prefix_forks,
    }
    if name not in table:
        raise SystemExit("unknown workload %r; choose from %s" % (name, sorted(table)))
    return table[name]()


class DeviceRun:
    """The workload resident on one GPU: pool, sequences with histories, and
    the per-layer step inputs."""

    def __init__(self, w, rank=0, kv_dtype="f32"):
        import torch
        import paged_kv_gqa_nx_gb300 as pkv
        from synth import workloads as wl
        self.torch, self.pkv, self.w = torch, pkv, w
        dev = torch.device("cuda", torch.cuda.current_device())
        bs = w.block_size
        self.stream = torch.cuda.current_stream()
        max_tok = w.max_tokens() + 2
        if w.name == "shared_prefix_forks":
            max_tok = int(w.extra["prefix"]) + 2 * 256 + 2
        self.bf16 = kv_dtype == "bf16"
        self.fp8 = kv_dtype == "fp8"
        self.elem = 1 if self.fp8 else 2 if self.bf16 else 4
        self.K = torch.empty((w.n_blocks, w.n_layers, bs, w.kv_dim), device=dev,
                             dtype=(torch.float8_e4m3fn if self.fp8 else
                                    torch.bfloat16 if self.bf16 else torch.float32))
        self.V = torch.empty_like(self.K)
        self.pool = pkv.pkv_pool_new(w.n_blocks, w.n_layers, w.kv_dim, bs, self.K, self.V,
                                     w.M + 8, -(-max_tok // bs) + 1, self.stream,
                                     flags=(pkv.PKV_POOL_FP8 if self.fp8 else
                                            pkv.PKV_POOL_BF16 if self.bf16 else 0))
        assert self.pool, pkv.pkv_last_error()
        # shuffle the free list through the public API
        ids = [pkv.pkv_alloc_block(self.pool) for _ in range(w.n_blocks)]
        assert ids[0] == 0 and ids[-1] == w.n_blocks - 1
        for b in wl.release_order(w.n_blocks, w.seed):
            pkv.pkv_unref_block(self.pool, int(b))
        seed = w.seed * 7919 + rank
        self.seqs = []
        if w.name == "shared_prefix_forks":
            prefix = int(w.extra["prefix"])
            root = pkv.pkv_seq_new(self.pool, max_tok)
            self._grow_and_fill(root, prefix, seed)
            self.root = root
            forks = [pkv.pkv_seq_fork(root) for _ in range(w.M)]
            div = [int(x) for x in w.n_q]
            self._chunk(forks, div, seed + 5)                 # divergent chunks, once
            self.seqs = forks
            self.n_q = [1] * w.M                              # timed step: batched decode
        else:
            for r in range(w.M):
                s = pkv.pkv_seq_new(self.pool, max_tok)
                self._grow_and_fill(s, int(w.past_len[r]), seed + 17 * r)
                self.seqs.append(s)
            self.n_q = [int(x) for x in w.n_q]
        self.base_len = [pkv.pkv_seq_len(s) for s in self.seqs]
        self.c_seqs = pkv.seq_array(self.seqs)
        self.c_nq = pkv.i32_array(self.n_q)
        self.c_base = pkv.i32_array(self.base_len)
        self.T = sum(self.n_q)
        self.inputs = []
        for layer in range(w.n_layers):
            self.inputs.append(tuple(wl.normal(shape, seed + 1000 * layer + k, dev) for k, shape in
                                     enumerate([(self.T, w.q_dim), (self.T, w.kv_dim), (self.T, w.kv_dim)])))
        self.out = torch.empty((self.T, w.q_dim), device=dev, dtype=torch.float32)
        # device addresses, marshalled once (the binding takes raw addresses)
        self.input_ptrs = [tuple(t.data_ptr() for t in qkv) for qkv in self.inputs]
        self.out_ptr = self.out.data_ptr()
        # algorithmic bytes: every visible K and V row read once per row and layer
        tk = [b + n for b, n in zip(self.base_len, self.n_q)]
        self.kv_bytes_per_layer = float(sum(tk)) * w.kv_dim * self.elem * 2
        self.kv_bytes = self.kv_bytes_per_layer * w.n_layers
        # unique bytes: distinct physical rows behind the visible positions
        # (forks share prefix pages), plus each row's new positions
        keys = []
        for s_, L in zip(self.seqs, self.base_len):
            if L:
                pt = np.asarray(pkv.pkv_seq_page_table(s_), dtype=np.int64)
                pos = np.arange(L, dtype=np.int64)
                keys.append(pt[pos // bs] * bs + pos % bs)
        n_unique = (np.unique(np.concatenate(keys)).size if keys else 0) + sum(self.n_q)
        self.unique_kv_bytes = float(n_unique) * w.kv_dim * self.elem * 2 * w.n_layers
        self.q_out_bytes = float(self.T) * w.q_dim * 4 * 2 * w.n_layers
        torch.cuda.synchronize()

    def _grow_and_fill(self, s, L, seed):
        from synth import workloads as wl
        pkv, torch, w = self.pkv, self.torch, self.w
        if L == 0:
            return
        pkv.check(pkv.pkv_ensure_append(s, L))
        pkv.check(pkv.pkv_advance(s, L))
        pt = torch.tensor(pkv.pkv_seq_page_table(s), device=self.K.device, dtype=torch.long)
        pos = torch.arange(L, device=self.K.device)
        for layer in range(w.n_layers):
            self.K[pt[pos // w.block_size], layer, pos % w.block_size] = wl.normal(
                (L, w.kv_dim), seed + 2 * layer, self.K.device).to(self.K.dtype)
            self.V[pt[pos // w.block_size], layer, pos % w.block_size] = wl.normal(
                (L, w.kv_dim), seed + 2 * layer + 1, self.K.device).to(self.V.dtype)

    def _chunk(self, seqs, ns, seed):
        from synth import workloads as wl
        pkv, w = self.pkv, self.w
        T = sum(ns)
        dev = self.K.device
        Q, K, V = (wl.normal((T, d), seed + i, dev) for i, d in enumerate([w.q_dim, w.kv_dim, w.kv_dim]))
        out = self.torch.empty((T, w.q_dim), device=dev)
        pkv.check(pkv.pkv_ensure_append_batch(seqs, ns))
        for layer in range(w.n_layers):
            pkv.check(pkv.pkv_attn_batch(seqs, ns, Q, K, V, w.n_heads, w.n_kv_heads, w.head_dim,
                                         layer, 1, w.scale, out))
        pkv.check(pkv.pkv_advance_batch(seqs, ns))

    def step(self, host=None):
        """One pass of the hot path.  host = (Qh, Kh, Vh, outh) pinned buffers
        to run it through the host-buffer entry point instead."""
        pkv, w = self.pkv, self.w
        seqs, nq = self.c_seqs, self.c_nq
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        for layer in range(w.n_layers):
            if host is None:
                Q, K, V = self.input_ptrs[layer]
                pkv.check(pkv.pkv_attn_batch(seqs, nq, Q, K, V, w.n_heads, w.n_kv_heads,
                                             w.head_dim, layer, 1, w.scale, self.out_ptr))
            else:
                Qh, Kh, Vh, oh = host[layer]
                pkv.check(pkv.pkv_attn_batch_host(seqs, nq, Qh, Kh, Vh, w.n_heads,
                                                  w.n_kv_heads, w.head_dim, layer, 1, w.scale, oh))
        pkv.check(pkv.pkv_advance_batch(seqs, nq))
        pkv.check(pkv.pkv_seq_truncate_batch(seqs, self.c_base))

    def host_buffers(self):
        bufs = []
        for layer in range(self.w.n_layers):
            Q, K, V = self.inputs[layer]
            bufs.append((Q.cpu().pin_memory(), K.cpu().pin_memory(), V.cpu().pin_memory(),
                         self.torch.empty(self.out.shape, dtype=self.torch.float32).pin_memory()))
        return bufs

    def histories_for(self, rows):
        """Host copies of the rows' K/V histories (layer 0) and step inputs."""
        torch, pkv, w = self.torch, self.pkv, self.w
        res = []
        offs = np.concatenate([[0], np.cumsum(self.n_q)])
        Q, K, V = (t.cpu().numpy() for t in self.inputs[0])
        for r in rows:
            L = self.base_len[r]
            pt = torch.tensor(pkv.pkv_seq_page_table(self.seqs[r]), device=self.K.device,
                              dtype=torch.long)
            pos = torch.arange(L, device=self.K.device)
            Kh = self.K[pt[pos // w.block_size], 0, pos % w.block_size].float().cpu().numpy()
            Vh = self.V[pt[pos // w.block_size], 0, pos % w.block_size].float().cpu().numpy()
            o, n = int(offs[r]), self.n_q[r]
            res.append((Q[o:o + n], np.concatenate([Kh, K[o:o + n]]), np.concatenate([Vh, V[o:o + n]]),
                        n, L + n))
        return res

    def close(self):
        self.torch.cuda.synchronize()
        self.pkv.pkv_pool_free(self.pool)


# ---------------------------------------------------------- oracle timing ----

def oracle_sample(w, lengths, budget_s, rng_seed=0, n_q=None, threads=1):
    """Choose rows of the workload for a bounded oracle run on `threads` host
    threads (0: all cores): rows in seeded order until their estimated time
    reaches the budget."""
    import oracle
    rng = np.random.default_rng(rng_seed)
    order = rng.permutation(len(lengths))
    # calibrate on a small synthetic row, on the thread count that will run
    L = 2048
    Q = np.ones((1, w.q_dim), np.float32)
    K = np.ones((L, w.kv_dim), np.float32)
    oracle.set_threads(threads)
    try:
        t0 = time.perf_counter()
        oracle.attend(Q, K, K, 1, L, w.n_heads, w.n_kv_heads, w.head_dim, 1, w.scale)
        per_key = (time.perf_counter() - t0) / L
    finally:
        oracle.set_threads(0)
    rows, est = [], 0.0
    for r in order:
        cost = per_key * lengths[r] * (1 if n_q is None else n_q[r])
        if rows and est + cost > budget_s:
            continue
        rows.append(int(r))
        est += cost
        if est >= budget_s:
            break
    return sorted(rows)


def time_oracle(samples, w, threads=1):
    """Seconds the oracle takes over `samples` on `threads` host threads (0:
    all cores), the K/V bytes it read, and the thread count in effect."""
    import oracle
    used = oracle.set_threads(threads)
    try:
        t0 = time.perf_counter()
        for (Q, K, V, n, tk) in samples:
            rc, _ = oracle.attend(Q, K, V, n, tk, w.n_heads, w.n_kv_heads, w.head_dim, 1, w.scale)
            assert rc == 0
        dt = time.perf_counter() - t0
    finally:
        oracle.set_threads(0)
    nbytes = sum(float(tk) * w.kv_dim * 8 for (_, _, _, _, tk) in samples)
    return dt, nbytes, used


# ------------------------------------------------------------------- arms ----

def dist_setup(n_gpus):
    import torch
    if n_gpus <= 1 and "WORLD_SIZE" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    backend = os.environ.get("PKV_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, dist


def max_over_ranks(value, dist):
    if dist is None:
        return value
    import torch
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([float(value)], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def timed_steps(run, steps, stream_sync=True):
    """Run `steps` steps between CUDA events on the pool stream with the
    library's per-launch profiling on; returns (device ms, host s, launches,
    per-kernel (ms, launches))."""
    import torch
    pkv = run.pkv
    pkv.pkv_profile_reset()
    pkv.pkv_profile_enable(True)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    launches0 = pkv.pkv_launch_count()
    h0 = time.perf_counter()
    ev0.record(run.stream)
    for _ in range(steps):
        run.step()
    ev1.record(run.stream)
    host_s = time.perf_counter() - h0
    torch.cuda.synchronize()
    launches = pkv.pkv_launch_count() - launches0
    pkv.pkv_profile_enable(False)
    kern = {pkv.KERNEL_NAMES[k]: pkv.pkv_profile_read(k) for k in range(pkv.PKV_KERNEL_KINDS)}
    return ev0.elapsed_time(ev1), host_s, launches, kern


def roofline_of(run, w, kern, steps, workload, kv_dtype, tensor_flops_per_layer):
    """The roofline entry of the kernel that takes most of the step."""
    dec_ms, dec_n = kern["decode"]
    pre_ms, pre_n = kern["prefill"]
    if pre_ms > dec_ms and pre_n:
        # flops per launch: one layer call's tensor-core work over its prefill launches
        pre_per_layer = pre_n / (steps * w.n_layers)
        pre_avg_s = pre_ms * 1e-3 / pre_n
        flops_per_launch = tensor_flops_per_layer / max(pre_per_layer, 1e-9)
        tpeak, detail = tensor_peak(kv_dtype)
        achieved = flops_per_launch / pre_avg_s / 1e12
        return {"bound": "tensor", "kernel": "prefill (tcgen05 kind::f16, split f32 operands)",
                "achieved": round(achieved, 1), "peak": round(tpeak, 1),
                "peak_source": ("measured dense bf16 rate (MEASURED_PEAKS.json, %.1f TFLOP/s; f16 the same) "
                                "/ %d f16 products per f32 product"
                                % (detail["f16_tflops"], detail["f16_products_per_f32_product"])),
                "peak_detail": detail,
                "unit": "TFLOP/s", "frac": round(achieved / tpeak, 4),
                "traffic": profiled_traffic(workload, "prefill", kv_dtype),
                "alg_flops_per_launch": flops_per_launch,
                "avg_launch_ms": round(pre_avg_s * 1e3, 4)}
    peak, peak_kind = measured_hbm_peak()
    dec_avg_s = dec_ms * 1e-3 / max(dec_n, 1)
    alg_bytes = run.kv_bytes_per_layer + run.T * w.q_dim * 4 * 2
    achieved = alg_bytes / dec_avg_s / 1e9 if dec_n else None
    return {"bound": "hbm", "kernel": "decode (split-K paged attention)",
            "achieved": round(achieved, 1) if achieved else None, "peak": peak,
            "peak_source": (peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                            else "fallback"), "unit": "GB/s",
            "frac": round(achieved / peak, 4) if achieved else None,
            "traffic": profiled_traffic(workload, "decode", kv_dtype), "alg_bytes_per_launch": alg_bytes,
            "avg_launch_ms": round(dec_avg_s * 1e3, 4)}


def tensor_flops(run, w):
    """Tensor-core work of one layer call as the library laid it out: the
    visible (query, key) pairs of the prefill rows and of the shared-prefix
    pass, 2 flops each for q.k and for p.v per head dimension."""
    work = run.pkv.pkv_pool_last_work(run.pool)
    return 4.0 * w.head_dim * w.n_heads * (work["prefill_pairs"] + work["prefix_pairs"])


# the other workloads the default run measures beside the headline one
EXTRA_WORKLOADS = ("batched_decode_m64", "chunked_prefill", "shared_prefix_forks")


def measure_extra(name, args, rank):
    """One more workload through the same step and timing: ms/step, KV GB/s
    and the dominant kernel's roofline."""
    import torch
    w = get_workload(name)
    run = DeviceRun(w, rank, "f32")
    try:
        for _ in range(max(3, args.warmup)):
            run.step()
        torch.cuda.synchronize()
        tfl = tensor_flops(run, w)
        steps = max(5, min(args.steps, 30))
        # two timed windows, the faster one kept: a host-side stall in one
        # window (the device idles while the host prepares a step) does not
        # decide the line
        windows = [timed_steps(run, steps) for _ in range(2)]
        ms_total, host_s, launches, kern = min(windows, key=lambda x: x[0])
        ms_step = ms_total / steps
        peak, _ = measured_hbm_peak()
        value = run.kv_bytes / (ms_step * 1e-3) / 1e9
        return {"ms_per_step": round(ms_step, 4), "kv_gbs": round(value, 2),
                "frac_of_hbm_peak": round(value / peak, 4),
                "unique_kv_gbs": round(run.unique_kv_bytes / (ms_step * 1e-3) / 1e9, 2),
                "rows_layers_per_s": round(run.T * w.n_layers / (ms_step * 1e-3), 1),
                "kv_bytes_per_step": run.kv_bytes, "steps": steps,
                "windows_ms_per_step": [round(x[0] / steps, 4) for x in windows],
                "host_ms_per_step": round(host_s * 1e3 / steps, 4),
                "gpu_launches": launches,
                "kernels_ms_per_step": {k: round(v[0] / steps, 4) for k, v in kern.items() if v[1]},
                "roofline": roofline_of(run, w, kern, steps, name, "f32", tfl)}
    finally:
        run.close()
        del run
        torch.cuda.empty_cache()


def run_pkv(args):
    import torch
    import paged_kv_gqa_nx_gb300 as pkv
    rank, world, dist = dist_setup(args.gpus)
    if args.split_keys:
        pkv.check(pkv.pkv_set_split_keys(args.split_keys))
    w = get_workload(args.workload)
    run = DeviceRun(w, rank, args.kv_dtype)
    if args.image_cache_mb:
        pkv.check(pkv.pkv_pool_set_image_cache(run.pool, args.image_cache_mb << 20))
    peak, peak_kind = measured_hbm_peak()

    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    tensor_flops_per_layer = tensor_flops(run, w)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    ms_total, host_s, launches, kern = timed_steps(run, args.steps)
    barrier(dist)
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, dist)
    ms_step = ms_total / args.steps
    value = world * run.kv_bytes * args.steps / (ms_total * 1e-3) / 1e9

    # end to end through the host-buffer entry point (pinned host memory)
    bufs = run.host_buffers()
    for _ in range(2):
        run.step(host=bufs)
    torch.cuda.synchronize()
    barrier(dist)
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        run.step(host=bufs)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist)
    e2e_value = world * run.kv_bytes * e2e_steps / e2e_s / 1e9
    h2d = run.T * (w.q_dim + 2 * w.kv_dim) * 4 * w.n_layers
    d2h = run.T * w.q_dim * 4 * w.n_layers
    del bufs

    roofline = roofline_of(run, w, kern, args.steps, args.workload, args.kv_dtype,
                           tensor_flops_per_layer)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on a bounded sample of the same rows: on one thread, then
        # on every host core (same arithmetic, same bits)
        lens = [b + n for b, n in zip(run.base_len, run.n_q)]
        rows = oracle_sample(w, lens, args.cpu_budget, n_q=run.n_q)
        samples = run.histories_for(rows)
        dt1, nbytes, _ = time_oracle(samples, w, threads=1)
        dtn, _, cores = time_oracle(samples, w, threads=0)
        what = "%d of %d rows (%d keys, layer 0) of the same workload, C oracle, double accumulation" % (
            len(rows), len(lens), sum(lens[r] for r in rows))
        cpu = {"value": round(nbytes / dtn / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": "%s, %d threads, %.2f s" % (what, cores, dtn),
               "one_thread": {"value": round(nbytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": "%s, one thread, %.1f s" % (what, dt1)}}
        del samples

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f32 math, fp8 e4m3 K/V storage" if run.fp8 else
                  "f32 math, bf16 K/V storage" if run.bf16 else "f32"),
        "data": "synthetic (seeded N(0,1) K/V/Q, seeded length draws)",
        "config": {
            "workload": w.name,
            "M": w.M, "n_q_per_row": sorted(set(run.n_q))[:4], "n_heads": w.n_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "n_layers": w.n_layers,
            "block_size": w.block_size, "n_blocks": w.n_blocks,
            "kv_bytes_per_step": run.kv_bytes, "split_keys": pkv.pkv_get_split_keys(),
            # keys per decode unit on this pool (the library scales the split
            # to the same bytes on bf16 / fp8 pools)
            "decode_split_keys": min(65536, pkv.pkv_get_split_keys() * (4 if run.fp8 else 2 if run.bf16 else 1)),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "image_cache_mb": args.image_cache_mb,
            "l2": "no flush: each step reads %.2f GB of K/V, far above the 129 MB L2" % (run.kv_bytes / 1e9),
        },
        "rows_layers_per_s": round(world * run.T * w.n_layers / (ms_step * 1e-3), 1),
        "unique_kv_bytes_per_step": run.unique_kv_bytes,
        "unique_kv_gbs": round(world * run.unique_kv_bytes * args.steps / (ms_total * 1e-3) / 1e9, 2),
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "host_ms_per_step": round(host_s * 1e3 / args.steps, 4),
        "kernels_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in kern.items() if v[1]},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clk,
    }
    run.close()
    del run
    torch.cuda.empty_cache()

    # the other configurations, measured the same way after the headline one
    # (its 78.6 GB pool freed first): decode M = 64, chunked prefill,
    # shared-prefix forks
    if (not args.no_extra and args.workload == "continuous_batching_m256" and args.kv_dtype == "f32"
            and not args.split_keys and not args.image_cache_mb):
        extra = {}
        for name in EXTRA_WORKLOADS:
            try:
                extra[name] = measure_extra(name, args, rank)
            except Exception as exc:  # keep the headline line whatever happens here
                extra[name] = {"error": "%s: %s" % (type(exc).__name__, exc)}
        line["extra_workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the same workload's rows."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    w = get_workload(args.workload)
    lens = [int(p + n) for p, n in zip(w.past_len, w.n_q)]
    total_s = max(20.0, min(150.0, 6.0 * (args.steps + args.warmup)))
    per_step = total_s / (args.steps + args.warmup)
    rows = oracle_sample(w, lens, per_step, rng_seed=1, n_q=[int(x) for x in w.n_q], threads=0)
    rng = np.random.default_rng(w.seed)
    samples = []
    for r in rows:
        n, tk = int(w.n_q[r]), lens[r]
        samples.append((rng.standard_normal((n, w.q_dim)).astype(np.float32),
                        rng.standard_normal((tk, w.kv_dim)).astype(np.float32),
                        rng.standard_normal((tk, w.kv_dim)).astype(np.float32), n, tk))
    for _ in range(args.warmup):
        time_oracle(samples, w, threads=0)
    dts, nbytes, cores = [], 0.0, 1
    for _ in range(args.steps):
        dt, nbytes, cores = time_oracle(samples, w, threads=0)
        dts.append(dt)
    t = sum(dts)
    value = nbytes * args.steps / t / 1e9
    sample = "%d of %d rows (%d keys) per step, C oracle, double accumulation, %d threads" % (
        len(rows), len(lens), sum(lens[r] for r in rows), cores)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": w.name, "M": w.M, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size, "n_layers": w.n_layers},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", default="continuous_batching_m256")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only --workload (the default run also measures %s)" % ", ".join(EXTRA_WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time")
    ap.add_argument("--split-keys", type=int, default=0, help="keys per split-K unit (0: library default)")
    ap.add_argument("--kv-dtype", choices=["f32", "bf16", "fp8"], default="f32",
                    help="K/V pool storage (bf16 / fp8 e4m3: rows rounded on write, f32 math)")
    ap.add_argument("--image-cache-mb", type=int, default=0,
                    help="keep tensor-core operand images of unchanged pages across steps "
                         "(pkv_pool_set_image_cache), up to this many MiB; 0 = off")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
