"""QSA benchmark: prefill tokens/s at 128K context and decode us/step at 256K x 64.

One step = one pass of the whole QSA hot path over one batch of synthetic input:
  prefill (drift_prefill_128k): key compression, indexer scores + top-k_B
      selection, sparse GQA attention for all 131072 rows of one sequence;
  decode (decode_256k_x64): block selection + sparse attention for one new
      token in each of 64 sequences with a 262144-token cache.
Inputs are resident in HBM when the timed region starts.  `value` is prefill
tokens/s (all ranks); the decode step time is reported beside it.  `e2e`
repeats the same step through the public binding with host buffers: the step's
inputs are copied from pinned host memory and its outputs read back inside the
timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qsa|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QSA prefill tokens/s at 128K and decode µs/step at 256K ctx (1×B300)"
PREFILL = "drift_prefill_128k"
DECODE = "decode_256k_x64"
L2_FLUSH_BYTES = 256 << 20


def reduce_max_over_ranks(vals, world: int, device):
    """Element-wise max of per-rank timings over all ranks: the slowest rank sets
    the job's time.  With one rank the values come back unchanged."""
    import torch
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world: int, tokens_per_rank: int, prefill_ms: float) -> float:
    """Whole-job prefill throughput: every rank runs its own replica of the
    workload (weak scaling), timed by the slowest rank."""
    return world * tokens_per_rank / (prefill_ms * 1e-3)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# kernel named, at the prefill workload named, from one ncu capture of it:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum --clock-control none
#       -k "regex:sparse_attn_prefill" -c 1 python bench.py --decode-workload none
#       --multi-decode-workload none --no-extras --steps 1 --warmup 3 --no-cpu-baseline --no-e2e
# A kernel or workload not listed (or a kernel changed since the capture) reports null.
MEASURED_TRAFFIC = {("attn_prefill", "drift_prefill_128k"): 2054448384 + 544514048}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def tensor_peak_for(clk: dict, pk: dict) -> tuple[float, str]:
    """The bf16 tensor peak a kernel timed in these steps is held to: the burst
    figure while the sampled clocks showed no power cap, the sustained
    (power-capped) one when they did."""
    if "sw_power_cap" in (clk.get("reasons") or []):
        return pk["bf16_tflops_sustained"], "sustained"
    return pk["bf16_tflops"], "burst"


# ----------------------------------------------------------------------------- algorithmic work

def prefill_work(n: int, r: int, k_b: int, hq: int, hkv: int, d: int = 128, h_idx: int = 4) -> dict:
    """Exact algorithmic work of one QSA prefill of n tokens (one sequence)."""
    i = __import__("numpy").arange(n, dtype="int64")
    c = (i + 1) // r
    sel = c.clip(max=k_b)
    t = sel * r + (i + 1 - c * r)
    sum_c, sum_t = int(c.sum()), int(t.sum())
    return {
        "sum_c": sum_c, "sum_t": sum_t,
        "index_flops": 2 * h_idx * d * sum_c,
        "attn_flops": 4 * d * hq * sum_t,
        "attn_gather_bytes": sum_t * hkv * 2 * d * 2,
        "compress_bytes": n * d * 2 + (n // r) * d * 2,
    }


def decode_work(batch: int, cache_len: int, r: int, k_b: int, hq: int, hkv: int, d: int = 128,
                h_idx: int = 4) -> dict:
    c = cache_len // r
    t = min(c, k_b) * r + (cache_len - c * r)
    kbar_bytes = c * d * 2
    gather = t * hkv * 2 * d * 2
    small = h_idx * d * 2 + hq * d * 2 * 2 + k_b * 4  # new q_idx, q, out, idx
    return {"bytes": batch * (kbar_bytes + gather + small), "kbar_bytes": batch * kbar_bytes,
            "gather_bytes": batch * gather, "tokens": t}


def decode_multi_work(batch: int, cache_len: int, next_n: int, r: int, k_b: int, hq: int, hkv: int,
                      d: int = 128, h_idx: int = 4) -> dict:
    """One multi-token decode step: the k-bar scan once per sequence (up to the
    last row's visible blocks), a gather per row, and the rows' small tensors."""
    c_last = cache_len // r
    kbar_bytes = c_last * d * 2
    gather = 0
    for j in range(next_n):
        i = cache_len - next_n + j
        c = (i + 1) // r
        gather += (min(c, k_b) * r + (i + 1 - c * r)) * hkv * 2 * d * 2
    small = next_n * (h_idx * d * 2 + hq * d * 2 * 2 + k_b * 4)
    return {"bytes": batch * (kbar_bytes + gather + small), "kbar_bytes": batch * kbar_bytes,
            "gather_bytes": batch * gather}


def multi_decode_measure(qsa, spec, steps: int, warmup: int, dev, hbm_gbs: float) -> dict:
    """Times the multi-token decode step (the pages' decode mode: batch 4, next_n
    = 4): qsa_index_topk for all rows of each sequence, then
    qsa_sparse_attn_decode_multi.  CUDA events around each step, L2 flushed
    between steps outside the events; the median step is reported."""
    import torch
    from block_sparse_long_17_b300.workloads import make_decode
    wl = make_decode(spec, dev)
    cfg = qsa.Config(r=spec.r, k_tokens=spec.k_tokens, rope_dims=spec.rope_dims, rope_base=spec.rope_base)
    B, nn = spec.batch, spec.next_n
    q_pos = wl["cache_lens"] - nn
    idx = torch.empty((B, nn, cfg.k_b), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, nn), dtype=torch.int32, device=dev)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, B, nn, wl["n_blocks"]),), dtype=torch.uint8, device=dev)
    out = torch.empty_like(wl["q"])
    lse = torch.empty((B, nn, spec.hq), dtype=torch.float32, device=dev)
    wsa = torch.empty((qsa.qsa_sparse_attn_decode_multi_workspace(cfg, B, nn, spec.hq, spec.hkv),),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        qsa.qsa_index_topk(cfg, wl["q_idx"], wl["kbar"], q_pos, wl["n_blocks"], idx, cnt, ws)
        qsa.qsa_sparse_attn_decode_multi(cfg, wl["q"], wl["k"], wl["v"], wl["cache_lens"], idx, cnt, out, wsa, lse)

    for _ in range(max(warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(steps, 10)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    assert qsa.qsa_read_device_error() == 0
    us = statistics.median(ts) * 1e3
    wk = decode_multi_work(B, wl["cache_len"], nn, spec.r, spec.k_b, spec.hq, spec.hkv)
    achieved = wk["bytes"] / (us * 1e-6) / 1e9
    # Any dense decode of these rows reads the whole K/V cache at least once:
    # its HBM time is a lower bound on every dense kernel at this shape.
    kv_bytes = B * spec.hkv * wl["cache_len"] * spec.d * 2 * 2
    floor_us = kv_bytes / (hbm_gbs * 1e9) * 1e6
    return {"workload": spec.name, "batch": B, "next_n": nn, "ctx_tokens": wl["cache_len"],
            "us_per_step": us, "bytes_per_step": wk["bytes"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs},
            "dense_floor": {"kv_bytes": kv_bytes, "hbm_floor_us": floor_us, "speedup_qsa_vs_dense_floor": floor_us / us,
                            "note": "dense decode of the same rows cannot read less than the whole K/V cache once"}}


def _median_step_ms(step, steps: int, warmup: int, flush) -> float:
    import torch
    for _ in range(max(warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(steps, 10)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def chunked_prefill_measure(qsa, cfg, pspec, wl, pre, chunk: int, steps: int, warmup: int, dev, flush) -> dict:
    """The pages' chunked-prefill mode: the last `chunk` query rows of the
    sequence against the whole cached prefix (k-bar already compressed): index +
    top-k for the chunk's rows, then sparse attention for them."""
    import torch
    n = pspec.n
    lo = n - chunk
    q_idx = wl["q_idx"][:, lo:].contiguous()
    q = wl["q"][:, lo:].contiguous()
    q_pos = torch.full((1,), lo, dtype=torch.int64, device=dev)
    idx = torch.empty((1, chunk, cfg.k_b), dtype=torch.int32, device=dev)
    cnt = torch.empty((1, chunk), dtype=torch.int32, device=dev)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, 1, chunk, pre.n_blocks),), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)

    def step():
        qsa.qsa_index_topk(cfg, q_idx, pre.kbar, q_pos, pre.n_blocks, idx, cnt, ws)
        qsa.qsa_sparse_attn_prefill(cfg, q, wl["k"], wl["v"], q_pos, idx, cnt, out, None)

    ms = _median_step_ms(step, steps, warmup, flush)
    assert qsa.qsa_read_device_error() == 0
    return {"chunk_tokens": chunk, "prefix_tokens": lo, "ms_per_chunk": ms, "tokens_per_s": chunk / (ms * 1e-3)}


def attention_kernels_measure(qsa, cfg, wl, pre, steps: int, warmup: int, flush) -> dict:
    """Prefill attention alone, each kernel of the library on the same inputs
    and selection (the last prefill's): the tcgen05 kernel (TMA-staged blocks,
    TMEM accumulators) and the mma.sync one.  Median of CUDA-event timings, L2
    flushed between runs."""
    res = {}
    for impl in ("tcgen05", "mma_sync"):
        def step():
            qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], pre.q_pos, pre.idx, pre.count,
                                        pre.out, pre.lse, impl=impl)
        try:
            res[impl] = {"ms": _median_step_ms(step, steps, warmup, flush)}
        except qsa.QsaError as ex:
            res[impl] = {"unavailable": str(ex)}
    assert qsa.qsa_read_device_error() == 0
    return res


def index_sweep_measure(qsa, pk: dict, steps: int, warmup: int, dev, flush, with_1m_r2: bool = False) -> list:
    """qsa_index_topk alone (query rotation, scores, top-k_B) at micro-block
    sizes r in {2, 4, 8, 16} over the 32K, 128K and 1M prefill workloads' indexer
    inputs (K = 2048, 4 indexer heads), the form of the pages' indexer-latency
    panels.  Each line: median ms over the timed calls (L2 flushed between
    them) and the indexer flops (2 H 128 per visible block and row) against the
    bf16 tensor peaks.  r = 2 gives k_B = 1024, beyond the fused indexer's 512,
    so it runs the one-pass scan path (score rows stored, then selected); at 1M
    that takes seconds per call and is timed only on request."""
    import torch
    from block_sparse_long_17_b300.workloads import WORKLOADS, make_prefill
    out = []
    for name in ("needle_prefill_32k", "drift_prefill_128k", "needle_prefill_1m"):
        spec = WORKLOADS[name]
        wl = make_prefill(spec, dev, indexer_only=True)
        n = spec.n
        for r in (2, 4, 8, 16):
            if r == 2 and n > (1 << 17) and not with_1m_r2:
                out.append({"workload": name, "r": r, "skipped": "scan path at k_B = 1024: seconds per call at 1M"})
                continue
            cfg = qsa.Config(r=r, k_tokens=spec.k_tokens, rope_dims=spec.rope_dims, rope_base=spec.rope_base)
            nb = n // r
            kbar = torch.empty((1, nb, spec.d), dtype=torch.bfloat16, device=dev)
            qsa.qsa_compress_keys(cfg, wl["k_idx"], 0, nb, kbar)
            q_pos = torch.zeros((1,), dtype=torch.int64, device=dev)
            idx = torch.empty((1, n, cfg.k_b), dtype=torch.int32, device=dev)
            cnt = torch.empty((1, n), dtype=torch.int32, device=dev)
            ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, 1, n, nb),), dtype=torch.uint8, device=dev)

            def step():
                qsa.qsa_index_topk(cfg, wl["q_idx"], kbar, q_pos, nb, idx, cnt, ws)

            st = 1 if (r == 2 and n > (1 << 17)) else min(steps, 5)
            ms = _median_step_ms(step, st, min(warmup, 3) if st > 1 else 1, flush)
            fb = qsa.qsa_index_topk_fallback_rows(cfg, 1, n, nb, ws)
            i = __import__("numpy").arange(n, dtype="int64")
            flops = 2 * spec.h_idx * spec.d * int(((i + 1) // r).sum())
            tf = flops / (ms * 1e-3) / 1e12
            out.append({"workload": name, "r": r, "k_b": cfg.k_b, "ms": ms, "tflops": tf,
                        "frac_of_burst": tf / pk["bf16_tflops"], "frac_of_sustained": tf / pk["bf16_tflops_sustained"],
                        "path": "fused tcgen05" if cfg.k_b <= 512 else "scan (k_B > 512)", "fallback_rows": fb})
            del kbar, idx, cnt, ws
            torch.cuda.empty_cache()
        del wl
        torch.cuda.empty_cache()
    assert qsa.qsa_read_device_error() == 0
    return out


def dense_decode_measure(qsa, dspec, dwl, dq, steps: int, warmup: int, dev, flush, hbm_gbs: float,
                         qsa_decode_us: float) -> dict:
    """Dense GQA decode at the decode step's shape, for the pages' form of
    comparison: the same decode attention kernel with every block of every
    sequence selected (k_B >= c), i.e. attention over the whole cache.  Its HBM
    floor (the whole K/V cache read once) is reported beside it."""
    import torch
    B, L = dspec.batch, dwl["cache_len"]
    c = L // dspec.r
    cfg = qsa.Config(r=dspec.r, k_tokens=c * dspec.r, rope_dims=dspec.rope_dims, rope_base=dspec.rope_base)
    idx = torch.arange(c, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    cnt = torch.full((B,), c, dtype=torch.int32, device=dev)
    ws = torch.empty((qsa.qsa_sparse_attn_decode_workspace(cfg, B, dspec.hq, dspec.hkv),), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, dspec.hq, dspec.d), dtype=torch.bfloat16, device=dev)

    def step():
        qsa.qsa_sparse_attn_decode(cfg, dq, dwl["k"], dwl["v"], dwl["cache_lens"], idx, cnt, out, ws, None)

    ms = _median_step_ms(step, steps, warmup, flush)
    assert qsa.qsa_read_device_error() == 0
    kv_bytes = B * dspec.hkv * L * dspec.d * 2 * 2
    floor_us = kv_bytes / (hbm_gbs * 1e9) * 1e6
    return {"us_per_step": ms * 1e3, "kv_bytes": kv_bytes, "hbm_floor_us": floor_us,
            "qsa_decode_us": qsa_decode_us, "speedup_qsa_vs_dense": ms * 1e3 / qsa_decode_us,
            "speedup_qsa_vs_dense_floor": floor_us / qsa_decode_us,
            "note": "dense = the decode attention kernel with every block selected; its own numbers, not the pages'"}


def dense_prefill_measure(wl, qsa_prefill_ms: float, steps: int, warmup: int, flush) -> dict:
    """Dense causal GQA over the same prefill (all 131072 rows, every earlier
    token), for the pages' form of comparison.  This arm is a library kernel
    (PyTorch scaled_dot_product_attention restricted to its cuDNN / flash
    backends, never the materialising one), not part of this library."""
    import torch
    try:
        from torch.nn.attention import SDPBackend, sdpa_kernel
        q = wl["q"].transpose(1, 2).contiguous()  # [B, Hq, n, d]
        k, v = wl["k"][:, :, :q.shape[2]], wl["v"][:, :, :q.shape[2]]

        def step():
            with sdpa_kernel([SDPBackend.CUDNN_ATTENTION, SDPBackend.FLASH_ATTENTION]):
                torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)

        ms = _median_step_ms(step, min(steps, 5), warmup, flush)
    except Exception as ex:  # PyTorch offers no fused dense backend here: report it instead
        return {"unavailable": str(ex).split("\n")[0][:160]}
    n, hq, d = q.shape[2], q.shape[1], q.shape[3]
    flops = 4 * hq * d * n * (n + 1) / 2
    return {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "qsa_prefill_ms": qsa_prefill_ms,
            "speedup_qsa_vs_dense": ms / qsa_prefill_ms,
            "note": "dense = library SDPA (cuDNN or flash backend), causal, GQA; QSA = compress + index + "
                    "sparse attention of this library"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.proc = None
        self.bus_id = bus_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def bus_id_of(dev) -> str | None:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ----------------------------------------------------------------------------- CPU oracle timing

def blas_threads() -> int:
    """Threads numpy's BLAS uses (the oracle's only multi-threaded part)."""
    try:
        from threadpoolctl import threadpool_info
        return max([p.get("num_threads", 1) for p in threadpool_info()] + [1])
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return os.cpu_count() or 1

def oracle_timing(pre_spec, dec_spec, rows_per_step: int, steps: int, seed: int = 0) -> dict:
    """Times the CPU oracle, as it stands, on a bounded sample of both workloads.

    Prefill: key compression of the whole sequence plus `rows_per_step` query rows
    at stratified positions (indexer scores, selection, attention).  The rows'
    time is extrapolated to all n rows by the work model of the path: a row i
    costs c_i * 1024 (indexer flops) + |T_i| * 8192 (attention flops per
    attended token over 16 heads), so the full prefill takes
    (sample time / sample work) x total work.  Decode: one sequence's step,
    times the batch.
    """
    import numpy as np

    from block_sparse_long_17_b300.workloads import make_decode, make_prefill
    from oracle import qsa_oracle as O

    n, r, k_b = pre_spec.n, pre_spec.r, pre_spec.k_b
    i_all = np.arange(n, dtype=np.int64)
    c_all = (i_all + 1) // r
    t_all = np.minimum(c_all, k_b) * r + (i_all + 1 - c_all * r)
    work = c_all * 1024.0 + t_all * 8192.0
    wl = make_prefill(pre_spec, "cpu")
    f32 = lambda t: t.float().numpy()
    q_idx, k_idx, q, k, v = f32(wl["q_idx"][0]), wl["k_idx"][0].double().numpy(), f32(wl["q"][0]), f32(wl["k"][0]), f32(wl["v"][0])
    dw = make_decode(dec_spec, "cpu", batch=1)
    rng = np.random.default_rng(seed)
    pre_times, dec_times = [], []
    for s in range(steps):
        t0 = time.perf_counter()
        kbar = O.compress_keys(k_idx, r, rope_dims=pre_spec.rope_dims, rope_base=pre_spec.rope_base)
        t1 = time.perf_counter()
        strata = (np.arange(rows_per_step) + rng.random(rows_per_step)) / rows_per_step
        rows = sorted({int(x) for x in (strata * n).astype(np.int64)})
        O.prefill_rows(q_idx, None, q, k, v, rows, r=r, k_tokens=pre_spec.k_tokens, kbar=kbar)
        t2 = time.perf_counter()
        pre_times.append((t1 - t0) + (t2 - t1) * float(work.sum()) / float(work[rows].sum()))
        t3 = time.perf_counter()
        O.decode_rows(dw["q_idx"][0, 0].double().numpy(), dw["q"][0, 0].double().numpy(),
                      dw["kbar"][0].float().numpy(), dw["k"][0].float().numpy(), dw["v"][0].float().numpy(),
                      dw["cache_len"], r=dec_spec.r, k_tokens=dec_spec.k_tokens)
        dec_times.append((time.perf_counter() - t3) * dec_spec.batch)
    threads = blas_threads()
    return {"prefill_s": statistics.mean(pre_times), "decode_s": statistics.mean(dec_times),
            "cores": threads, "host_cpus": os.cpu_count(),
            "sample": (f"per step: compress all {n // r} blocks + {rows_per_step} of {n} prefill rows "
                       f"(stratified), extrapolated by the work model c_i*1024 + |T_i|*8192 per row; "
                       f"decode: 1 of {dec_spec.batch} sequences x {dec_spec.batch}; cores = threads of "
                       f"numpy's BLAS, the oracle's only threaded part")}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20; the CPU reference arm: 5)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["qsa", "reference"], default="qsa")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--prefill-workload", default=PREFILL,
                    help="prefill workload name (smaller ones serve profiling runs)")
    ap.add_argument("--decode-workload", default=DECODE, help="decode workload name, or 'none'")
    ap.add_argument("--multi-decode-workload", default="decode_1m_b4_next4",
                    help="multi-token decode workload timed beside the main step, or 'none'")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the chunked-prefill and dense-decode lines timed after the main step")
    ap.add_argument("--no-index-sweep", action="store_true",
                    help="skip the indexer timing over micro-block sizes and context lengths")
    ap.add_argument("--index-sweep-1m-r2", action="store_true",
                    help="also time r = 2 at 1M in the indexer sweep (seconds per call)")
    ap.add_argument("--attention-kernels-only", action="store_true",
                    help="select the prefill workload's blocks once, then time only the two prefill "
                         "attention kernels (tcgen05, mma.sync) on them, and print that line")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 5 if args.impl == "reference" else 20

    import torch
    from block_sparse_long_17_b300.workloads import WORKLOADS

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    pspec = WORKLOADS[args.prefill_workload]
    dspec = WORKLOADS[DECODE if args.decode_workload == "none" else args.decode_workload]
    do_decode = args.decode_workload != "none"
    pk = peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        steps = max(args.steps, 1)
        ot = oracle_timing(pspec, dspec, rows_per_step=16, steps=steps)
        val = pspec.n / ot["prefill_s"]
        line = {"metric": METRIC, "value": val, "unit": "tokens/s", "impl": "reference",
                "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
                "ms_per_step": (ot["prefill_s"] + ot["decode_s"]) * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "decode_us_per_step": ot["decode_s"] * 1e6,
                "config": {"workload": f"{PREFILL} + {DECODE}", "prefill_tokens": pspec.n,
                           "decode_batch": dspec.batch, "decode_ctx": dspec.ctx, "K": pspec.k_tokens,
                           "r": pspec.r},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": ot["cores"], "kind": "oracle",
                                 "host_cpus": ot["host_cpus"], "sample": ot["sample"]},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    from block_sparse_long_17_b300 import qsa
    from block_sparse_long_17_b300.workloads import make_decode, make_prefill

    qsa.load_library()  # raises if the CUDA library is missing: no fallback path exists
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)

    if args.attention_kernels_only:
        cfg = qsa.Config(r=pspec.r, k_tokens=pspec.k_tokens, rope_dims=pspec.rope_dims, rope_base=pspec.rope_base)
        wl = make_prefill(pspec, dev)
        pre = qsa.QsaPrefill(cfg, 1, pspec.n, pspec.hq, pspec.hkv, device=dev)
        pre(wl["q_idx"], wl["k_idx"], wl["q"], wl["k"], wl["v"])
        for impl in ("tcgen05", "mma_sync"):  # one untimed call each first (the profiling target)
            qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], pre.q_pos, pre.idx, pre.count, pre.out,
                                        pre.lse, impl=impl)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        kern = attention_kernels_measure(qsa, cfg, wl, pre, args.steps, args.warmup, flush)
        pw = prefill_work(pspec.n, pspec.r, pspec.k_b, pspec.hq, pspec.hkv)
        for v in kern.values():
            if "ms" in v:
                v["tflops"] = pw["attn_flops"] / (v["ms"] * 1e-3) / 1e12
                v["gathered_tb_s"] = pw["attn_gather_bytes"] / (v["ms"] * 1e-3) / 1e12
        if rank == 0:
            print(json.dumps({"workload": pspec.name, "attention_kernels": kern}), flush=True)
        return

    # The multi-token decode step is a separate workload, timed first on a clean
    # device and its buffers freed before the main step's are drawn.
    decode_multi = None
    if args.multi_decode_workload != "none":
        decode_multi = multi_decode_measure(qsa, WORKLOADS[args.multi_decode_workload], args.steps, args.warmup,
                                            dev, pk["hbm_gbs"])
        torch.cuda.empty_cache()

    cfg = qsa.Config(r=pspec.r, k_tokens=pspec.k_tokens, rope_dims=pspec.rope_dims, rope_base=pspec.rope_base)
    wl = make_prefill(pspec, dev)
    pre = qsa.QsaPrefill(cfg, 1, pspec.n, pspec.hq, pspec.hkv, device=dev)
    dcfg = qsa.Config(r=dspec.r, k_tokens=dspec.k_tokens, rope_dims=dspec.rope_dims, rope_base=dspec.rope_base)
    if do_decode:
        dwl = make_decode(dspec, dev)
        dec = qsa.QsaDecode(dcfg, dspec.batch, dwl["n_blocks"], dspec.hq, dspec.hkv, device=dev)
        dq = dwl["q"][:, 0].contiguous()
        dq_pos = dwl["cache_lens"] - 1  # the new token's position: decode state, like the caches
    else:
        dwl = {"cache_len": dspec.cache_len}
        dec = dq = dq_pos = None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    names = ["compress", "index_prefill", "attn_prefill", "index_decode", "attn_decode"]

    def step(evs):
        evs[0].record(stream)
        qsa.qsa_compress_keys(cfg, wl["k_idx"], 0, pre.n_blocks, pre.kbar)
        evs[1].record(stream)
        qsa.qsa_index_topk(cfg, wl["q_idx"], pre.kbar, pre.q_pos, pre.n_blocks, pre.idx, pre.count, pre.ws)
        evs[2].record(stream)
        qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], pre.q_pos, pre.idx, pre.count,
                                    pre.out, pre.lse)
        evs[3].record(stream)
        if do_decode:
            qsa.qsa_index_topk(dcfg, dwl["q_idx"], dwl["kbar"], dq_pos, dwl["n_blocks"], dec.idx, dec.count,
                               dec.ws_idx)
        evs[4].record(stream)
        if do_decode:
            qsa.qsa_sparse_attn_decode(dcfg, dq, dwl["k"], dwl["v"], dwl["cache_lens"],
                                       dec.idx.view(dspec.batch, -1), dec.count.view(dspec.batch), dec.out,
                                       dec.ws_attn, dec.lse)
        evs[5].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for _ in range(args.warmup):
        flush.zero_()
        step(mk())
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0

    clocks = ClockSampler(bus_id_of(dev))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = qsa.qsa_launch_count()
    all_evs = []
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the step's events
        evs = mk()
        step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = (qsa.qsa_launch_count() - launches0) // args.steps
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()

    parts = {nm: [] for nm in names}
    for evs in all_evs:
        for j, nm in enumerate(names):
            parts[nm].append(evs[j].elapsed_time(evs[j + 1]))
    mean = {nm: statistics.mean(v) for nm, v in parts.items()}
    prefill_ms = mean["compress"] + mean["index_prefill"] + mean["attn_prefill"]
    prefill_each = [parts["compress"][j] + parts["index_prefill"][j] + parts["attn_prefill"][j]
                    for j in range(len(all_evs))]
    decode_each = [parts["index_decode"][j] + parts["attn_decode"][j] for j in range(len(all_evs))]
    decode_ms = mean["index_decode"] + mean["attn_decode"]
    step_ms = prefill_ms + decode_ms
    prefill_ms, decode_ms, step_ms = reduce_max_over_ranks([prefill_ms, decode_ms, step_ms], world, dev)
    value = job_tokens_per_s(world, pspec.n, prefill_ms)

    # Roofline of each part (algorithmic work / measured mean duration).
    tensor_peak, tensor_peak_kind = tensor_peak_for(clk, pk)
    pw = prefill_work(pspec.n, pspec.r, pspec.k_b, pspec.hq, pspec.hkv)
    dwk = decode_work(dspec.batch, dwl["cache_len"], dspec.r, dspec.k_b, dspec.hq, dspec.hkv)
    hbm = pk["hbm_gbs"]
    roofs = {
        "compress": {"bound": "hbm", "achieved": pw["compress_bytes"] / (mean["compress"] * 1e-3) / 1e9,
                     "peak": hbm, "unit": "GB/s"},
        "index_prefill": {"bound": "tensor", "achieved": pw["index_flops"] / (mean["index_prefill"] * 1e-3) / 1e12,
                          "peak": tensor_peak, "peak_kind": tensor_peak_kind, "unit": "TFLOP/s"},
        # Sparse attention is a bf16 contraction over gathered K/V: graded on the
        # tensor peak, with its measured DRAM traffic against the HBM peak beside
        # it.  Neither is its limit: the gathers come from L2 (ncu: 99% hit rate),
        # at about 16 flop per gathered byte.
        "attn_prefill": {"bound": "tensor", "achieved": pw["attn_flops"] / (mean["attn_prefill"] * 1e-3) / 1e12,
                         "peak": tensor_peak, "peak_kind": tensor_peak_kind, "unit": "TFLOP/s",
                         "gathered_bytes": pw["attn_gather_bytes"],
                         "gathered_tb_s": pw["attn_gather_bytes"] / (mean["attn_prefill"] * 1e-3) / 1e12},
    }
    if do_decode:
        roofs["decode"] = {"bound": "hbm", "achieved": dwk["bytes"] / (decode_ms * 1e-3) / 1e9, "peak": hbm,
                           "unit": "GB/s"}
    for v in roofs.values():
        v["frac"] = v["achieved"] / v["peak"]
    for nm in ("index_prefill", "attn_prefill"):
        roofs[nm]["frac_of_burst"] = roofs[nm]["achieved"] / pk["bf16_tflops"]
        roofs[nm]["frac_of_sustained"] = roofs[nm]["achieved"] / pk["bf16_tflops_sustained"]
    attn_traffic = MEASURED_TRAFFIC.get(("attn_prefill", pspec.name))
    roofs["attn_prefill"]["traffic"] = attn_traffic
    roofs["attn_prefill"]["frac_of_hbm"] = (attn_traffic / (mean["attn_prefill"] * 1e-3) / 1e9 / hbm
                                            if attn_traffic else None)
    dominant = max(["compress", "index_prefill", "attn_prefill"], key=lambda nm: mean[nm])
    roof = dict(roofs[dominant])
    roof["kernel"] = dominant
    roof["traffic"] = MEASURED_TRAFFIC.get((dominant, pspec.name))

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "decode_us_per_step": decode_ms * 1e3,
        "prefill_ms": prefill_ms,
        # medians over the timed steps (the value above uses the means)
        "prefill_ms_median": statistics.median(prefill_each),
        "decode_us_median": statistics.median(decode_each) * 1e3 if do_decode else None,
        "parts_ms": mean,
        "config": {"workload": f"{pspec.name} + {dspec.name if do_decode else 'no decode'}",
                   "prefill_tokens": pspec.n, "prefill_batch": 1,
                   "decode_batch": dspec.batch, "decode_ctx": dspec.ctx, "K": pspec.k_tokens, "r": pspec.r,
                   "Hq": pspec.hq, "Hkv": pspec.hkv, "H_idx": pspec.h_idx, "d": pspec.d,
                   "l2": "256 MiB buffer written between steps, outside the timed events",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "rooflines": roofs, "peaks_source": pk["source"],
        "gpu_launches": int(launches), "clocks": clk, "wall_s_timed": wall,
        # rows of the last prefill that the indexer's exact full-row fallback selected
        "index_fallback_rows": pre.fallback_rows(stream),
    }

    if not do_decode:
        line["decode_us_per_step"] = None
    if decode_multi is not None:
        line["decode_multi"] = decode_multi
    if not args.no_extras:
        kern = attention_kernels_measure(qsa, cfg, wl, pre, args.steps, args.warmup, flush)
        for impl, v in kern.items():
            if "ms" in v:
                v["tflops"] = pw["attn_flops"] / (v["ms"] * 1e-3) / 1e12
                v["frac_of_burst"] = v["tflops"] / pk["bf16_tflops"]
                v["gathered_tb_s"] = pw["attn_gather_bytes"] / (v["ms"] * 1e-3) / 1e12
        line["rooflines"]["attn_prefill"]["kernels"] = kern
        chunk = min(16384, pspec.n)
        line["chunked_prefill"] = chunked_prefill_measure(qsa, cfg, pspec, wl, pre, chunk, args.steps, args.warmup,
                                                          dev, flush)
        if do_decode:
            line["dense_decode"] = dense_decode_measure(qsa, dspec, dwl, dq, args.steps, args.warmup, dev, flush,
                                                        hbm, decode_ms * 1e3)
        line["dense_prefill"] = dense_prefill_measure(wl, prefill_ms, args.steps, args.warmup, flush)
    if not args.no_extras and not args.no_index_sweep:
        line["index_sweep"] = index_sweep_measure(qsa, pk, args.steps, args.warmup, dev, flush,
                                                  with_1m_r2=args.index_sweep_1m_r2)
    if not args.no_e2e and rank == 0 and do_decode:
        line["e2e"] = e2e_measure(qsa, cfg, dcfg, wl, dwl, pre, dec, dspec, args, stream, dev)
    if not args.no_cpu_baseline and rank == 0 and do_decode:
        ot = oracle_timing(pspec, dspec, rows_per_step=64, steps=1)
        line["cpu_baseline"] = {"value": pspec.n / ot["prefill_s"], "unit": "tokens/s", "cores": ot["cores"],
                                "kind": "oracle", "sample": ot["sample"], "host_cpus": ot["host_cpus"],
                                "decode_us_per_step": ot["decode_s"] * 1e6}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e_chunk_bounds(n: int, wave: int, r: int) -> list:
    """Row bounds of the end-to-end prefill's chunks.  `wave`: rows of one wave of
    the indexer (qsa_index_rows_per_wave).  Chunks of 1K, 2K and 4K rows and one
    wave first (each chunk's copy-in fits inside the compute of the chunk before
    it, so little of the host-to-device copy is exposed), then chunks of two
    waves (whole waves for the indexer), then one wave and a quarter wave (the
    copy-out after the last kernel stays short).  Any leftover rows form one
    chunk after the first four.  Bounds are multiples of r except n."""
    q = lambda x: max(r, x // r * r)
    head = [q(x) for x in (1024, 2048, 4096, wave)]
    tail = [q(wave), q(wave // 4)]
    mid = q(2 * wave)
    if sum(head) + sum(tail) >= n:  # short sequences: chunks of one wave
        return list(range(0, n, q(wave))) + [n]
    b = [0]
    for x in head:
        b.append(b[-1] + x)
    k = (n - b[-1] - sum(tail)) // mid
    rem = n - b[-1] - sum(tail) - k * mid
    if rem > 0:
        b.append(b[-1] + rem)
    b += [b[-1] + mid * (j + 1) for j in range(k)]
    for x in tail:
        b.append(b[-1] + x)
    return b


def e2e_measure(qsa, cfg, dcfg, wl, dwl, pre, dec, dspec, args, stream, dev) -> dict:
    """The same step through the binding with host buffers: H2D of the step's
    inputs from pinned memory and D2H of its outputs, all inside the timed
    region.  The prefill runs as chunked prefill (the pages' mode) over the
    chunks of e2e_chunk_bounds: one stream copies chunk i in (the indexer's
    inputs first), one computes it (compress its blocks and select its rows as
    soon as those are in, attend its rows against the prefix once its q, K and
    V are), one copies its output back, so that the copies of one chunk
    overlap the kernels of another.  The decode step runs first on the compute stream, while the
    first chunk's inputs come in."""
    import torch
    host_in = {k: wl[k].cpu().pin_memory() for k in ("q_idx", "k_idx", "q", "k", "v")}
    dev_in = {k: torch.empty_like(wl[k]) for k in host_in}
    dq_h = dwl["q"][:, 0].contiguous().cpu().pin_memory()
    dqi_h = dwl["q_idx"].cpu().pin_memory()
    dq_d, dqi_d = torch.empty_like(dq_h, device=dev), torch.empty_like(dqi_h, device=dev)
    dq_pos = dwl["cache_lens"] - 1  # decode state (positions), device-resident like the caches
    out_h = torch.empty(pre.out.shape, dtype=pre.out.dtype).pin_memory()
    dout_h = torch.empty(dec.out.shape, dtype=dec.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + dq_h.numel() * 2 + dqi_h.numel() * 2
    d2h = out_h.numel() * 2 + dout_h.numel() * 2
    n, r, hkv = wl["q"].shape[1], cfg.r, wl["k"].shape[1]
    bounds = e2e_chunk_bounds(n, qsa.qsa_index_rows_per_wave(cfg), r)
    chunks = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    qpos = [torch.full((1,), lo, dtype=torch.int64, device=dev) for lo, _ in chunks]
    ws_c = torch.empty((qsa.qsa_index_topk_workspace(cfg, 1, max(b - a for a, b in chunks), pre.n_blocks),),
                       dtype=torch.uint8, device=dev)
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    ref = pre.out.clone()  # the one-call device step's output, for the check below

    def one():
        go = torch.cuda.Event()
        go.record(main)
        for s in (s_in, s_cmp, s_out):
            s.wait_event(go)
        with torch.cuda.stream(s_in):
            dq_d.copy_(dq_h, non_blocking=True)
            dqi_d.copy_(dqi_h, non_blocking=True)
            dec_in = torch.cuda.Event()
            dec_in.record(s_in)
        # The decode step needs none of the prefill: it runs first, while the
        # first chunk's inputs are still coming in.
        s_cmp.wait_event(dec_in)
        qsa.qsa_index_topk(dcfg, dqi_d, dwl["kbar"], dq_pos, dwl["n_blocks"], dec.idx, dec.count, dec.ws_idx,
                           stream=s_cmp)
        qsa.qsa_sparse_attn_decode(dcfg, dq_d, dwl["k"], dwl["v"], dwl["cache_lens"], dec.idx.view(dspec.batch, -1),
                                   dec.count.view(dspec.batch), dec.out, dec.ws_attn, dec.lse, stream=s_cmp)
        done = torch.cuda.Event()
        done.record(s_cmp)
        s_out.wait_event(done)
        with torch.cuda.stream(s_out):
            dout_h.copy_(dec.out, non_blocking=True)
        for i, (lo, hi) in enumerate(chunks):
            # The indexer's inputs first, on their own event, so that the
            # chunk's selection runs while its q, K and V rows (80% of its
            # bytes) are still coming in; the attention waits for all of them.
            with torch.cuda.stream(s_in):
                for key in ("k_idx", "q_idx"):
                    dev_in[key][:, lo:hi].copy_(host_in[key][:, lo:hi], non_blocking=True)
                idx_ready = torch.cuda.Event()
                idx_ready.record(s_in)
                dev_in["q"][:, lo:hi].copy_(host_in["q"][:, lo:hi], non_blocking=True)
                for key in ("k", "v"):
                    for g in range(hkv):
                        dev_in[key][0, g, lo:hi].copy_(host_in[key][0, g, lo:hi], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            s_cmp.wait_event(idx_ready)
            b0, b1 = lo // r, hi // r
            qsa.qsa_compress_keys(cfg, dev_in["k_idx"], b0, b1 - b0, pre.kbar, stream=s_cmp)
            qsa.qsa_index_topk(cfg, dev_in["q_idx"][:, lo:hi], pre.kbar, qpos[i], b1, pre.idx[:, lo:hi],
                               pre.count[:, lo:hi], ws_c, stream=s_cmp)
            s_cmp.wait_event(ready)
            qsa.qsa_sparse_attn_prefill(cfg, dev_in["q"][:, lo:hi], dev_in["k"], dev_in["v"], qpos[i],
                                        pre.idx[:, lo:hi], pre.count[:, lo:hi], pre.out[:, lo:hi],
                                        pre.lse[:, lo:hi], stream=s_cmp)
            done = torch.cuda.Event()
            done.record(s_cmp)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                out_h[:, lo:hi].copy_(pre.out[:, lo:hi], non_blocking=True)
        for s in (s_in, s_cmp, s_out):
            fin = torch.cuda.Event()
            fin.record(s)
            main.wait_event(fin)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k = max(1, args.steps)  # as many steps as the device-timed value
    e0.record(main)
    for _ in range(k):
        one()
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / k
    # The chunked pipeline computes the same rows as the one-call prefill.
    same = bool(torch.equal(out_h.to(dev), ref))
    return {"value": n / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "chunk_rows": [b - a for a, b in chunks], "output_matches_device_step": same,
            "steps": k,
            "note": "tokens/s of the prefill sequence over the whole step incl. copies and decode; chunked "
                    "prefill with copies on their own streams; the decode step's state (16 GiB K/V cache and "
                    "compressed-key cache) stays device-resident, only its new-token queries and outputs cross"}


if __name__ == "__main__":
    main()
