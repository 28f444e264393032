"""Seeded synthetic workloads for QSA prefill and decode.

This module only draws inputs.  It holds none of the attention arithmetic, so
the CUDA library and the CPU oracle can both be fed from it.

Recipe (the pages publish no data; every workload is synthetic):
  * One ``torch.Generator`` per workload, seeded with the workload seed, draws
    the tensors in a fixed order: q_idx, k_idx (or the compressed-key cache
    for decode), q, k, v.  Each is drawn as fp32 N(0, 1) and cast to bf16
    (round to nearest even).  Large tensors are drawn on the target device.
  * Needles (planted blocks): a numpy ``Generator(seed + 1000)`` picks, for
    needle j, a query row i_j uniform in [r*k_B, n), a block b_j uniform in
    [0, floor((i_j+1)/r)), and sets the r indexer keys of that block to
    q_idx[i_j, head 0] + 0.1 * N(0, 1).  Attention keys stay N(0, 1).
  * Drift: indexer keys and attention keys get an additive AR(1) process per
    dim, a_t = 0.99 a_{t-1} + sqrt(1 - 0.99^2) eps_t with a_0 ~ N(0, 1)
    (stationary, unit variance), drawn in fp64 by a numpy Generator(seed + 2000).
Layouts: q_idx [B, n, H_idx, d]; k_idx [B, n, d]; q [B, n, Hq, d];
k, v [B, Hkv, L, d]; decode compressed-key cache [B, N_b, d].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

__all__ = ["PrefillSpec", "DecodeSpec", "WORKLOADS", "make_prefill", "make_decode"]


@dataclass(frozen=True)
class PrefillSpec:
    name: str
    n: int                      # tokens per sequence
    k_tokens: int               # K; k_B = ceil(K / r)
    seed: int
    batch: int = 1
    r: int = 4
    h_idx: int = 4
    d: int = 128
    rope_dims: int = 64
    rope_base: float = 10000.0
    hq: int = 16
    hkv: int = 2
    needles: int = 0
    drift: bool = False

    @property
    def k_b(self) -> int:
        return -(-self.k_tokens // self.r)


@dataclass(frozen=True)
class DecodeSpec:
    name: str
    batch: int                  # independent sequences
    ctx: int                    # cached tokens before the new one
    k_tokens: int
    seed: int
    r: int = 4
    h_idx: int = 4
    d: int = 128
    rope_dims: int = 64
    rope_base: float = 10000.0
    hq: int = 16
    hkv: int = 2
    extra_cap: int = 4          # spare cache slots past the new token
    next_n: int = 1             # new tokens per step (the token plus its draft tokens)

    @property
    def k_b(self) -> int:
        return -(-self.k_tokens // self.r)

    @property
    def cache_len(self) -> int:  # includes the new tokens
        return self.ctx + self.next_n

    @property
    def n_blocks(self) -> int:   # compressed blocks the new token can score
        return self.cache_len // self.r

    @property
    def l_cap(self) -> int:
        return self.cache_len + self.extra_cap


WORKLOADS = {
    "tiny_prefill_2k": PrefillSpec("tiny_prefill_2k", n=2048, k_tokens=512, seed=0),
    "needle_prefill_32k": PrefillSpec("needle_prefill_32k", n=32768, k_tokens=2048, seed=1, needles=64),
    "drift_prefill_128k": PrefillSpec("drift_prefill_128k", n=131072, k_tokens=2048, seed=2, drift=True),
    "decode_256k_x64": DecodeSpec("decode_256k_x64", batch=64, ctx=262144, k_tokens=2048, seed=3),
    "needle_prefill_1m": PrefillSpec("needle_prefill_1m", n=1048576, k_tokens=2048, seed=4, needles=256),
    # A smaller decode step of the same shape family (a few GB on the device),
    # for profiling captures.
    "decode_64k_x64": DecodeSpec("decode_64k_x64", batch=64, ctx=65536, k_tokens=2048, seed=5),
    # Multi-token decode as timed in the pages' decode panels: batch 4, next_n = 4, 1M context.
    "decode_1m_b4_next4": DecodeSpec("decode_1m_b4_next4", batch=4, ctx=1048576 - 4, k_tokens=2048, seed=6, next_n=4),
}


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _ar1_drift(n: int, width: int, rng: np.random.Generator, rho: float = 0.99) -> np.ndarray:
    """Stationary unit-variance AR(1) paths, [n, width] fp64."""
    from scipy.signal import lfilter
    eps = rng.standard_normal((n, width))
    eps[0] = rng.standard_normal(width) / np.sqrt(1.0 - rho * rho)  # a_0 ~ N(0,1) after scaling
    return lfilter([np.sqrt(1.0 - rho * rho)], [1.0, -rho], eps, axis=0)


def make_prefill(spec: PrefillSpec, device="cpu", *, n: int | None = None, indexer_only: bool = False) -> dict:
    """Draw one prefill workload.  `n` overrides the sequence length (smaller test cases).
    indexer_only: draw only q_idx and k_idx (the first two draws, so their values
    are those of the full workload); q, k, v are None."""
    n = spec.n if n is None else n
    B, d = spec.batch, spec.d
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    q_idx = _randn_bf16((B, n, spec.h_idx, d), gen, device)
    k_idx = _randn_bf16((B, n, d), gen, device)
    q = k = v = None
    if not indexer_only:
        q = _randn_bf16((B, n, spec.hq, d), gen, device)
        k = _randn_bf16((B, spec.hkv, n, d), gen, device)
        v = _randn_bf16((B, spec.hkv, n, d), gen, device)
    needles = []
    if spec.needles:
        rng = np.random.default_rng(spec.seed + 1000)
        lo = spec.r * spec.k_b
        for _ in range(spec.needles):
            bb = int(rng.integers(0, B))
            i = int(rng.integers(min(lo, n - 1), n))
            blk = int(rng.integers(0, max(1, (i + 1) // spec.r)))
            noise = torch.from_numpy(0.1 * rng.standard_normal((spec.r, d)).astype(np.float32))
            base = q_idx[bb, i, 0].float().cpu()
            k_idx[bb, blk * spec.r:(blk + 1) * spec.r] = (base[None] + noise).to(torch.bfloat16).to(device)
            needles.append((bb, i, blk))
    if spec.drift:
        rng = np.random.default_rng(spec.seed + 2000)
        for bb in range(B):
            a_idx = _ar1_drift(n, d, rng)
            k_idx[bb] = (k_idx[bb].float() + torch.from_numpy(a_idx).float().to(device)).to(torch.bfloat16)
            if indexer_only:
                continue
            for g in range(spec.hkv):
                a_k = _ar1_drift(n, d, rng)
                k[bb, g] = (k[bb, g].float() + torch.from_numpy(a_k).float().to(device)).to(torch.bfloat16)
    return {"spec": spec, "n": n, "q_idx": q_idx, "k_idx": k_idx, "q": q, "k": k, "v": v,
            "needles": needles}


def make_decode(spec: DecodeSpec, device="cpu", *, batch: int | None = None, ctx: int | None = None) -> dict:
    """Draw one decode step: new-token queries, compressed-key cache and KV cache.

    The compressed-key cache is drawn directly (already pooled and rotated), as
    N(0, 1) bf16, for the n_blocks blocks the last new token can score.  The KV
    cache holds cache_len = ctx + next_n valid tokens (the last next_n are the
    new tokens, queried together).
    """
    B = spec.batch if batch is None else batch
    ctx = spec.ctx if ctx is None else ctx
    nn = spec.next_n
    cache_len = ctx + nn
    n_blocks = cache_len // spec.r
    l_cap = cache_len + spec.extra_cap
    d = spec.d
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    q_idx = _randn_bf16((B, nn, spec.h_idx, d), gen, device)
    kbar = _randn_bf16((B, n_blocks, d), gen, device)
    q = _randn_bf16((B, nn, spec.hq, d), gen, device)
    k = torch.empty((B, spec.hkv, l_cap, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((B, spec.hkv, l_cap, d), dtype=torch.bfloat16, device=device)
    for bb in range(B):  # per sequence, to bound the fp32 temporaries
        k[bb] = _randn_bf16((spec.hkv, l_cap, d), gen, device)
    for bb in range(B):
        v[bb] = _randn_bf16((spec.hkv, l_cap, d), gen, device)
    cache_lens = torch.full((B,), cache_len, dtype=torch.int64, device=device)
    return {"spec": spec, "batch": B, "ctx": ctx, "cache_len": cache_len, "n_blocks": n_blocks,
            "l_cap": l_cap, "q_idx": q_idx, "kbar": kbar, "q": q, "k": k, "v": v,
            "cache_lens": cache_lens}
