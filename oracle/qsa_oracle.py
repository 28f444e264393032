"""CPU oracle for Qwen Sparse Attention (QSA) -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, fp64 statement of what the QSA hot path
computes.  It exists to check the CUDA library, never to stand in for it:
only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path and imports
nothing from the product package.

Source: "On the Design of Qwen3.8-Next Architecture" (arXiv:2608.30320), as
restated on two pages:
  * research-hub notes, "Key ideas", QSA compressed-indexer bullet: MQA indexer
    (4 query heads + 1 shared 128-dim key head), keys average-pooled into blocks
    of r, partial RoPE (64 of 128 dims) applied after compression, block score
    I_ib = sum_h ReLU(<q_i^h, kbar_b>), top k_B = ceil(K/r) blocks plus the
    current-block tail, K = 2048 and r = 4.
  * paperglide reader, "Qwen Sparse Attention" toy walk-through (steps 1-5) and
    Fig. 3 caption: block-causal mask, selected blocks expanded back to tokens,
    plus the tokens of the incomplete final block, then sparse core attention.

Readings taken where the pages are silent:
  * RoPE pairs dims (j, j + rope_dims/2) for j < rope_dims/2 ("rotate-half"),
    frequencies theta_j = base^(-2j/rope_dims), base 10000.
  * Key block b sits at RoPE position b; query token i at position floor(i/r),
    so both live on the block-index scale.  Queries are rotated too.
  * Optional RMSNorm (unit weight) between pooling and RoPE, off by default
    (the paperglide toy mentions it, the Key-ideas bullet does not).
  * Block b is visible to token i iff b*r + r - 1 <= i, so token i sees
    c_i = floor((i+1)/r) blocks; a trailing partial block is never pooled.
  * Rows with c_i <= k_B keep every visible block.  Otherwise the k_B highest
    scores are kept, equal scores going to the lower block index.
  * Tail = tokens [c_i*r, i]; empty when token i closes its own block.
  * One selection per token, shared by every attention head.
  * The compressed keys and the rotated indexer queries are stored in bf16
    (round-to-nearest-even); the oracle rounds at exactly those two points and
    computes everything else in fp64.

Every function below takes and returns fp64 numpy arrays (bf16 inputs are
converted exactly with :func:`bf16_bits_to_f64`).  Loops over rows are plain
Python; no blocking, fusion or reordering beyond the definitions.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "round_to_bf16",
    "rope_inv_freq",
    "apply_partial_rope",
    "visible_blocks",
    "n_select",
    "compress_keys",
    "rotate_queries",
    "index_scores",
    "select_blocks",
    "token_set",
    "attend",
    "prefill_rows",
    "decode_rows",
]

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


# ---------------------------------------------------------------- bf16 values

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 values of bf16 numbers given as uint16 bit patterns."""
    u32 = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 number, ties to even.

    bf16 keeps 8 significant bits.  For |x| in [2^e', 2^(e'+1)) the spacing of
    bf16 numbers is 2^(e'-7); below the smallest normal (2^-126) it is the
    subnormal spacing 2^-133.  x is scaled by that spacing (exact: a power of
    two), rounded to an integer half-to-even, and scaled back, so the result
    is rounded once, straight from fp64.  Values that round past the largest
    finite bf16 become infinite.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e with 0.5 <= |m| < 1, so 2^(e-1) <= |x|
    quantum_exp = np.maximum(e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(x, -quantum_exp)), quantum_exp)
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, x), y)
    return np.where(np.isfinite(x), y, x)


# ---------------------------------------------------------------- RoPE

def rope_inv_freq(rope_dims: int, base: float) -> np.ndarray:
    """theta_j = base^(-2j / rope_dims) for j = 0 .. rope_dims/2 - 1."""
    j = np.arange(rope_dims // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * j / rope_dims)


def apply_partial_rope(x: np.ndarray, pos, rope_dims: int, base: float) -> np.ndarray:
    """Rotate dims [0, rope_dims) of x at position pos; other dims unchanged.

    Pair (j, j + rope_dims/2) is rotated by angle pos * theta_j:
        x_j'        = x_j cos(phi) - x_{j+h} sin(phi)
        x_{j+h}'    = x_j sin(phi) + x_{j+h} cos(phi)
    x has shape [..., d]; pos broadcasts against x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    if rope_dims == 0:
        return x.copy()
    h = rope_dims // 2
    phi = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(rope_dims, base)
    c, s = np.cos(phi), np.sin(phi)
    out = x.copy()
    x1 = x[..., :h]
    x2 = x[..., h:rope_dims]
    out[..., :h] = x1 * c - x2 * s
    out[..., h:rope_dims] = x1 * s + x2 * c
    return out


# ---------------------------------------------------------------- block structure

def visible_blocks(i: int, r: int) -> int:
    """c_i: number of completed blocks token i may score (block b needs b*r+r-1 <= i)."""
    return (i + 1) // r


def n_select(k_tokens: int, r: int) -> int:
    """k_B = ceil(K / r)."""
    return -(-k_tokens // r)


# ---------------------------------------------------------------- indexer keys and queries

def compress_keys(k_idx: np.ndarray, r: int, *, rope_dims: int = 64, rope_base: float = 10000.0,
                  rmsnorm: bool = False, rms_eps: float = 1e-6) -> np.ndarray:
    """Compressed indexer keys kbar [N_b, d] for indexer keys k_idx [n, d].

    kbar_b = (1/r) * sum_{t=b*r}^{b*r+r-1} k_t for the N_b = floor(n/r) complete
    blocks, then (optionally) RMSNorm with unit weight, then partial RoPE at
    position b, then rounding to bf16 (the library's storage point).
    """
    k_idx = np.asarray(k_idx, dtype=np.float64)
    n, d = k_idx.shape
    nb = n // r
    pooled = np.zeros((nb, d), dtype=np.float64)
    for t in range(r):
        pooled += k_idx[t: nb * r: r][:nb]
    pooled = pooled / r
    if rmsnorm:
        ms = np.mean(pooled * pooled, axis=-1, keepdims=True)
        pooled = pooled / np.sqrt(ms + rms_eps)
    rotated = apply_partial_rope(pooled, np.arange(nb), rope_dims, rope_base)
    return round_to_bf16(rotated)


def rotate_queries(q_idx: np.ndarray, positions, r: int, *, rope_dims: int = 64,
                   rope_base: float = 10000.0) -> np.ndarray:
    """Rotated indexer queries qtilde [m, H, d] (bf16-rounded) for tokens at `positions`.

    Token i is rotated at position floor(i / r), the index of the block it lies in.
    """
    q_idx = np.asarray(q_idx, dtype=np.float64)
    p = np.asarray(positions, dtype=np.int64) // r
    rotated = apply_partial_rope(q_idx, p[:, None], rope_dims, rope_base)
    return round_to_bf16(rotated)


def index_scores(qt: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """I_b = sum_h ReLU(<qt^h, kbar_b>) for every row b of kbar.  qt is [H, d]."""
    dots = np.asarray(kbar, np.float64) @ np.asarray(qt, np.float64).T  # [c, H]
    return np.maximum(dots, 0.0).sum(axis=1)


def select_blocks(scores: np.ndarray, k_b: int) -> np.ndarray:
    """Top-k_B block ids of one row, ascending.

    All blocks when there are at most k_B of them; otherwise the k_B largest
    scores, an equal score going to the lower block id.
    """
    c = scores.shape[0]
    if c <= k_b:
        return np.arange(c, dtype=np.int64)
    order = np.lexsort((np.arange(c), -scores))  # primary: score desc; secondary: id asc
    return np.sort(order[:k_b]).astype(np.int64)


def token_set(i: int, sel: np.ndarray, r: int) -> np.ndarray:
    """Tokens attended by token i: each selected block [b*r, b*r+r) plus the tail [c_i*r, i]."""
    c = visible_blocks(i, r)
    parts = [np.arange(b * r, b * r + r, dtype=np.int64) for b in np.asarray(sel)]
    parts.append(np.arange(c * r, i + 1, dtype=np.int64))
    return np.concatenate(parts)


# ---------------------------------------------------------------- sparse core attention

def attend(q_row: np.ndarray, k: np.ndarray, v: np.ndarray, tokens: np.ndarray,
           scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of one token over `tokens`, grouped-query layout.

    q_row [Hq, d]; k, v [Hkv, L, d].  Head h reads kv head h // (Hq/Hkv).
    o_h = sum_t p_t v_t with p = softmax_t(scale * <q_h, k_t>); lse_h = log sum_t exp(...).
    """
    hq, d = q_row.shape
    hkv = k.shape[0]
    g = hq // hkv
    out = np.zeros((hq, d), dtype=np.float64)
    lse = np.zeros(hq, dtype=np.float64)
    for h in range(hq):
        kk = k[h // g][tokens]
        vv = v[h // g][tokens]
        logits = scale * (kk @ q_row[h])
        m = logits.max()
        w = np.exp(logits - m)
        z = w.sum()
        out[h] = (w @ vv) / z
        lse[h] = m + math.log(z)
    return out, lse


# ---------------------------------------------------------------- whole-path drivers

def prefill_rows(q_idx, k_idx, q, k, v, rows, *, r: int, k_tokens: int, q_pos0: int = 0,
                 rope_dims: int = 64, rope_base: float = 10000.0, rmsnorm: bool = False,
                 rms_eps: float = 1e-6, scale: float | None = None, kbar=None,
                 with_attention: bool = True) -> dict:
    """QSA for selected query rows of one sequence.

    q_idx [n_q, H_idx, d], q [n_q, Hq, d]: rows of the chunk; row j is token q_pos0 + j.
    k_idx [L, d], k/v [Hkv, L, d]: the whole sequence up to the last query token.
    kbar: optional precomputed compressed keys (used as given, e.g. a decode cache).
    Returns per requested row: scores, selected blocks, tokens, output, lse.
    """
    d = q_idx.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if kbar is None:
        kbar = compress_keys(k_idx, r, rope_dims=rope_dims, rope_base=rope_base,
                             rmsnorm=rmsnorm, rms_eps=rms_eps)
    k_b = n_select(k_tokens, r)
    rows = [int(j) for j in rows]
    pos = np.array([q_pos0 + j for j in rows], dtype=np.int64)
    qt = rotate_queries(np.asarray(q_idx, np.float64)[rows], pos, r,
                        rope_dims=rope_dims, rope_base=rope_base)
    res = {"kbar": kbar, "k_b": k_b, "rows": rows, "pos": pos, "scores": [], "sel": [],
           "tokens": [], "out": None, "lse": None}
    outs, lses = [], []
    for n_row, i in enumerate(pos):
        c = visible_blocks(int(i), r)
        s = index_scores(qt[n_row], kbar[:c])
        sel = select_blocks(s, k_b)
        toks = token_set(int(i), sel, r)
        res["scores"].append(s)
        res["sel"].append(sel)
        res["tokens"].append(toks)
        if with_attention:
            o, l = attend(np.asarray(q[rows[n_row]], np.float64), k, v, toks, scale)
            outs.append(o)
            lses.append(l)
    if with_attention:
        res["out"] = np.stack(outs) if outs else np.zeros((0,) + tuple(q.shape[1:]))
        res["lse"] = np.stack(lses) if lses else np.zeros((0, q.shape[1]))
    return res


def decode_rows(q_idx_new, q_new, kbar, k_cache, v_cache, cache_len: int, *, r: int,
                k_tokens: int, rope_dims: int = 64, rope_base: float = 10000.0,
                scale: float | None = None) -> dict:
    """One decode step of one sequence: the new token sits at i = cache_len - 1.

    q_idx_new [H_idx, d], q_new [Hq, d]; kbar [>= c_i, d] is the compressed-key cache
    (already rotated, bf16 values); k_cache/v_cache [Hkv, >= cache_len, d].
    """
    i = cache_len - 1
    return prefill_rows(np.asarray(q_idx_new)[None], None, np.asarray(q_new)[None],
                        k_cache, v_cache, [0], r=r, k_tokens=k_tokens, q_pos0=i,
                        rope_dims=rope_dims, rope_base=rope_base, scale=scale, kbar=kbar)
