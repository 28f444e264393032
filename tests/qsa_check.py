"""Comparison helpers shared by the GPU parity tests (no test functions here).

The CUDA path and the oracle only meet here, on the test side: the oracle's
expected values are computed from the same seeded inputs, never from CUDA
results.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import qsa_oracle as O

# Block selection: a row may differ from the oracle only where the oracle's
# k_B-th and (k_B+1)-th scores are within this relative margin, and only by
# blocks whose oracle scores lie inside that margin around the k_B-th score.
SEL_REL_MARGIN = 1e-3
# Absolute floor of that margin, for rows whose k_B-th score is exactly 0
# (fp32 dot products of ReLU-zeroed heads may land at +-1e-7 instead of 0).
SEL_ABS_FLOOR = 1e-6
# Attention outputs (unit-variance V): max abs error.
OUT_ATOL = 1e-2
# Log-sum-exp per head.
LSE_ATOL = 1e-3


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a bf16 tensor."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_to_np32(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 copy of a bf16 tensor (half the memory of fp64; the oracle
    promotes every product with it to fp64)."""
    return t.detach().to("cpu").to(torch.float32).numpy()


def ulp_distance_bf16(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    """Distance in bf16 units in the last place (monotone integer mapping)."""
    def key(t):
        x = t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.int32) & 0xFFFF
        neg = (x & 0x8000) != 0
        mag = x & 0x7FFF
        return np.where(neg, -mag, mag)
    return np.abs(key(a) - key(b))


def check_selection_row(scores: np.ndarray, oracle_sel: np.ndarray, gpu_idx: np.ndarray,
                        gpu_count: int, c: int, k_b: int) -> str:
    """Returns "exact", "margin" (accepted near-tie swap) or raises AssertionError."""
    want = min(c, k_b)
    assert gpu_count == want, f"count {gpu_count} != {want}"
    sel = gpu_idx[:gpu_count]
    assert (gpu_idx[gpu_count:] == -1).all(), "padding past count must be -1"
    assert (np.diff(sel) > 0).all() if len(sel) > 1 else True, "ids must be strictly ascending"
    if len(sel):
        assert sel[0] >= 0 and sel[-1] < c, "ids must be visible blocks"
    if np.array_equal(sel, oracle_sel):
        return "exact"
    assert c > k_b, "rows with c <= k_B keep every block"
    srt = np.sort(scores)[::-1]
    tk, tk1 = srt[k_b - 1], srt[k_b]
    margin = SEL_REL_MARGIN * abs(tk) + SEL_ABS_FLOOR
    assert tk - tk1 < margin, f"selection differs but the k_B-th gap {tk - tk1:.3e} exceeds {margin:.3e}"
    swapped = np.setxor1d(sel, oracle_sel)
    assert (np.abs(scores[swapped] - tk) <= margin).all(), "swapped blocks lie outside the margin"
    return "margin"


def oracle_rows(wl: dict, rows, *, cfg, with_attention=True, q_pos0: int = 0) -> dict:
    """Oracle prefill results for `rows` of sequence 0 of a workload dict.  The
    attention inputs ride along in res["attn"], so that rows whose selection is
    an accepted near-tie swap can be re-attended on the GPU's own selection."""
    q, k, v = bf16_to_np32(wl["q"][0]), bf16_to_np32(wl["k"][0]), bf16_to_np32(wl["v"][0])
    res = O.prefill_rows(
        bf16_to_np32(wl["q_idx"][0]), bf16_to_np(wl["k_idx"][0]), q, k, v, rows, r=cfg.r,
        k_tokens=cfg.k_tokens, q_pos0=q_pos0, rope_dims=cfg.rope_dims, rope_base=cfg.rope_base,
        rmsnorm=cfg.rmsnorm, rms_eps=cfg.rms_eps, with_attention=with_attention)
    res["attn"] = (q, k, v)
    return res


def compare_prefill(res: dict, idx: np.ndarray, count: np.ndarray, out: np.ndarray | None,
                    lse: np.ndarray | None, k_b: int, r: int, row_offset: int = 0, attn=None,
                    scale: float | None = None) -> dict:
    """Checks GPU idx/count and out/lse against oracle rows.

    idx/count/out/lse are indexed by query row (row j of the chunk); res["rows"]
    lists which rows the oracle computed.  On a row whose selection matches the
    oracle's, out/lse are compared with the oracle's own attention; on a row
    accepted as a near-tie swap ("margin"), with the oracle's attention over the
    token set of the GPU's selection (its blocks plus the row's tail), computed
    from `attn` = (q [n_q, Hq, d], k [Hkv, L, d], v) or res["attn"].  Returns
    counts of exact / margin rows and the largest errors.
    """
    stats = {"exact": 0, "margin": 0, "max_out_err": 0.0, "max_lse_err": 0.0}
    if attn is None:
        attn = res.get("attn")
    for n, j in enumerate(res["rows"]):
        i = int(res["pos"][n])
        c = O.visible_blocks(i, r)
        kind = check_selection_row(res["scores"][n], res["sel"][n], idx[j], int(count[j]), c, k_b)
        stats[kind] += 1
        if out is None or res["out"] is None:
            continue
        if kind == "exact":
            want_o, want_l = res["out"][n], res["lse"][n]
        else:
            assert attn is not None, f"row {j}: near-tie row without attention inputs to check its output"
            q, k, v = attn
            sc = default_scale(q.shape[-1]) if scale is None else scale
            toks = O.token_set(i, idx[j][:int(count[j])].astype(np.int64), r)
            want_o, want_l = O.attend(np.asarray(q[res["rows"][n]], np.float64), k, v, toks, sc)
        err = float(np.abs(out[j] - want_o).max())
        assert err <= OUT_ATOL, f"row {j} ({kind}): output error {err}"
        stats["max_out_err"] = max(stats["max_out_err"], err)
        if lse is not None:
            e2 = float(np.abs(lse[j] - want_l).max())
            assert e2 <= LSE_ATOL, f"row {j} ({kind}): lse error {e2}"
            stats["max_lse_err"] = max(stats["max_lse_err"], e2)
    return stats


def sample_rows(n: int, k_b: int, r: int, extra, count: int, seed: int) -> list[int]:
    """Rows that cover the regimes: the c <= k_B prefix edge, ragged tail, random."""
    rng = np.random.default_rng(seed)
    edge = r * k_b
    rows = set(range(min(n, 8)))
    rows |= set(range(max(0, edge - 6), min(n, edge + 6)))
    rows |= set(range(max(0, n - 8), n))
    rows |= {int(x) for x in extra if 0 <= x < n}
    rows |= {int(x) for x in rng.integers(0, n, size=count)}
    return sorted(rows)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
