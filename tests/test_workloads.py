"""The synthetic input recipe on CPU: the named workloads carry the stated
configurations, draws are reproducible from the seed, the drift is the stated
stationary AR(1) process, and planted needle blocks sit where the recipe puts
them.  The recipe holds no QSA arithmetic; these tests pin the inputs that the
parity tests and the bench feed to both the oracle and the CUDA library."""
import numpy as np
import torch

from block_sparse_long_17_b300 import workloads as W


def test_named_workloads_match_their_configurations():
    t = W.WORKLOADS["tiny_prefill_2k"]
    assert (t.n, t.k_tokens, t.k_b, t.r, t.seed, t.needles, t.drift) == (2048, 512, 128, 4, 0, 0, False)
    s = W.WORKLOADS["needle_prefill_32k"]
    assert (s.n, s.k_tokens, s.k_b, s.seed, s.needles) == (32768, 2048, 512, 1, 64)
    m = W.WORKLOADS["drift_prefill_128k"]
    assert (m.n, m.k_b, m.seed, m.drift, m.needles) == (131072, 512, 2, True, 0)
    d = W.WORKLOADS["decode_256k_x64"]
    assert (d.batch, d.ctx, d.cache_len, d.n_blocks, d.k_b, d.seed) == (64, 262144, 262145, 65536, 512, 3)
    g = W.WORKLOADS["needle_prefill_1m"]
    assert (g.n, g.k_b, g.seed, g.needles) == (1 << 20, 512, 4, 256)
    x = W.WORKLOADS["decode_1m_b4_next4"]
    assert (x.batch, x.next_n, x.cache_len, x.n_blocks) == (4, 4, 1 << 20, 1 << 18)
    for spec in W.WORKLOADS.values():  # head layout shared by every config
        assert (spec.h_idx, spec.d, spec.rope_dims, spec.rope_base, spec.hq, spec.hkv) == (4, 128, 64, 10000.0, 16, 2)


def test_prefill_draws_are_reproducible_and_bf16():
    spec = W.PrefillSpec("t", n=96, k_tokens=64, seed=5)
    a, b = W.make_prefill(spec), W.make_prefill(spec)
    for key in ("q_idx", "k_idx", "q", "k", "v"):
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
    assert a["q_idx"].shape == (1, 96, 4, 128) and a["k_idx"].shape == (1, 96, 128)
    assert a["q"].shape == (1, 96, 16, 128) and a["k"].shape == (1, 2, 96, 128) == a["v"].shape
    c = W.make_prefill(W.PrefillSpec("t", n=96, k_tokens=64, seed=6))
    assert not torch.equal(a["q_idx"], c["q_idx"])
    # N(0, 1) draws: moments of the 98304 attention-query entries
    qf = a["q"].float()
    assert abs(qf.mean().item()) < 0.02 and abs(qf.std().item() - 1.0) < 0.02


def test_ar1_drift_is_stationary_with_unit_variance_and_lag1_correlation():
    rng = np.random.default_rng(0)
    a = W._ar1_drift(200000, 8, rng)
    assert abs(a.var(axis=0).mean() - 1.0) < 0.06
    lag1 = np.mean([np.corrcoef(a[:-1, j], a[1:, j])[0, 1] for j in range(8)])
    assert abs(lag1 - 0.99) < 0.002
    # the first step is N(0, 1) too (a_0 drawn from the stationary law)
    starts = np.array([W._ar1_drift(1, 1, np.random.default_rng(s))[0, 0] for s in range(2000)])
    assert abs(starts.std() - 1.0) < 0.05


def test_drift_is_added_to_indexer_and_attention_keys_only():
    plain = W.make_prefill(W.PrefillSpec("t", n=64, k_tokens=64, seed=2))
    drift = W.make_prefill(W.PrefillSpec("t", n=64, k_tokens=64, seed=2, drift=True))
    for key in ("q_idx", "q", "v"):
        assert torch.equal(plain[key], drift[key])
    for key in ("k_idx", "k"):
        assert not torch.equal(plain[key], drift[key])


def test_needles_are_planted_where_the_recipe_says():
    spec = W.PrefillSpec("t", n=4096, k_tokens=256, seed=9, needles=8)
    wl = W.make_prefill(spec)
    assert len(wl["needles"]) == 8
    k_idx, q_idx = wl["k_idx"].float(), wl["q_idx"].float()
    for bb, i, blk in wl["needles"]:
        assert bb == 0 and spec.r * spec.k_b <= i < spec.n
        assert 0 <= blk < (i + 1) // spec.r
        keys = k_idx[bb, blk * spec.r:(blk + 1) * spec.r]
        # q_idx[i, head 0] + 0.1 N(0, 1), rounded to bf16: within a few noise sigmas
        dev = (keys - q_idx[bb, i, 0][None]).abs()
        assert dev.max().item() < 0.6 and dev.mean().item() < 0.12


def test_decode_draws_layout_and_cache_lengths():
    spec = W.DecodeSpec("t", batch=3, ctx=100, k_tokens=64, seed=1, next_n=2)
    wl = W.make_decode(spec)
    assert wl["cache_len"] == 102 and wl["n_blocks"] == 25 and wl["l_cap"] == 106
    assert wl["q_idx"].shape == (3, 2, 4, 128) and wl["q"].shape == (3, 2, 16, 128)
    assert wl["kbar"].shape == (3, 25, 128)
    assert wl["k"].shape == (3, 2, 106, 128) == wl["v"].shape
    assert torch.equal(wl["cache_lens"], torch.full((3,), 102, dtype=torch.int64))
    again = W.make_decode(spec)
    for key in ("q_idx", "kbar", "q", "k", "v"):
        assert torch.equal(wl[key], again[key])
