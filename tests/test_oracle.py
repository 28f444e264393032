"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a closed form, a library routine, a
brute-force enumeration or the paperglide toy walk-through, so that a dropped
term, a wrong sign, an off-by-one in the causal mask or a transposed operand
fails here before the oracle is trusted against the CUDA path.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ bf16 rounding

def test_round_to_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    ours = O.round_to_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ours, ref)


def test_round_to_bf16_hand_cases():
    # Spacing of bf16 at 1.0 is 2^-7.  Halfway cases go to the even neighbour.
    assert O.round_to_bf16(1 + 2.0 ** -8) == 1.0
    assert O.round_to_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    # Just above halfway rounds up; going through fp32 first would lose the 2^-30
    # and round down to 1.0 (double rounding), so this pins single rounding from fp64.
    assert O.round_to_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert O.round_to_bf16(-(1 + 2.0 ** -8 + 2.0 ** -30)) == -(1 + 2.0 ** -7)
    # Subnormal spacing 2^-133: half of it ties to zero, 1.5 of it ties to 2.
    assert O.round_to_bf16(2.0 ** -134) == 0.0
    assert O.round_to_bf16(3 * 2.0 ** -134) == 2.0 ** -132
    # Largest finite bf16 is (2 - 2^-7) * 2^127; at or past halfway to 2^128 -> inf.
    assert O.round_to_bf16(3.39e38) == (2 - 2.0 ** -7) * 2.0 ** 127
    assert np.isinf(O.round_to_bf16(3.40e38))
    assert O.round_to_bf16(0.0) == 0.0


def test_bf16_bits_roundtrip():
    t = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), t.double().numpy())


# ------------------------------------------------------------------ RoPE

def test_rope_frequencies_closed_form():
    th = O.rope_inv_freq(64, 10000.0)
    assert th.shape == (32,)
    assert th[0] == 1.0
    assert th[8] == pytest.approx(0.1, rel=1e-15)    # 10000^(-16/64)
    assert th[16] == pytest.approx(0.01, rel=1e-15)  # 10000^(-32/64)
    assert th[24] == pytest.approx(0.001, rel=1e-15)


def test_rope_hand_case_and_identity():
    x = np.zeros(128)
    x[16] = 1.0
    y = O.apply_partial_rope(x, 100, 64, 10000.0)  # angle 100 * 0.01 = 1 rad on pair (16, 48)
    assert y[16] == pytest.approx(math.cos(1.0), abs=1e-14)
    assert y[48] == pytest.approx(math.sin(1.0), abs=1e-14)
    assert np.count_nonzero(np.abs(y) > 1e-14) == 2
    rng = np.random.default_rng(1)
    z = rng.standard_normal((5, 128))
    np.testing.assert_array_equal(O.apply_partial_rope(z, 0, 64, 10000.0), z)


def test_rope_equals_complex_rotation():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 128))
    pos = np.array([0, 1, 5, 77, 1000, 65535, 262143])
    y = O.apply_partial_rope(x, pos, 64, 10000.0)
    theta = 10000.0 ** (-np.arange(32) / 32.0)
    zc = (x[:, :32] + 1j * x[:, 32:64]) * np.exp(1j * pos[:, None] * theta)
    np.testing.assert_allclose(y[:, :32], zc.real, rtol=0, atol=1e-9)
    np.testing.assert_allclose(y[:, 32:64], zc.imag, rtol=0, atol=1e-9)
    np.testing.assert_array_equal(y[:, 64:], x[:, 64:])


def test_rope_relative_position_property():
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    for p, q in [(10, 3), (500, 17), (4096, 4000)]:
        lhs = O.apply_partial_rope(a, p, 64, 10000.0) @ O.apply_partial_rope(b, q, 64, 10000.0)
        rhs = O.apply_partial_rope(a, p - q, 64, 10000.0) @ b
        assert lhs == pytest.approx(rhs, rel=1e-10, abs=1e-10)


# ------------------------------------------------------------------ key compression

def test_compress_keys_pooling_closed_form():
    n, r = 18, 4
    k = np.arange(n, dtype=np.float64)[:, None] * np.ones((1, 128))
    kb = O.compress_keys(k, r, rope_dims=0)
    assert kb.shape == (4, 128)  # trailing partial block (tokens 16, 17) is not pooled
    for b in range(4):
        np.testing.assert_array_equal(kb[b], np.full(128, b * r + (r - 1) / 2))


def test_compress_keys_rope_at_block_index_and_bf16_storage():
    rng = np.random.default_rng(4)
    k = O.round_to_bf16(rng.standard_normal((64, 128)))
    kb = O.compress_keys(k, 4)
    pooled = k.reshape(16, 4, 128).mean(axis=1)
    np.testing.assert_array_equal(kb[:, 64:], O.round_to_bf16(pooled[:, 64:]))
    np.testing.assert_array_equal(kb[0], O.round_to_bf16(pooled[0]))  # block 0: position 0
    ref = O.round_to_bf16(O.apply_partial_rope(pooled, np.arange(16), 64, 10000.0))
    np.testing.assert_array_equal(kb, ref)
    np.testing.assert_array_equal(O.round_to_bf16(kb), kb)


def test_compress_keys_rmsnorm_matches_library():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((32, 128)) * 3.0
    kb = O.compress_keys(k, 4, rope_dims=0, rmsnorm=True, rms_eps=1e-6)
    pooled = torch.from_numpy(k.reshape(8, 4, 128).mean(axis=1))
    ref = torch.nn.functional.rms_norm(pooled, (128,), eps=1e-6).numpy()
    np.testing.assert_array_equal(kb, O.round_to_bf16(ref))


# ------------------------------------------------------------------ indexer scores

def test_index_scores_bruteforce_and_relu():
    rng = np.random.default_rng(6)
    qt = rng.standard_normal((4, 128))
    kb = rng.standard_normal((9, 128))
    got = O.index_scores(qt, kb)
    for b in range(9):
        tot = 0.0
        for h in range(4):
            dot = sum(qt[h, j] * kb[b, j] for j in range(128))
            tot += dot if dot > 0 else 0.0
        assert got[b] == pytest.approx(tot, rel=1e-12, abs=1e-12)
    assert (got >= 0).all()


def test_index_scores_zero_iff_all_heads_nonpositive():
    qt = np.zeros((4, 128))
    qt[:, 0] = [1.0, 2.0, -1.0, 0.5]
    kb = np.zeros((3, 128))
    kb[0, 0] = -1.0   # dots: -1, -2, +1, -0.5 -> only head 2 positive
    kb[1, 0] = 2.0    # dots: 2, 4, -2, 1     -> 7
    kb[2, 1] = 5.0    # dots all 0            -> 0
    np.testing.assert_array_equal(O.index_scores(qt, kb), [1.0, 7.0, 0.0])
    qneg = -np.abs(qt)
    assert O.index_scores(qneg, np.abs(kb))[1] == 0.0


# ------------------------------------------------------------------ top-k_B selection

@pytest.mark.parametrize("c,k_b", [(c, k) for c in range(1, 9) for k in (1, 2, 3)])
def test_select_blocks_bruteforce(c, k_b):
    rng = np.random.default_rng(100 * c + k_b)
    for trial in range(20):
        s = rng.integers(0, 4, size=c).astype(np.float64)  # many exact ties
        if trial % 2:
            s = rng.standard_normal(c)
        got = O.select_blocks(s, k_b)
        if c <= k_b:
            np.testing.assert_array_equal(got, np.arange(c))
            continue
        best = max(sum(s[list(sub)]) for sub in itertools.combinations(range(c), k_b))
        maximisers = [sub for sub in itertools.combinations(range(c), k_b)
                      if sum(s[list(sub)]) == best]
        assert tuple(got) == min(maximisers)  # lexicographically smallest maximiser


def test_select_blocks_ties_prefer_lower_ids():
    np.testing.assert_array_equal(O.select_blocks(np.zeros(10), 3), [0, 1, 2])
    s = np.array([0.0, 5.0, 0.0, 5.0, 0.0, 5.0])
    np.testing.assert_array_equal(O.select_blocks(s, 2), [1, 3])


# ------------------------------------------------------------------ toy walk-through

def test_toy_walkthrough_structure():
    with open(os.path.join(GOLDEN, "toy_walkthrough.json")) as f:
        g = json.load(f)
    r, i, k_b = g["r"], g["token"], g["k_b"]
    c = O.visible_blocks(i, r)
    assert list(range(c)) == g["visible_blocks"]
    # Keys pooled per the page (block 0 = mean of keys 0, 1; block 1 = mean of 2, 3).
    k = np.zeros((6, 128))
    k[:, 0] = [1, 3, 4, 6, 7, 9]
    kb = O.compress_keys(k, r, rope_dims=0)
    assert kb[0, 0] == 2.0 and kb[1, 0] == 5.0 and kb[2, 0] == 8.0
    # Two indexer heads; a query along +dim0 makes the later blocks score higher.
    qt = np.zeros((g["n_idx_heads"], 128))
    qt[:, 0] = 1.0
    s = O.index_scores(qt, kb[:c])
    sel = O.select_blocks(s, k_b)
    assert list(sel) == g["selected_blocks"]
    toks = O.token_set(i, sel, r)
    assert list(toks) == g["selected_tokens"] + g["tail_tokens"]
    assert len(toks) == g["attended_token_count"]
    # Token 4 has one completed block fewer and a one-token tail.
    assert O.visible_blocks(4, r) == 2
    assert list(O.token_set(4, np.array([0, 1]), r)) == [0, 1, 2, 3, 4]


def test_visible_blocks_and_tail_sizes():
    r, k_b = 4, 3
    for i in range(40):
        c = O.visible_blocks(i, r)
        assert c * r <= i + 1 < c * r + r
        sel = np.arange(min(c, k_b))
        toks = O.token_set(i, sel, r)
        assert len(toks) == min(c, k_b) * r + (i + 1 - c * r)
        assert toks.max() <= i and len(set(toks.tolist())) == len(toks)


# ------------------------------------------------------------------ sparse attention

def _dense_gqa_sdpa(q, k, v, scale):
    """Causal grouped-query attention from torch's SDPA, fp64, q [n,Hq,d], k/v [Hkv,n,d]."""
    g = q.shape[1] // k.shape[0]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).repeat_interleave(g, dim=0)[None]
    vt = torch.from_numpy(v).repeat_interleave(g, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_full_selection_equals_dense_causal_gqa():
    rng = np.random.default_rng(7)
    n, d = 37, 128
    q_idx = rng.standard_normal((n, 4, d))
    k_idx = rng.standard_normal((n, d))
    q = rng.standard_normal((n, 16, d))
    k = rng.standard_normal((2, n, d))
    v = rng.standard_normal((2, n, d))
    res = O.prefill_rows(q_idx, k_idx, q, k, v, range(n), r=4, k_tokens=4 * 64)
    ref = _dense_gqa_sdpa(q, k, v, 1 / math.sqrt(d))
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-12)
    for i in range(n):
        assert len(res["tokens"][i]) == i + 1


def test_attend_single_token_constant_v_and_lse():
    from scipy.special import logsumexp
    rng = np.random.default_rng(8)
    q = rng.standard_normal((16, 128))
    k = rng.standard_normal((2, 10, 128))
    v = rng.standard_normal((2, 10, 128))
    o, lse = O.attend(q, k, v, np.array([6]), 0.1)
    np.testing.assert_array_equal(o[:8], np.broadcast_to(v[0, 6], (8, 128)))
    np.testing.assert_array_equal(o[8:], np.broadcast_to(v[1, 6], (8, 128)))
    vc = np.ones_like(v) * 0.75
    o2, _ = O.attend(q, k, vc, np.array([0, 3, 9]), 0.1)
    np.testing.assert_allclose(o2, 0.75, rtol=0, atol=1e-15)
    toks = np.array([1, 2, 5, 7])
    _, lse = O.attend(q, k, v, toks, 0.1)
    for h in range(16):
        assert lse[h] == pytest.approx(logsumexp(0.1 * (k[h // 8][toks] @ q[h])), rel=1e-14)


def test_selection_restricts_attention():
    """Rows past the k_B budget attend exactly the selected blocks plus the tail."""
    rng = np.random.default_rng(9)
    n, r, K = 64, 4, 16  # k_B = 4 blocks
    q_idx = rng.standard_normal((n, 4, 128))
    k_idx = rng.standard_normal((n, 128))
    q = rng.standard_normal((n, 16, 128))
    k = rng.standard_normal((2, n, 128))
    v = rng.standard_normal((2, n, 128))
    res = O.prefill_rows(q_idx, k_idx, q, k, v, [62, 63], r=r, k_tokens=K)
    for j, i in enumerate([62, 63]):
        sel = res["sel"][j]
        assert len(sel) == 4
        s = res["scores"][j]
        assert s[sel].min() >= np.delete(s, sel).max()
        o, _ = O.attend(q[i], k, v, res["tokens"][j], 1 / math.sqrt(128))
        np.testing.assert_array_equal(res["out"][j], o)
    assert len(res["tokens"][0]) == 4 * 4 + 3   # token 62: tail 60..62
    assert len(res["tokens"][1]) == 4 * 4       # token 63 closes block 15: empty tail


def test_decode_equals_last_prefill_row():
    rng = np.random.default_rng(10)
    L, r = 203, 4
    q_idx = rng.standard_normal((L, 4, 128))
    k_idx = rng.standard_normal((L, 128))
    q = rng.standard_normal((L, 16, 128))
    k = rng.standard_normal((2, L, 128))
    v = rng.standard_normal((2, L, 128))
    pre = O.prefill_rows(q_idx, k_idx, q, k, v, [L - 1], r=r, k_tokens=64)
    kbar = O.compress_keys(k_idx, r)
    dec = O.decode_rows(q_idx[L - 1], q[L - 1], kbar, k, v, L, r=r, k_tokens=64)
    np.testing.assert_array_equal(dec["sel"][0], pre["sel"][0])
    np.testing.assert_array_equal(dec["out"], pre["out"])


# ------------------------------------------------------------------ query rotation and k_B
# The query-side reading (research-hub notes, "Key ideas", QSA bullet: partial
# RoPE after compression; keys sit at block index b, so query token i sits at
# the index floor(i / r) of the block it lies in, and the rotated query is
# stored in bf16).  Each pin below is computed without the oracle's own rotation
# routine: complex multiplication for the rotation, torch for the bf16 rounding.

def _complex_rope(x: np.ndarray, angle_pos: float, base: float = 10000.0) -> np.ndarray:
    """Rotate dims 0..63 of x by pos * base^(-j/32) as complex numbers x_j + i x_{j+32}."""
    theta = base ** (-np.arange(32) / 32.0)
    z = (x[..., :32] + 1j * x[..., 32:64]) * np.exp(1j * angle_pos * theta)
    out = np.array(x, dtype=np.float64, copy=True)
    out[..., :32] = z.real
    out[..., 32:64] = z.imag
    return out


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def test_rotate_queries_is_rounded_rotation_at_block_index():
    """Each rotated query is the rotation at floor(i / r), rounded once to bf16."""
    rng = np.random.default_rng(20)
    r = 4
    positions = np.array([0, 1, 3, 4, 7, 9, 130, 131, 4097, 262143])
    q = O.round_to_bf16(rng.standard_normal((len(positions), 4, 128)))  # bf16 inputs, as the library gets
    got = O.rotate_queries(q, positions, r)
    assert got.shape == q.shape
    np.testing.assert_array_equal(O.round_to_bf16(got), got)  # stored as bf16 numbers
    for n, i in enumerate(positions):
        ref = _torch_bf16(_complex_rope(q[n], i // r))
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
        assert np.all(np.abs(got[n] - ref) <= ulp), i  # fp64 rotation order may flip a halfway case
        assert (got[n] == ref).mean() > 0.99, i
        np.testing.assert_array_equal(got[n][:, 64:], q[n][:, 64:])  # unrotated dims pass through


def test_rotate_queries_hand_cases():
    # Dim 0 rotates at theta_0 = 1 rad per block: token 9 with r = 4 is in block 2.
    q = np.zeros((1, 4, 128))
    q[0, :, 0] = 1.0
    got = O.rotate_queries(q, [9], 4)
    assert got[0, 0, 0] == _torch_bf16(math.cos(2.0)) and got[0, 0, 32] == _torch_bf16(math.sin(2.0))
    assert got[0, 0, 0] == -0.416015625 and got[0, 0, 32] == 0.91015625  # bf16(cos 2), bf16(sin 2)
    assert np.count_nonzero(got[0]) == 8
    # A base with theta_16 = pi / 2: token 6 with r = 4 (block 1) turns dim 16 onto
    # dim 48; at position 6 (the token index) it would land on -dim 16, and with
    # the sign of the angle flipped on -dim 48.
    base = (2.0 / math.pi) ** 2
    q = np.zeros((1, 1, 128))
    q[0, 0, 16] = 1.0
    got = O.rotate_queries(q, [6], 4, rope_base=base)[0, 0]
    assert got[48] == 1.0
    assert abs(got[16]) < 1e-15
    assert np.count_nonzero(np.abs(got) > 1e-15) == 1


def test_indexer_score_depends_on_block_distance_only():
    """<qt_i, kbar_b> equals <q, R_(b - floor(i/r)) pooled_b> for every token i of a
    block and every block b it sees, within the bf16 storage bound; when token i
    closes its own block b (b = floor(i/r)) the rotations cancel and the product
    is the unrotated one."""
    rng = np.random.default_rng(21)
    r, n = 4, 64
    k = O.round_to_bf16(rng.standard_normal((n, 128)))
    pooled = k.reshape(n // r, r, 128).mean(axis=1)
    kbar = O.compress_keys(k, r)
    q = rng.standard_normal((1, 4, 128))
    for i in range(36, 40):  # the four tokens of block 9
        p = i // r
        assert p == 9
        qt = O.rotate_queries(q, [i], r)[0]
        for b in range(O.visible_blocks(i, r)):
            rel = _complex_rope(pooled[b], b - p)
            want = rel @ q[0].T  # [4 heads]
            got = kbar[b] @ qt.T
            # q and kbar each carry one bf16 rounding (relative 2^-9 per element).
            bound = 2.0 ** -8 * (np.abs(q[0]) @ np.abs(rel)) * 1.01
            assert np.all(np.abs(got - want) <= bound), (i, b)
        if i == 39:  # token 39 closes block 9, which it now sees
            own = kbar[9] @ qt.T
            bound = 2.0 ** -8 * (np.abs(q[0]) @ np.abs(pooled[9])) * 1.01
            assert np.all(np.abs(own - q[0] @ pooled[9]) <= bound)


def test_n_select_is_a_ceiling():
    assert O.n_select(2048, 4) == 512
    assert O.n_select(2049, 4) == 513
    assert O.n_select(6, 4) == 2
    assert O.n_select(1, 16) == 1
    assert O.n_select(512, 4) == 128
    for K in range(1, 70):
        for r in (1, 2, 4, 8, 16):
            kb = O.n_select(K, r)
            assert (kb - 1) * r < K <= kb * r
