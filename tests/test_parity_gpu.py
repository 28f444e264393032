"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle
on identical seeded inputs.

Selections must match the oracle exactly except at near-ties (see
qsa_check.check_selection_row); attention outputs must be within 1e-2 max-abs
of the fp64 oracle for unit-variance V.
"""
import math

import numpy as np
import pytest
import torch

from block_sparse_long_17_b300 import qsa
from block_sparse_long_17_b300.workloads import WORKLOADS, DecodeSpec, PrefillSpec, make_decode, make_prefill
from oracle import qsa_oracle as O
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cfg_for(spec, **kw) -> qsa.Config:
    base = dict(r=spec.r, rope_dims=spec.rope_dims, rope_base=spec.rope_base, k_tokens=spec.k_tokens,
                n_idx_heads=spec.h_idx)
    base.update(kw)
    return qsa.Config(**base)


def run_prefill(cfg: qsa.Config, wl: dict, q_pos0: int = 0, rows: slice | None = None, impl: str = "auto"):
    """Full GPU prefill of sequence batch `wl` through the binding; returns numpy views.
    impl picks the attention kernel ("auto", "tcgen05" or "mma_sync")."""
    q_idx, k_idx, q, k, v = wl["q_idx"], wl["k_idx"], wl["q"], wl["k"], wl["v"]
    if rows is not None:  # chunk of query rows at positions q_pos0 + j
        q_idx, q = q_idx[:, rows].contiguous(), q[:, rows].contiguous()
    B, n_q = q_idx.shape[0], q_idx.shape[1]
    L = k_idx.shape[1]
    nb = L // cfg.r
    kbar = torch.empty((B, max(nb, 1), 128), dtype=torch.bfloat16, device=DEV)
    qsa.qsa_compress_keys(cfg, k_idx, 0, nb, kbar)
    q_pos = torch.full((B,), q_pos0, dtype=torch.int64, device=DEV)
    idx = torch.empty((B, n_q, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, n_q), dtype=torch.int32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, B, n_q, nb),), dtype=torch.uint8, device=DEV)
    qsa.qsa_index_topk(cfg, q_idx, kbar, q_pos, nb, idx, cnt, ws)
    fallback_rows = qsa.qsa_index_topk_fallback_rows(cfg, B, n_q, nb, ws)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    qsa.qsa_sparse_attn_prefill(cfg, q, k, v, q_pos, idx, cnt, out, lse, impl=impl)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    return {"kbar": kbar, "idx": idx.cpu().numpy(), "count": cnt.cpu().numpy(),
            "out": out.float().cpu().numpy(), "lse": lse.cpu().numpy(), "fallback_rows": fallback_rows}


# ----------------------------------------------------------------------------- key compression

@pytest.mark.parametrize("r,rope_dims,rmsnorm,n", [(4, 64, False, 2048), (4, 64, True, 2048),
                                                    (2, 64, False, 999), (8, 128, False, 1030),
                                                    (16, 32, True, 517), (4, 0, False, 64)])
def test_compress_keys_matches_oracle(r, rope_dims, rmsnorm, n):
    spec = PrefillSpec("t", n=n, k_tokens=64, seed=11, r=r, rope_dims=rope_dims)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec, rmsnorm=rmsnorm)
    nb = n // r
    kbar = torch.zeros((1, nb, 128), dtype=torch.bfloat16, device=DEV)
    qsa.qsa_compress_keys(cfg, wl["k_idx"], 0, nb, kbar)
    ref = O.compress_keys(QC.bf16_to_np(wl["k_idx"][0]), r, rope_dims=rope_dims,
                          rope_base=cfg.rope_base, rmsnorm=rmsnorm, rms_eps=cfg.rms_eps)
    ref_t = torch.from_numpy(ref).to(torch.bfloat16)  # exact: ref values are bf16 numbers
    d = QC.ulp_distance_bf16(kbar[0].cpu(), ref_t)
    assert d.max() <= 1, "kbar off by more than one bf16 ulp"
    assert (d > 0).mean() < 1e-3, f"too many 1-ulp differences: {(d > 0).mean()}"


def test_compress_keys_decode_append_touches_only_its_block():
    spec = DecodeSpec("t", batch=3, ctx=203, k_tokens=64, seed=5)
    gen = torch.Generator(device=DEV).manual_seed(5)
    L = 208
    k_idx = torch.randn((3, L, 128), generator=gen, device=DEV).to(torch.bfloat16)
    cfg = cfg_for(spec)
    kbar = torch.full((3, 64, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    qsa.qsa_compress_keys(cfg, k_idx, 51, 1, kbar)  # block 51 = tokens 204..207
    kb = kbar.cpu()
    for bb in range(3):
        ref = O.compress_keys(QC.bf16_to_np(k_idx[bb]), 4)[51]
        d = QC.ulp_distance_bf16(kb[bb, 51], torch.from_numpy(ref).to(torch.bfloat16))
        assert d.max() <= 1
        assert (kb[bb, :51] == 7.0).all() and (kb[bb, 52:] == 7.0).all()


# ----------------------------------------------------------------------------- tiny prefill (cfg 0)

@pytest.fixture(scope="module")
def tiny():
    spec = WORKLOADS["tiny_prefill_2k"]
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    res = QC.oracle_rows(wl, range(spec.n), cfg=cfg)
    return spec, cfg, wl, gpu, res


def test_tiny_prefill_selection_and_output_all_rows(tiny):
    spec, cfg, wl, gpu, res = tiny
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0],
                            cfg.k_b, cfg.r)
    assert st["exact"] + st["margin"] == spec.n
    assert st["margin"] <= spec.n // 100, st


@pytest.mark.parametrize("impl", ["tcgen05", "mma_sync"])
def test_tiny_attention_on_oracle_selection(tiny, impl):
    """Each attention kernel alone, fed the oracle's own selection, on every row."""
    spec, cfg, wl, gpu, res = tiny
    n, k_b = spec.n, cfg.k_b
    idx = np.full((1, n, k_b), -1, dtype=np.int32)
    cnt = np.zeros((1, n), dtype=np.int32)
    for j in range(n):
        s = res["sel"][j]
        idx[0, j, :len(s)] = s
        cnt[0, j] = len(s)
    q_pos = torch.zeros((1,), dtype=torch.int64, device=DEV)
    out = torch.empty_like(wl["q"])
    lse = torch.empty(wl["q"].shape[:3], dtype=torch.float32, device=DEV)
    qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], q_pos, torch.from_numpy(idx).to(DEV),
                                torch.from_numpy(cnt).to(DEV), out, lse, impl=impl)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    o = out.float().cpu().numpy()[0]
    assert np.abs(o - res["out"]).max() <= QC.OUT_ATOL
    assert np.abs(lse.cpu().numpy()[0] - res["lse"]).max() <= QC.LSE_ATOL


def test_tiny_rotated_query_scores_match_oracle(tiny):
    """Selections agree with the oracle on >= 99% of the rows that must choose."""
    spec, cfg, wl, gpu, res = tiny
    choosing = [j for j in range(spec.n) if O.visible_blocks(j, cfg.r) > cfg.k_b]
    same = sum(np.array_equal(gpu["idx"][0, j, :cfg.k_b], res["sel"][j]) for j in choosing)
    assert same >= 0.99 * len(choosing)


# ----------------------------------------------------------------------------- edge cases

def small_case(n, k_tokens, r=4, hq=16, hkv=2, seed=3, rope_dims=64):
    spec = PrefillSpec("e", n=n, k_tokens=k_tokens, seed=seed, r=r, hq=hq, hkv=hkv, rope_dims=rope_dims)
    return spec, make_prefill(spec, DEV)


@pytest.mark.parametrize("impl", ["auto", "tcgen05"])
@pytest.mark.parametrize("n,k_tokens,r,hq,hkv", [
    (1, 64, 4, 16, 2),       # one token, no complete block: tail only
    (3, 64, 4, 16, 2),       # n < r
    (37, 4096, 4, 16, 2),    # k_B >= every block: dense causal attention
    (300, 64, 4, 8, 8),      # group size 1 (MHA)
    (300, 64, 4, 32, 2),     # group size 16: two head chunks per kv head
    (300, 64, 4, 12, 4),     # group size 3: padded head chunk
    (401, 40, 2, 16, 2),     # r = 2, k_B = 20
    (777, 128, 8, 16, 2),    # r = 8
    (515, 48, 16, 16, 1),    # r = 16, one kv head, group size 16
    (515, 48, 16, 8, 1),     # r = 16, one kv head, group size 8
    (1999, 300, 4, 16, 2),   # k_B = 75: a last stage of 11 slots (odd, padded to a whole K-step)
])
def test_edge_shapes_match_oracle(n, k_tokens, r, hq, hkv, impl):
    """Every shape through "auto" (the mma.sync kernel), and through the tcgen05
    kernel where it applies (8 query heads per kv head, r in {4, 8, 16})."""
    if impl == "tcgen05" and not (hq == 8 * hkv and r in (4, 8, 16)):
        pytest.skip("shape outside the tcgen05 kernel (its refusal is tested separately)")
    spec, wl = small_case(n, k_tokens, r, hq, hkv)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl, impl=impl)
    res = QC.oracle_rows(wl, range(n), cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0],
                            cfg.k_b, cfg.r)
    assert st["exact"] >= 0.98 * n


def test_tcgen05_kernel_refuses_unsupported_shapes():
    """The tcgen05 kernel serves 8 query heads per kv head and r in {4, 8, 16};
    asked for anything else it returns QSA_ERR_UNSUPPORTED and launches nothing."""
    for (hq, hkv, r) in [(16, 1, 4), (12, 4, 4), (16, 2, 2)]:
        spec, wl = small_case(64, 64, r, hq, hkv)
        cfg = cfg_for(spec)
        q_pos = torch.zeros((1,), dtype=torch.int64, device=DEV)
        idx = torch.zeros((1, 64, cfg.k_b), dtype=torch.int32, device=DEV)
        cnt = torch.zeros((1, 64), dtype=torch.int32, device=DEV)
        out = torch.empty_like(wl["q"])
        launches = qsa.qsa_launch_count()
        with pytest.raises(qsa.QsaError) as ei:
            qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], q_pos, idx, cnt, out, impl="tcgen05")
        assert ei.value.status == 2
        assert qsa.qsa_launch_count() == launches


def test_tcgen05_and_mma_sync_kernels_agree_at_32k():
    """The two attention kernels on the needle workload's own GPU selection: both
    within the output tolerance of each other on every row (they differ in
    rounding order only)."""
    spec = WORKLOADS["needle_prefill_32k"]
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    a = run_prefill(cfg, wl, impl="tcgen05")
    b = run_prefill(cfg, wl, impl="mma_sync")
    np.testing.assert_array_equal(a["idx"], b["idx"])
    assert np.abs(a["out"] - b["out"]).max() <= QC.OUT_ATOL
    assert np.abs(a["lse"] - b["lse"]).max() <= QC.LSE_ATOL


def test_dense_limit_equals_torch_sdpa():
    """k_B >= every block: QSA is dense causal GQA (checked against torch SDPA, fp32)."""
    spec, wl = small_case(129, 1 << 12)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    q = wl["q"][0].float().permute(1, 0, 2)[None]
    k = wl["k"][0].float().repeat_interleave(8, dim=0)[None]
    v = wl["v"][0].float().repeat_interleave(8, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)[0].permute(1, 0, 2)
    assert np.abs(gpu["out"][0] - ref.cpu().numpy()).max() <= QC.OUT_ATOL


def test_attention_rescales_when_later_scores_jump():
    """The online softmax keeps its running maximum until a score exceeds it by
    more than 8 (log2 units) and only then rescales O and the sum.  The
    attention keys of the sequence's second half are scaled by 12, so that a
    row's scores jump far above its running maximum once its token set (the
    selected blocks in ascending order, then the tail) reaches them; the rows
    are checked against the oracle, and the same rows with the keys unscaled
    exercise the path that never rescales after its first stage."""
    spec, wl = small_case(2048, 512, seed=21)
    cfg = cfg_for(spec)
    rows = [1030, 1100, 1500, 1777, 2000, 2047]
    for factor in (12.0, 1.0):
        k = wl["k"].float()
        k[:, :, 1024:] *= factor
        w = {**wl, "k": k.to(torch.bfloat16)}
        gpu = run_prefill(cfg, w)
        res = QC.oracle_rows(w, rows, cfg=cfg)
        # Selections as everywhere (the indexer keys are unchanged) ...
        st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], None, None, cfg.k_b, cfg.r)
        assert st["exact"] == len(rows), st
        # ... outputs within the bound of the kernel's two bf16 roundings: P for
        # the PV product (2^-9 of each weight, so at most 2^-9 max|v| in o) and
        # o itself (half an ulp, 2^-9 |o| <= 2^-9 max|v|).  With the keys scaled
        # a row's softmax is dominated by a token or two and |o| nears max|v|,
        # beyond the fixed tolerance meant for averaging softmaxes.
        v = QC.bf16_to_np32(w["v"][0]).astype(np.float64)
        for n, j in enumerate(rows):
            toks = O.token_set(j, gpu["idx"][0][j][:int(gpu["count"][0][j])].astype(np.int64), cfg.r)
            vmax = np.abs(v[:, toks]).max()
            err = np.abs(gpu["out"][0][j] - res["out"][n]).max()
            assert err <= 2.0 ** -8 * vmax + 1e-4, (factor, j, err, vmax)
            assert np.abs(gpu["lse"][0][j] - res["lse"][n]).max() <= 1e-3 * max(1.0, factor)


def test_exact_ties_take_lowest_block_ids():
    """All-zero indexer keys: every score is 0, so the first k_B blocks win."""
    spec, wl = small_case(300, 64)
    wl["k_idx"].zero_()
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    for j in range(300):
        c = O.visible_blocks(j, 4)
        want = np.arange(min(c, cfg.k_b))
        np.testing.assert_array_equal(gpu["idx"][0, j, :len(want)], want)


@pytest.mark.parametrize("group,seed", [(3, 21), (40, 22)])
def test_tied_key_groups_keep_their_lowest_blocks(group, seed):
    """Indexer keys equal over groups of consecutive blocks, and zero in the
    rotated dims, so that blocks of one group score exactly alike at every
    query position.  A row that keeps part of a group must keep the group's
    lowest block ids (research-hub notes, Key ideas, top-k_B bullet; ties go to
    the lower block id).  Groups of 3 leave a short tied run at the k_B-th
    score; groups of 40 leave a tied run longer than a warp."""
    spec, wl = small_case(8192, 512, seed=seed)
    cfg = cfg_for(spec)
    g = torch.Generator(device="cpu").manual_seed(seed)
    nb = spec.n // spec.r
    gv = torch.randn((nb + group - 1) // group, 64, generator=g)
    keys = torch.zeros(spec.n, 128)
    keys[:, 64:] = gv.repeat_interleave(group, 0)[:nb].repeat_interleave(spec.r, 0)
    wl["k_idx"][0] = keys.to(torch.bfloat16).to(DEV)
    gpu = run_prefill(cfg, wl)
    selecting = spec.n - spec.r * (cfg.k_b + 1) + 1  # rows with c > k_B
    assert gpu["fallback_rows"] < selecting // 2  # most rows went through the entry buffers
    split = 0
    for i in range(spec.n):
        sel = gpu["idx"][0, i, :gpu["count"][0, i]]
        later = sel[sel % group != 0]  # members after their group's first block
        assert np.isin(later - 1, sel).all(), i  # each keeps the member before it
        cut = ((sel + 1) % group != 0) & (sel + 1 < O.visible_blocks(i, spec.r)) & ~np.isin(sel + 1, sel)
        split += int(cut.sum())
    assert split > 0  # some rows cut a visible group at the k_B-th score
    rows = QC.sample_rows(spec.n, cfg.k_b, spec.r, [], 120, seed)
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= len(rows) - 1, st


def test_planted_block_always_selected():
    """A key block equal to a row's query direction outranks every random block."""
    spec, wl = small_case(2048, 256, seed=9)
    cfg = cfg_for(spec)
    i, blk = 1500, 100
    wl["k_idx"][0, 4 * blk:4 * blk + 4] = (wl["q_idx"][0, i, 0].float() * 4).to(torch.bfloat16)
    gpu = run_prefill(cfg, wl)
    assert blk in gpu["idx"][0, i, :gpu["count"][0, i]]
    res = QC.oracle_rows(wl, [i], cfg=cfg)
    QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, 4)


def test_unsampled_high_blocks_take_the_exact_fallback():
    """Rows that see 3072 to 4096 blocks are pilot-sampled at the first few
    block residues mod 16 (as many phases of every 16th block as reach the
    pilot's minimum sample count: two or three).  Here only blocks of residues
    12..15 score high, so those rows' thresholds come from the low scores,
    they collect more entries than their buffer holds, and the exact full-row
    fallback must select them: the result is still the oracle's."""
    spec, wl = small_case(16384, 2048, seed=11)
    cfg = cfg_for(spec)
    g = torch.Generator(device="cpu").manual_seed(11)
    d = torch.zeros(128)
    d[64:] = torch.randn(64, generator=g)  # past the rotated dims: the same at every position
    wl["q_idx"][:] = d.to(torch.bfloat16).to(DEV)  # every row and head
    nb = spec.n // spec.r
    high = (torch.arange(nb) % 16 >= 12).repeat_interleave(spec.r)
    keys = 0.1 * torch.randn(spec.n, 128, generator=g)
    keys[high] = 2 * d + 0.05 * torch.randn(int(high.sum()), 128, generator=g)
    wl["k_idx"][0] = keys.to(torch.bfloat16).to(DEV)
    gpu = run_prefill(cfg, wl)
    assert gpu["fallback_rows"] > 0  # the path under test was taken
    rows = list(range(spec.n - 16, spec.n)) + [12295, 13000, 14000, 15000, 15500]
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= len(rows) - 1, st


def test_chunked_prefill_rows_at_offset():
    """A chunk of query rows at positions 1000.. against the whole cached prefix."""
    spec, wl = small_case(2048, 512, seed=12)
    cfg = cfg_for(spec)
    lo, hi = 1000, 1400
    gpu = run_prefill(cfg, wl, q_pos0=lo, rows=slice(lo, hi))
    res = QC.oracle_rows({**wl, "q_idx": wl["q_idx"][:, lo:hi], "q": wl["q"][:, lo:hi]},
                         range(hi - lo), cfg=cfg, q_pos0=lo)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0],
                            cfg.k_b, cfg.r)
    assert st["exact"] >= 0.98 * (hi - lo)


def test_offset_chunk_across_launch_ranges():
    """A 51000-row chunk at positions 49000 .. 99999 of a 100000-token
    sequence: 1063 tiles whose positions start at the chunk's offset, launched
    as [39, 1063) then [0, 39).  Whole tiles at the seam and at both ends of
    the chunk, and sampled rows, match the oracle."""
    spec = PrefillSpec("oc", n=100000, k_tokens=2048, seed=53)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    lo, hi = 49000, 100000
    gpu = run_prefill(cfg, wl, q_pos0=lo, rows=slice(lo, hi))
    n_q = hi - lo
    rows = set(range(48)) | set(range(38 * 48, 40 * 48)) | set(range(1062 * 48, n_q))
    rows |= {int(x) for x in np.random.default_rng(53).integers(0, n_q, size=24)}
    rows = sorted(rows)
    res = QC.oracle_rows({**wl, "q_idx": wl["q_idx"][:, lo:hi], "q": wl["q"][:, lo:hi]}, rows, cfg=cfg, q_pos0=lo)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= len(rows) - 2, st


def test_rows_per_wave_and_chunks_of_it_match_the_one_call_prefill():
    """qsa_index_rows_per_wave is the indexer's tile rows times the SM count.  A
    prefill run as chunks shaped like the end-to-end pipeline's (small chunks
    first, then one wave's rows, then the rest) selects the same blocks and
    writes the same output, bit for bit, as the one-call prefill: every chunk
    of at least 64 rows takes the fused indexer, whose selection is exact
    whatever tiles the chunk makes, and each row's attention depends on that
    row alone."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    wave = qsa.qsa_index_rows_per_wave(qsa.Config())
    assert wave == 48 * sms
    assert qsa.qsa_index_rows_per_wave(qsa.Config(n_idx_heads=8)) == 24 * sms
    n = 7168 + wave + 3000
    spec = PrefillSpec("w", n=n, k_tokens=2048, seed=14, drift=True)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    one = run_prefill(cfg, wl)
    bounds = [0, 1024, 3072, 7168, 7168 + wave, n]
    nb = n // cfg.r
    kbar = torch.empty((1, nb, 128), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((1, n, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((1, n), dtype=torch.int32, device=DEV)
    out = torch.empty_like(wl["q"])
    lse = torch.empty(wl["q"].shape[:3], dtype=torch.float32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, 1, max(b - a for a, b in zip(bounds, bounds[1:])), nb),),
                     dtype=torch.uint8, device=DEV)
    fallback = 0
    for lo, hi in zip(bounds, bounds[1:]):
        q_pos = torch.full((1,), lo, dtype=torch.int64, device=DEV)
        qsa.qsa_compress_keys(cfg, wl["k_idx"], lo // cfg.r, hi // cfg.r - lo // cfg.r, kbar)
        qsa.qsa_index_topk(cfg, wl["q_idx"][:, lo:hi], kbar, q_pos, hi // cfg.r, idx[:, lo:hi], cnt[:, lo:hi], ws)
        fallback += qsa.qsa_index_topk_fallback_rows(cfg, 1, hi - lo, hi // cfg.r, ws)
        qsa.qsa_sparse_attn_prefill(cfg, wl["q"][:, lo:hi], wl["k"], wl["v"], q_pos, idx[:, lo:hi],
                                    cnt[:, lo:hi], out[:, lo:hi], lse[:, lo:hi])
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    # A row of the exact fallback is scored by another MMA instruction, whose fp32
    # sums may round differently; this workload sends no row there.
    assert one["fallback_rows"] == 0 and fallback == 0
    assert np.array_equal(cnt.cpu().numpy(), one["count"])
    assert np.array_equal(idx.cpu().numpy(), one["idx"])
    assert np.array_equal(out.float().cpu().numpy(), one["out"])
    assert np.array_equal(lse.cpu().numpy(), one["lse"])


@pytest.mark.parametrize("impl", ["auto", "tcgen05"])
def test_batched_prefill_sequences_at_different_offsets(impl):
    """Three sequences in one call, each a 500-row chunk at its own position
    (0, 1100, 2100) against its own prefix: every (sequence, row) is checked
    against the oracle run on that sequence alone, through each attention
    kernel."""
    spec = PrefillSpec("b3", n=2600, k_tokens=512, seed=51, batch=3)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    n_q, offs = 500, [0, 1100, 2100]
    q_idx = torch.stack([wl["q_idx"][b, o:o + n_q] for b, o in enumerate(offs)]).contiguous()
    q = torch.stack([wl["q"][b, o:o + n_q] for b, o in enumerate(offs)]).contiguous()
    nb = spec.n // cfg.r
    kbar = torch.empty((3, nb, 128), dtype=torch.bfloat16, device=DEV)
    qsa.qsa_compress_keys(cfg, wl["k_idx"], 0, nb, kbar)
    q_pos = torch.tensor(offs, dtype=torch.int64, device=DEV)
    idx = torch.empty((3, n_q, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((3, n_q), dtype=torch.int32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, 3, n_q, nb),), dtype=torch.uint8, device=DEV)
    qsa.qsa_index_topk(cfg, q_idx, kbar, q_pos, nb, idx, cnt, ws)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    qsa.qsa_sparse_attn_prefill(cfg, q, wl["k"], wl["v"], q_pos, idx, cnt, out, lse, impl=impl)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    rows = [0, 1, 250, 498, 499]
    exact = 0
    for b, o in enumerate(offs):
        qb, kb, vb = QC.bf16_to_np32(q[b]), QC.bf16_to_np32(wl["k"][b]), QC.bf16_to_np32(wl["v"][b])
        res = O.prefill_rows(QC.bf16_to_np32(q_idx[b]), QC.bf16_to_np(wl["k_idx"][b]), qb, kb, vb, rows, r=cfg.r,
                             k_tokens=cfg.k_tokens, q_pos0=o, rope_dims=cfg.rope_dims, rope_base=cfg.rope_base)
        st = QC.compare_prefill(res, idx[b].cpu().numpy(), cnt[b].cpu().numpy(), out[b].float().cpu().numpy(),
                                lse[b].cpu().numpy(), cfg.k_b, cfg.r, attn=(qb, kb, vb))
        exact += st["exact"]
    assert exact >= 3 * len(rows) - 1


def test_batched_prefill_across_launch_ranges():
    """Three whole 20000-row sequences in one call: 3 x 417 tiles, launched as
    the ranges [227, 1251) and [0, 227), so the seam falls inside sequence 0
    and the sequence boundaries (tiles 416 | 417 and 833 | 834) inside the
    first launch, and the first range's finalize reads its entry buffer beside
    the second launch.  Whole tiles at the seam and at every sequence's ends
    match the oracle run on that sequence alone."""
    spec = PrefillSpec("b3r", n=20000, k_tokens=2048, seed=52, batch=3)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    last = range(19968, 20000)  # local tile 416 holds 32 rows
    rows_of = {0: list(range(48)) + list(range(226 * 48, 228 * 48)) + list(last),
               1: list(range(48)) + list(last),
               2: list(range(48)) + list(last)}
    exact = total = 0
    for b, rows in rows_of.items():
        rows = sorted(set(rows) | set(QC.sample_rows(spec.n, cfg.k_b, spec.r, [], 12, 52 + b)))
        one = {k: wl[k][b:b + 1] for k in ("q_idx", "k_idx", "q", "k", "v")}
        res = QC.oracle_rows(one, rows, cfg=cfg)
        st = QC.compare_prefill(res, gpu["idx"][b], gpu["count"][b], gpu["out"][b], gpu["lse"][b], cfg.k_b, cfg.r)
        exact += st["exact"]
        total += len(rows)
    assert exact >= total - 2, (exact, total)


# ----------------------------------------------------------------------------- indexer head counts

@pytest.mark.parametrize("h_idx", [1, 2, 8])
def test_indexer_head_counts_prefill_fused_path(h_idx):
    """H indexer query heads through the fused tcgen05 indexer (n_q >= 64 rows,
    k_B <= 512): tiles of 48 tokens (24 with 8 heads), N = tokens x H."""
    spec = PrefillSpec("h", n=3000, k_tokens=512, seed=60 + h_idx, h_idx=h_idx)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    rows = list(range(0, 3000, 7)) + list(range(2040, 2060)) + [2999]
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= 0.98 * len(rows), st


def test_eight_head_prefill_across_launch_ranges():
    """8 indexer heads (24-token tiles) over 53248 rows: 2219 tiles in three
    fused launches of at most 1024 tiles, heaviest first ([1195, 2219),
    [171, 1195), [0, 171)), the finalize of the first two running beside the
    next launch from the other entry buffer.  Whole tiles on both sides of
    each seam, the first and the last tile, and sampled rows match the oracle."""
    spec = PrefillSpec("h8", n=53248, k_tokens=2048, seed=68, h_idx=8)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    tiles = [0, 170, 171, 1194, 1195, 2218]  # the last tile holds rows 53232 .. 53247 only
    rows = sorted({24 * t + j for t in tiles for j in range(24) if 24 * t + j < spec.n}
                  | set(QC.sample_rows(spec.n, cfg.k_b, spec.r, [], 40, 68)))
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= len(rows) - 2, st


@pytest.mark.parametrize("h_idx", [1, 2, 8])
def test_indexer_head_counts_scan_path(h_idx):
    """A 40-row chunk (fewer than 64 rows: the one-pass scan path, 8 / H rows per
    MMA tile) at offset 1500, and r = 2 rows of a whole prefill (k_B = 1024 >
    512: the scan path too)."""
    spec = PrefillSpec("h", n=2600, k_tokens=512, seed=70 + h_idx, h_idx=h_idx)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    lo, hi = 1500, 1540
    gpu = run_prefill(cfg, wl, q_pos0=lo, rows=slice(lo, hi))
    res = QC.oracle_rows({**wl, "q_idx": wl["q_idx"][:, lo:hi], "q": wl["q"][:, lo:hi]}, range(hi - lo), cfg=cfg,
                         q_pos0=lo)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= hi - lo - 1, st
    spec2 = PrefillSpec("h2", n=2600, k_tokens=2048, seed=80 + h_idx, h_idx=h_idx, r=2)
    wl2 = make_prefill(spec2, DEV)
    cfg2 = cfg_for(spec2)
    gpu2 = run_prefill(cfg2, wl2)
    rows = [0, 1, 2047, 2048, 2049, 2050, 2599] + list(range(100, 2600, 97))
    res2 = QC.oracle_rows(wl2, rows, cfg=cfg2)
    st2 = QC.compare_prefill(res2, gpu2["idx"][0], gpu2["count"][0], gpu2["out"][0], gpu2["lse"][0], cfg2.k_b, cfg2.r)
    assert st2["exact"] >= len(rows) - 1, st2


@pytest.mark.parametrize("h_idx,next_n", [(1, 1), (2, 3), (8, 1), (8, 3), (1, 4)])
def test_indexer_head_counts_decode(h_idx, next_n):
    """Decode with H indexer heads: the k-bar scan puts 8 / H query rows in each
    MMA tile (one new token, or next_n tokens scored in one pass)."""
    spec = DecodeSpec("dh", batch=3, ctx=5003, k_tokens=512, seed=90 + h_idx, next_n=next_n, h_idx=h_idx)
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode_multi(cfg, wl)
    exact = sum(check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse)["exact"] for bb in range(3))
    assert exact >= 3 * next_n - 1


def test_rmsnorm_variant_end_to_end():
    spec, wl = small_case(700, 128, seed=13)
    cfg = cfg_for(spec, rmsnorm=True)
    gpu = run_prefill(cfg, wl)
    res = QC.oracle_rows(wl, range(0, 700, 7), cfg=cfg)
    QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, 4)


def test_bounded_wait_timeout_reports_and_context_survives():
    """A device wait that nothing satisfies gives up after its limit (about 1 ms
    here) and reports QSA_ERR_TIMEOUT through the device error word; the
    context stays usable and the next prefill still matches the oracle."""
    assert qsa.qsa_read_device_error() == 0
    qsa.qsa_selftest_wait_timeout(2_000_000)
    assert qsa.qsa_read_device_error() == 5  # QSA_ERR_TIMEOUT
    assert qsa.qsa_read_device_error() == 0  # read and cleared
    spec, wl = small_case(512, 128, seed=41)
    cfg = cfg_for(spec)
    gpu = run_prefill(cfg, wl)
    res = QC.oracle_rows(wl, [0, 200, 511], cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= 2


def test_invalid_selection_reports_instead_of_faulting():
    spec, wl = small_case(64, 16, seed=14)
    cfg = cfg_for(spec)
    q_pos = torch.zeros((1,), dtype=torch.int64, device=DEV)
    idx = torch.full((1, 64, cfg.k_b), 10 ** 6, dtype=torch.int32, device=DEV)  # out of range ids
    cnt = torch.full((1, 64), cfg.k_b, dtype=torch.int32, device=DEV)
    out = torch.empty_like(wl["q"])
    qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], q_pos, idx, cnt, out)
    assert qsa.qsa_read_device_error() == 1  # QSA_ERR_INVALID_ARG
    assert qsa.qsa_read_device_error() == 0  # the word is cleared by the read
    assert torch.isfinite(out.float()).all()


# ----------------------------------------------------------------------------- decode

def run_decode(cfg, wl, Hq=16, Hkv=2):
    B = wl["batch"]
    dec = qsa.QsaDecode(cfg, B, wl["n_blocks"], Hq, Hkv)
    out = dec(wl["q_idx"], wl["q"][:, 0].contiguous(), wl["kbar"], wl["k"], wl["v"], wl["cache_lens"])
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    return dec.idx.view(B, -1).cpu().numpy(), dec.count.view(B).cpu().numpy(), out.float().cpu().numpy(), dec.lse.cpu().numpy()


def check_decode_seq(cfg, wl, bb, idx, cnt, out, lse):
    L = int(wl["cache_lens"][bb])
    res = O.decode_rows(QC.bf16_to_np(wl["q_idx"][bb, 0]), QC.bf16_to_np(wl["q"][bb, 0]),
                        QC.bf16_to_np(wl["kbar"][bb]), QC.bf16_to_np(wl["k"][bb]),
                        QC.bf16_to_np(wl["v"][bb]), L, r=cfg.r, k_tokens=cfg.k_tokens)
    kind = QC.check_selection_row(res["scores"][0], res["sel"][0], idx[bb], int(cnt[bb]),
                                  O.visible_blocks(L - 1, cfg.r), cfg.k_b)
    if kind == "exact":
        want_o, want_l = res["out"][0], res["lse"][0]
    else:  # a near-tie swap: the oracle's attention over the GPU's own selection
        toks = O.token_set(L - 1, idx[bb][:int(cnt[bb])].astype(np.int64), cfg.r)
        want_o, want_l = O.attend(QC.bf16_to_np(wl["q"][bb, 0]), QC.bf16_to_np32(wl["k"][bb]),
                                  QC.bf16_to_np32(wl["v"][bb]), toks, QC.default_scale(128))
    assert np.abs(out[bb] - want_o).max() <= QC.OUT_ATOL
    assert np.abs(lse[bb] - want_l).max() <= QC.LSE_ATOL
    return kind


@pytest.mark.parametrize("ctx", [2, 100, 2047, 2048, 5003])
def test_decode_small_matches_oracle(ctx):
    spec = DecodeSpec("d", batch=3, ctx=ctx, k_tokens=512, seed=21)
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode(cfg, wl)
    kinds = [check_decode_seq(cfg, wl, bb, idx, cnt, out, lse) for bb in range(3)]
    assert kinds.count("exact") >= 2


@pytest.mark.parametrize("r,ctx", [(2, 3001), (8, 5003), (16, 9001)])
def test_decode_other_block_sizes(r, ctx):
    """Decode with micro-blocks of 2, 8 and 16 tokens: the scan's count of
    visible blocks and the attention's expansion of the selected blocks and
    of the tail (up to r - 1 tokens) depend on r."""
    spec = DecodeSpec("dr", batch=3, ctx=ctx, k_tokens=512, seed=33 + r, r=r)
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode(cfg, wl)
    kinds = [check_decode_seq(cfg, wl, bb, idx, cnt, out, lse) for bb in range(3)]
    assert kinds.count("exact") >= 2


def test_decode_ragged_cache_lengths():
    """Sequences of one batch at different lengths (each its own c_i and tail)."""
    spec = DecodeSpec("d", batch=4, ctx=3000, k_tokens=256, seed=22)
    wl = make_decode(spec, DEV)
    wl["cache_lens"] = torch.tensor([3001, 17, 2050, 1203], dtype=torch.int64, device=DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode(cfg, wl)
    for bb in range(4):
        check_decode_seq(cfg, wl, bb, idx, cnt, out, lse)


def test_decode_ignores_nonfinite_workspace_contents():
    """The decode workspace holds whatever its last user left (here: NaN in every
    byte).  Short and ragged caches leave most splits empty; their partial
    outputs are never written and must not enter the combine."""
    spec = DecodeSpec("d", batch=3, ctx=9000, k_tokens=2048, seed=23)
    wl = make_decode(spec, DEV)
    wl["cache_lens"] = torch.tensor([3, 17, 9001], dtype=torch.int64, device=DEV)
    cfg = cfg_for(spec)
    B = 3
    dec = qsa.QsaDecode(cfg, B, wl["n_blocks"], 16, 2)
    dec.ws_attn.fill_(0xFF)  # 0xFFFFFFFF is a NaN in every fp32 slot
    out = dec(wl["q_idx"], wl["q"][:, 0].contiguous(), wl["kbar"], wl["k"], wl["v"], wl["cache_lens"])
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    o, lse = out.float().cpu().numpy(), dec.lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    idx, cnt = dec.idx.view(B, -1).cpu().numpy(), dec.count.view(B).cpu().numpy()
    for bb in range(B):
        check_decode_seq(cfg, wl, bb, idx, cnt, o, lse)


def test_decode_tied_and_extreme_scores_select_exactly():
    """Decode rows built to stress the top-k's first pass, which bins scores at
    1/32 octave over [2^-30, 2^34): sequence 0 has compressed keys equal over
    groups of 3 blocks and sequence 1 over groups of 40 (zero in the rotated
    dims, so a group's blocks score exactly alike and ties go to the lower block
    id), sequence 2 has all-zero keys (every score 0: the first k_B blocks win,
    through the whole-row path since 5000 blocks tie), and sequence 3 keys
    scaled by 2^-45 .. 2^40, so that its scores run past both clamped ends."""
    spec = DecodeSpec("d", batch=4, ctx=20000, k_tokens=2048, seed=24)
    wl = make_decode(spec, DEV)
    g = torch.Generator(device="cpu").manual_seed(24)
    nb = wl["n_blocks"]
    kb = torch.zeros(4, nb, 128)
    for bb, group in ((0, 3), (1, 40)):
        gv = torch.randn((nb + group - 1) // group, 64, generator=g)
        kb[bb, :, 64:] = gv.repeat_interleave(group, 0)[:nb]
    scale = torch.exp2(torch.randint(-45, 41, (nb, 1), generator=g).float())
    kb[3] = torch.randn(nb, 128, generator=g) * scale
    wl["kbar"] = kb.to(torch.bfloat16).to(DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode(cfg, wl)
    np.testing.assert_array_equal(idx[2], np.arange(cfg.k_b))
    for bb in range(4):
        assert check_decode_seq(cfg, wl, bb, idx, cnt, out, lse) == "exact", bb


@pytest.mark.slow
def test_decode_full_size_sampled_sequences():
    """The 64 x 256K decode step in the bench's launch configuration; 4 sequences checked."""
    spec = WORKLOADS["decode_256k_x64"]
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode(cfg, wl)
    for bb in (0, 17, 42, 63):
        check_decode_seq(cfg, wl, bb, idx, cnt, out, lse)


def run_decode_multi(cfg, wl, Hq=16, Hkv=2):
    """Multi-token decode step: all next_n rows of each sequence selected in one
    qsa_index_topk call, then qsa_sparse_attn_decode_multi.  Results stay on the device."""
    B, nn = wl["batch"], wl["q"].shape[1]
    q_pos = wl["cache_lens"] - nn
    idx = torch.empty((B, nn, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, nn), dtype=torch.int32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, B, nn, wl["n_blocks"]),), dtype=torch.uint8, device=DEV)
    qsa.qsa_index_topk(cfg, wl["q_idx"], wl["kbar"], q_pos, wl["n_blocks"], idx, cnt, ws)
    out = torch.empty_like(wl["q"])
    lse = torch.empty((B, nn, Hq), dtype=torch.float32, device=DEV)
    wsa = torch.empty((qsa.qsa_sparse_attn_decode_multi_workspace(cfg, B, nn, Hq, Hkv),), dtype=torch.uint8,
                      device=DEV)
    qsa.qsa_sparse_attn_decode_multi(cfg, wl["q"], wl["k"], wl["v"], wl["cache_lens"], idx, cnt, out, wsa, lse)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    return idx, cnt, out, lse


def check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse):
    """Rows j of sequence bb are tokens L - next_n + j; the oracle scores them
    against the given compressed-key cache like prefill rows at those positions."""
    L, nn = int(wl["cache_lens"][bb]), wl["q"].shape[1]
    qb, kb, vb = QC.bf16_to_np32(wl["q"][bb]), QC.bf16_to_np32(wl["k"][bb]), QC.bf16_to_np32(wl["v"][bb])
    res = O.prefill_rows(QC.bf16_to_np32(wl["q_idx"][bb]), None, qb, kb, vb, range(nn), r=cfg.r,
                         k_tokens=cfg.k_tokens, q_pos0=L - nn, rope_dims=cfg.rope_dims, rope_base=cfg.rope_base,
                         kbar=QC.bf16_to_np(wl["kbar"][bb]))
    return QC.compare_prefill(res, idx[bb].cpu().numpy(), cnt[bb].cpu().numpy(), out[bb].float().cpu().numpy(),
                              lse[bb].cpu().numpy(), cfg.k_b, cfg.r, attn=(qb, kb, vb))


@pytest.mark.parametrize("next_n,ctx", [(2, 3001), (3, 5003), (4, 4096), (4, 700)])
def test_multi_token_decode_matches_oracle(next_n, ctx):
    """next_n new tokens per sequence (the token and its draft tokens) scored in
    one pass over the compressed keys; each row keeps its own selection and tail."""
    spec = DecodeSpec("dm", batch=3, ctx=ctx, k_tokens=512, seed=31, next_n=next_n)
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode_multi(cfg, wl)
    exact = sum(check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse)["exact"] for bb in range(3))
    assert exact >= 3 * next_n - 1


@pytest.mark.parametrize("r", [2, 16])
def test_multi_token_decode_other_block_sizes(r):
    """next_n = 4 rows per sequence with micro-blocks of 2 and 16 tokens: the
    rows' visible block counts and tails differ, by row, with r."""
    spec = DecodeSpec("dmr", batch=3, ctx=6007, k_tokens=512, seed=35 + r, next_n=4, r=r)
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode_multi(cfg, wl)
    exact = sum(check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse)["exact"] for bb in range(3))
    assert exact >= 3 * 4 - 1


def test_multi_token_decode_ragged_cache_lengths():
    spec = DecodeSpec("dm", batch=3, ctx=3000, k_tokens=256, seed=32, next_n=4)
    wl = make_decode(spec, DEV)
    wl["cache_lens"] = torch.tensor([3004, 9, 1207], dtype=torch.int64, device=DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode_multi(cfg, wl)
    for bb in range(3):
        check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse)


@pytest.mark.slow
def test_multi_token_decode_1m_full_size():
    """Batch 4, next_n = 4 at a 1M-token cache, as in the bench's multi-token
    decode line; every row checked."""
    spec = WORKLOADS["decode_1m_b4_next4"]
    wl = make_decode(spec, DEV)
    cfg = cfg_for(spec)
    idx, cnt, out, lse = run_decode_multi(cfg, wl)
    exact = sum(check_decode_multi_seq(cfg, wl, bb, idx, cnt, out, lse)["exact"] for bb in range(spec.batch))
    assert exact >= spec.batch * spec.next_n - 1


@pytest.mark.slow
def test_long_context_chunk_rows_past_bitmap_range():
    """A 128-row chunk at positions 135000.. of a drift workload: every row sees
    more than 32768 blocks, so its winners are ordered by merging the sorted
    segments rather than through the block bitmap."""
    spec = PrefillSpec("long_chunk", n=135128, k_tokens=2048, seed=21, drift=True)
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    lo, hi = 135000, 135128
    assert (lo + 1) // cfg.r > 32768
    gpu = run_prefill(cfg, wl, q_pos0=lo, rows=slice(lo, hi))
    rows = [0, 1, 2, 31, 63, 64, 100, 126, 127]
    res = QC.oracle_rows({**wl, "q_idx": wl["q_idx"][:, lo:hi], "q": wl["q"][:, lo:hi]}, rows, cfg=cfg, q_pos0=lo)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0], cfg.k_b, cfg.r)
    assert st["exact"] >= len(rows) - 1, st


@pytest.mark.slow
def test_million_token_prefill_sampled_rows():
    """The 2^20-token needle workload end to end (index + attention on the GPU),
    checked on sampled rows; results stay on the device and only the sampled
    rows are copied back."""
    spec = WORKLOADS["needle_prefill_1m"]
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    n, nb = spec.n, spec.n // spec.r
    kbar = torch.empty((1, nb, 128), dtype=torch.bfloat16, device=DEV)
    qsa.qsa_compress_keys(cfg, wl["k_idx"], 0, nb, kbar)
    q_pos = torch.zeros((1,), dtype=torch.int64, device=DEV)
    idx = torch.empty((1, n, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((1, n), dtype=torch.int32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, 1, n, nb),), dtype=torch.uint8, device=DEV)
    qsa.qsa_index_topk(cfg, wl["q_idx"], kbar, q_pos, nb, idx, cnt, ws)
    del ws
    out = torch.empty_like(wl["q"])
    lse = torch.empty(wl["q"].shape[:3], dtype=torch.float32, device=DEV)
    qsa.qsa_sparse_attn_prefill(cfg, wl["q"], wl["k"], wl["v"], q_pos, idx, cnt, out, lse)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    k_idx = QC.bf16_to_np(wl["k_idx"][0])
    kb_o = O.compress_keys(k_idx, cfg.r, rope_dims=cfg.rope_dims, rope_base=cfg.rope_base)
    # Within one bf16 ulp, except where the rotation cancels to far below the
    # row's scale: there the fp32 rounding of the products (~2^-24 of the
    # operands) decides, a few 2^-20 of the row's largest entry at most.
    g = kbar[0].float().cpu().numpy().astype(np.float64)
    err = np.abs(g - kb_o)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(kb_o), 1e-30))) - 7)
    row_scale = np.abs(kb_o).max(axis=1, keepdims=True)
    assert np.all(err <= ulp + 2.0 ** -20 * row_scale), float((err / (ulp + 2.0 ** -20 * row_scale)).max())
    k, v = QC.bf16_to_np32(wl["k"][0]), QC.bf16_to_np32(wl["v"][0])
    needle_rows = [i for (_, i, _) in wl["needles"]][:16]
    rows = QC.sample_rows(n, cfg.k_b, cfg.r, needle_rows, 16, seed=spec.seed)
    exact = 0
    for i in rows:
        qi = QC.bf16_to_np32(wl["q"][0, i:i + 1])
        res = O.prefill_rows(QC.bf16_to_np32(wl["q_idx"][0, i:i + 1]), None, qi,
                             k, v, [0], r=cfg.r, k_tokens=cfg.k_tokens, q_pos0=i, rope_dims=cfg.rope_dims,
                             rope_base=cfg.rope_base, kbar=kb_o)
        st = QC.compare_prefill(res, idx[0, i:i + 1].cpu().numpy(), cnt[0, i:i + 1].cpu().numpy(),
                                out[0, i:i + 1].float().cpu().numpy(), lse[0, i:i + 1].cpu().numpy(), cfg.k_b, cfg.r,
                                attn=(qi, k, v))
        exact += st["exact"]
    assert exact >= 0.9 * len(rows), (exact, len(rows))


# ----------------------------------------------------------------------------- full-size prefill, sampled rows

@pytest.fixture(scope="module")
def prefill_128k():
    """One GPU prefill of drift_prefill_128k in the bench's launch configuration,
    shared by the tests below."""
    spec = WORKLOADS["drift_prefill_128k"]
    wl = make_prefill(spec, DEV)
    cfg = cfg_for(spec)
    return spec, cfg, wl, run_prefill(cfg, wl)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["needle_prefill_32k", "drift_prefill_128k"])
def test_large_prefill_sampled_rows(name, request):
    if name == "drift_prefill_128k":
        spec, cfg, wl, gpu = request.getfixturevalue("prefill_128k")
    else:
        spec = WORKLOADS[name]
        wl = make_prefill(spec, DEV)
        cfg = cfg_for(spec)
        gpu = run_prefill(cfg, wl)
    needle_rows = [i for (_, i, _) in wl["needles"]][:16]
    rows = QC.sample_rows(spec.n, cfg.k_b, cfg.r, needle_rows, 24, seed=spec.seed)
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0],
                            cfg.k_b, cfg.r)
    assert st["exact"] >= 0.9 * len(rows), st


# The prefill indexer works on tiles of 48 consecutive query rows and the host
# launches it over ranges of at most 1024 tiles, the last range first.  At
# n = 131072 (2731 tiles) the ranges are tiles 1707-2730, 683-1706 and 0-682.
INDEX_TILE_ROWS = 48
INDEX_TILES_PER_LAUNCH = 1024


def seam_tiles(n: int) -> list[int]:
    """First tile, the tiles on each side of every launch seam, the tile where
    rows start to choose (c_i crosses k_B = 512 at row 2047) and the last tile."""
    n_tiles = -(-n // INDEX_TILE_ROWS)
    tiles = {0, 2047 // INDEX_TILE_ROWS, n_tiles - 1}
    for t_end in range(n_tiles, 0, -INDEX_TILES_PER_LAUNCH):
        t_begin = max(0, t_end - INDEX_TILES_PER_LAUNCH)
        if t_begin > 0:
            tiles |= {t_begin - 1, t_begin}
    return sorted(tiles)


@pytest.mark.slow
def test_prefill_128k_whole_tiles_at_launch_seams(prefill_128k):
    """Every row of whole indexer tiles at 128K: the first and last tiles, the
    tile where selection starts, and the tiles on both sides of each launch
    seam; selection, output and LSE of every row against the oracle."""
    spec, cfg, wl, gpu = prefill_128k
    tiles = seam_tiles(spec.n)
    assert {682, 683, 1706, 1707, 0, 2730} <= set(tiles)
    rows = [j for t in tiles for j in range(t * INDEX_TILE_ROWS, min(spec.n, (t + 1) * INDEX_TILE_ROWS))]
    assert 32784 in rows and 81936 in rows and 131071 in rows
    res = QC.oracle_rows(wl, rows, cfg=cfg)
    st = QC.compare_prefill(res, gpu["idx"][0], gpu["count"][0], gpu["out"][0], gpu["lse"][0],
                            cfg.k_b, cfg.r)
    assert st["exact"] + st["margin"] == len(rows)
    assert st["exact"] >= 0.97 * len(rows), st
