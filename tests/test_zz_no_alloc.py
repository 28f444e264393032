"""qsa_sparse_attn_decode_noalloc against qsa_sparse_attn_decode.

The no-alloc entry point serves callers that cannot allocate device memory (it
keeps the split partials in the library's own static device array instead of a
caller workspace).  It must give the same decode results as the regular entry
point, including on back-to-back calls, where the second call finds the first
call's partials still in the shared array.  This file is named to be collected
last, so a failing run that stops at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_long_17_b300 import qsa
from block_sparse_long_17_b300.workloads import DecodeSpec, make_decode
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_case(seed, batch, ctx, cache_lens=None):
    spec = DecodeSpec("noalloc", batch=batch, ctx=ctx, k_tokens=2048, seed=seed)
    wl = make_decode(spec, DEV)
    if cache_lens is not None:
        wl["cache_lens"] = torch.tensor(cache_lens, dtype=torch.int64, device=DEV)
    cfg = qsa.Config(k_tokens=spec.k_tokens)
    # Block selection through the regular indexer entry point (its workspace is
    # the test's own; only the attention step is under test here).
    B = batch
    idx = torch.empty((B, 1, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, 1), dtype=torch.int32, device=DEV)
    ws = torch.empty((qsa.qsa_index_topk_workspace(cfg, B, 1, wl["n_blocks"]),), dtype=torch.uint8, device=DEV)
    qsa.qsa_index_topk(cfg, wl["q_idx"], wl["kbar"], wl["cache_lens"] - 1, wl["n_blocks"], idx, cnt, ws)
    return cfg, wl, idx.view(B, -1), cnt.view(B)


def _both(cfg, wl, idx, cnt):
    B = wl["batch"]
    q = wl["q"][:, 0].contiguous()
    ref = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=DEV)
    ref_lse = torch.empty((B, 16), dtype=torch.float32, device=DEV)
    ws = torch.empty((qsa.qsa_sparse_attn_decode_workspace(cfg, B, 16, 2),), dtype=torch.uint8, device=DEV)
    qsa.qsa_sparse_attn_decode(cfg, q, wl["k"], wl["v"], wl["cache_lens"], idx, cnt, ref, ws, ref_lse)
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_lse)
    qsa.qsa_sparse_attn_decode_noalloc(cfg, q, wl["k"], wl["v"], wl["cache_lens"], idx, cnt, out, lse)
    torch.cuda.synchronize()
    assert qsa.qsa_read_device_error() == 0
    return ref.float().cpu().numpy(), ref_lse.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    # Call 1: 8 sequences with 40000 cached tokens.
    cfg, wl, idx, cnt = _decode_case(31, 8, 40000)
    ref, ref_lse, out, lse = _both(cfg, wl, idx, cnt)
    assert np.abs(out - ref).max() <= QC.OUT_ATOL
    assert np.abs(lse - ref_lse).max() <= QC.LSE_ATOL
    # Call 2, right after: other data, ragged and shorter caches, so fewer splits
    # are live than the first call left in the shared array.
    cfg2, wl2, idx2, cnt2 = _decode_case(32, 5, 9000, cache_lens=[9001, 17, 2051, 5000, 3])
    ref2, ref_lse2, out2, lse2 = _both(cfg2, wl2, idx2, cnt2)
    assert np.abs(out2 - ref2).max() <= QC.OUT_ATOL
    assert np.abs(lse2 - ref_lse2).max() <= QC.LSE_ATOL


def test_noalloc_rejects_batches_beyond_its_scratch():
    cfg = qsa.Config()
    B = 4096  # needs far more than the fixed scratch at K = 2048, r = 4
    assert qsa.qsa_sparse_attn_decode_workspace(cfg, B, 16, 2) > qsa.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, 16, 128), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((B, 2, 8, 128), dtype=torch.bfloat16, device=DEV)
    cl = torch.full((B,), 8, dtype=torch.int64, device=DEV)
    idx = torch.zeros((B, cfg.k_b), dtype=torch.int32, device=DEV)
    cnt = torch.zeros((B,), dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    with pytest.raises(qsa.QsaError) as ei:
        qsa.qsa_sparse_attn_decode_noalloc(cfg, q, kc, kc, cl, idx, cnt, out)
    assert ei.value.status == 3  # QSA_ERR_WORKSPACE


def test_noalloc_ignores_stale_nonfinite_partials():
    """The shared array keeps what the last call left in it.  A first call whose
    V holds Inf leaves non-finite partials behind; the next call, a ragged batch
    with short caches (so that many of its splits are empty), must still match
    the regular entry point and be finite."""
    cfg, wl, idx, cnt = _decode_case(33, 8, 40000)
    wl["v"][:, :, :4096] = float("inf")
    q = wl["q"][:, 0].contiguous()
    out = torch.empty((8, 16, 128), dtype=torch.bfloat16, device=DEV)
    qsa.qsa_sparse_attn_decode_noalloc(cfg, q, wl["k"], wl["v"], wl["cache_lens"], idx, cnt, out)
    torch.cuda.synchronize()
    assert not torch.isfinite(out.float()).all()  # the poison reached the partials
    cfg2, wl2, idx2, cnt2 = _decode_case(34, 5, 9000, cache_lens=[3, 17, 9001, 40, 2051])
    ref, ref_lse, out2, lse2 = _both(cfg2, wl2, idx2, cnt2)
    assert np.isfinite(out2).all() and np.isfinite(lse2).all()
    assert np.abs(out2 - ref).max() <= QC.OUT_ATOL
    assert np.abs(lse2 - ref_lse).max() <= QC.LSE_ATOL


def test_noalloc_rejects_a_stream_of_another_device():
    """The scratch array is per device: a tensor that is not device memory of the
    current device is refused before any launch."""
    cfg = qsa.Config()
    q = torch.zeros((2, 16, 128), dtype=torch.bfloat16)  # host memory
    lib = qsa.load_library()
    c = cfg.c_struct()
    fake = torch.zeros(16, dtype=torch.int64, device=DEV)
    st = lib.qsa_sparse_attn_decode_noalloc(ctypes.byref(c), q.data_ptr(), fake.data_ptr(), fake.data_ptr(), 8,
                                            fake.data_ptr(), fake.data_ptr(), fake.data_ptr(), 2, 16, 2, 0.0,
                                            fake.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == 1  # QSA_ERR_INVALID_ARG
    assert qsa.qsa_read_device_error() == 0
