"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/qsa.h, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from block_sparse_long_17_b300 import build, qsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qsa.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert header_functions() == sorted(qsa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_library_links_no_torch(lib):
    with open(qsa.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"libtorch" not in blob and b"libc10" not in blob


def test_default_config_and_k_b(lib):
    c = qsa.qsa_config()
    lib.qsa_default_config(ctypes.byref(c))
    assert (c.r, c.n_idx_heads, c.head_dim, c.rope_dims, c.rmsnorm, c.k_tokens) == (4, 4, 128, 64, 0, 2048)
    assert c.rope_base == 10000.0
    assert lib.qsa_num_selected_blocks(ctypes.byref(c)) == 512
    c.k_tokens = 513
    assert lib.qsa_num_selected_blocks(ctypes.byref(c)) == 129  # ceil(513 / 4)
    assert lib.qsa_num_selected_blocks(None) == 0


def test_status_strings_and_version(lib):
    assert lib.qsa_status_string(0) == b"QSA_OK"
    assert lib.qsa_status_string(5) == b"QSA_ERR_TIMEOUT"
    assert lib.qsa_version().startswith(b"qsa-b300")


def _cfg(**kw):
    c = qsa.Config(**kw)
    return c.c_struct()


@pytest.mark.parametrize("field,value,status", [
    ("r", 3, 1), ("r", 0, 1), ("r", 32, 1), ("rope_dims", 63, 1), ("rope_dims", 130, 1),
    ("rope_base", -1.0, 1), ("k_tokens", 0, 1), ("rmsnorm", 2, 1),
    ("head_dim", 64, 2), ("n_idx_heads", 3, 2), ("n_idx_heads", 16, 2), ("n_idx_heads", 0, 2),
])
def test_invalid_config_rejected_before_launch(lib, field, value, status):
    c = _cfg()
    setattr(c, field, value)
    fake = ctypes.c_void_p(256)  # never dereferenced: the check fails first
    st = lib.qsa_compress_keys(ctypes.byref(c), fake, 0, 1, 0, 1, fake, 0, None)
    assert st == status
    assert lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 16, 4) == 0


def test_null_and_negative_arguments(lib):
    c = _cfg()
    fake = ctypes.c_void_p(256)
    # null pointers
    assert lib.qsa_compress_keys(ctypes.byref(c), None, 0, 1, 0, 1, fake, 0, None) == 1
    assert lib.qsa_index_topk(ctypes.byref(c), fake, fake, 0, None, 1, 4, 1, fake, fake, fake, 1 << 20, None) == 1
    # negative sizes
    assert lib.qsa_compress_keys(ctypes.byref(c), fake, 0, -1, 0, 1, fake, 0, None) == 1
    assert lib.qsa_sparse_attn_prefill(ctypes.byref(c), fake, fake, fake, 8, fake, fake, fake, 1, -1,
                                       16, 2, 0.1, fake, None, None) == 1
    # empty work is a no-op that succeeds
    assert lib.qsa_compress_keys(ctypes.byref(c), None, 0, 0, 0, 0, None, 0, None) == 0
    assert lib.qsa_index_topk(ctypes.byref(c), None, None, 0, None, 1, 0, 0, None, None, None, 0, None) == 0
    # Hq not a multiple of Hkv
    assert lib.qsa_sparse_attn_prefill(ctypes.byref(c), fake, fake, fake, 8, fake, fake, fake, 1, 1,
                                       12, 5, 0.1, fake, None, None) == 2
    # misaligned tensor pointer
    odd = ctypes.c_void_p(258)
    assert lib.qsa_compress_keys(ctypes.byref(c), odd, 0, 1, 0, 1, fake, 0, None) == 1
    # K/V buffers longer than 32-bit token indices reach
    big = 1 << 31
    assert lib.qsa_sparse_attn_prefill(ctypes.byref(c), fake, fake, fake, big, fake, fake, fake, 1, 1,
                                       16, 2, 0.1, fake, None, None) == 2
    assert lib.qsa_sparse_attn_decode(ctypes.byref(c), fake, fake, fake, big, fake, fake, fake, 1, 16, 2, 0.1,
                                      fake, None, fake, 1 << 30, None) == 2
    assert lib.qsa_sparse_attn_decode_multi(ctypes.byref(c), fake, fake, fake, big, fake, fake, fake, 1, 2, 16, 2,
                                            0.1, fake, None, fake, 1 << 30, None) == 2


def test_workspace_sizes_and_checks(lib):
    c = _cfg()
    ws = lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 2048, 512)
    assert ws >= 2048 * 4 * 128 * 2  # at least the rotated queries
    assert ws % 256 == 0
    fake = ctypes.c_void_p(256)
    # too small a workspace is reported as such, before any launch
    assert lib.qsa_index_topk(ctypes.byref(c), fake, fake, 0, fake, 1, 2048, 512, fake, fake, fake,
                              ws - 1, None) == 3
    # workspace not 256-byte aligned
    assert lib.qsa_index_topk(ctypes.byref(c), fake, fake, 0, fake, 1, 2048, 512, fake, fake,
                              ctypes.c_void_p(272), ws, None) == 1
    wd = lib.qsa_sparse_attn_decode_workspace(ctypes.byref(c), 64, 16, 2)
    assert wd > 0 and wd % 256 == 0
    assert lib.qsa_sparse_attn_decode(ctypes.byref(c), fake, fake, fake, 16, fake, fake, fake, 64, 16, 2,
                                      0.1, fake, None, fake, wd - 1, None) == 3


def test_fallback_rows_checks_before_any_cuda_call(lib):
    c = _cfg()
    fake = ctypes.c_void_p(256)
    rows = ctypes.c_int64(-7)
    ws = lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 2048, 512)
    # no output pointer, or too small a workspace: rejected on the host
    assert lib.qsa_index_topk_fallback_rows(ctypes.byref(c), 1, 2048, 512, fake, ws, None, None) == 1
    assert lib.qsa_index_topk_fallback_rows(ctypes.byref(c), 1, 2048, 512, fake, ws - 1,
                                            ctypes.byref(rows), None) == 3
    # empty work and the one-pass scan path (fewer than 64 rows) report 0 without a launch
    assert lib.qsa_index_topk_fallback_rows(ctypes.byref(c), 1, 0, 512, None, 0, ctypes.byref(rows), None) == 0
    assert rows.value == 0
    rows.value = -7
    ws_scan = lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 4, 512)
    assert lib.qsa_index_topk_fallback_rows(ctypes.byref(c), 1, 4, 512, fake, ws_scan,
                                            ctypes.byref(rows), None) == 0
    assert rows.value == 0


@pytest.mark.parametrize("h", [1, 2, 4, 8])
def test_indexer_head_counts_are_accepted(lib, h):
    """1, 2, 4 or 8 indexer query heads: the workspace grows with the rotated
    queries (n_q x h x 128 bf16) and nothing is refused on the host."""
    c = _cfg(n_idx_heads=h)
    ws = lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 2048, 512)
    assert ws >= 2048 * h * 128 * 2
    assert lib.qsa_index_topk_workspace(ctypes.byref(c), 1, 3, 512) >= 3 * h * 128 * 2


def test_attention_kernel_choice_checked_on_the_host(lib):
    """qsa_sparse_attn_prefill_impl: a kernel choice outside the enum is an
    invalid argument and the tcgen05 kernel's shape limits are checked before
    any launch (no device pointer is touched)."""
    c = _cfg()
    fake = ctypes.c_void_p(256)
    args = (ctypes.byref(c), fake, fake, fake, 8, fake, fake, fake, 1, 4, 16, 2, 0.0, fake, None)
    assert lib.qsa_sparse_attn_prefill_impl(*args, 7, None) == 1
    assert lib.qsa_sparse_attn_prefill_impl(*args, -1, None) == 1
    c12 = _cfg()
    bad = (ctypes.byref(c12), fake, fake, fake, 8, fake, fake, fake, 1, 4, 12, 4, 0.0, fake, None)
    assert lib.qsa_sparse_attn_prefill_impl(*bad, 1, None) == 2   # tcgen05: 3 query heads per kv head
    c2 = _cfg(r=2)
    r2 = (ctypes.byref(c2), fake, fake, fake, 8, fake, fake, fake, 1, 4, 16, 2, 0.0, fake, None)
    assert lib.qsa_sparse_attn_prefill_impl(*r2, 1, None) == 2     # tcgen05: r = 2
    # empty work succeeds without a launch
    assert lib.qsa_sparse_attn_prefill_impl(ctypes.byref(c), None, None, None, 8, None, None, None, 0, 0, 16, 2,
                                            0.0, None, None, 1, None) == 0


def test_rows_per_wave_checks_arguments(lib):
    """qsa_index_rows_per_wave: bad arguments are refused before the device is
    queried; without a GPU the query itself reports QSA_ERR_CUDA and leaves the
    output untouched."""
    import torch
    c = _cfg()
    rows = ctypes.c_int64(-7)
    assert lib.qsa_index_rows_per_wave(None, ctypes.byref(rows)) == 1
    assert lib.qsa_index_rows_per_wave(ctypes.byref(c), None) == 1
    bad = _cfg()
    bad.n_idx_heads = 3
    assert lib.qsa_index_rows_per_wave(ctypes.byref(bad), ctypes.byref(rows)) == 2
    assert rows.value == -7
    if not torch.cuda.is_available():
        assert lib.qsa_index_rows_per_wave(ctypes.byref(c), ctypes.byref(rows)) == 4
        assert rows.value == -7
