"""Thin Python binding of the QSA C ABI (``include/qsa.h``).

Argument marshalling only: every function here checks tensor dtypes, devices and
layouts, passes raw device pointers and the current CUDA stream to the entry
point of the same name, and raises :class:`QsaError` on a non-OK status.  All
arithmetic runs in the CUDA kernels of ``libqsa.so``; there is no other code
path.  PyTorch supplies device memory (including the workspaces the library
asks for) and streams.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")

QSA_OK = 0
STATUS_NAMES = {0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED",
                3: "QSA_ERR_WORKSPACE", 4: "QSA_ERR_CUDA", 5: "QSA_ERR_TIMEOUT"}

EXPORTED = [
    "qsa_default_config", "qsa_num_selected_blocks", "qsa_compress_keys",
    "qsa_index_topk_workspace", "qsa_index_rows_per_wave", "qsa_index_topk", "qsa_index_topk_fallback_rows",
    "qsa_sparse_attn_prefill",
    "qsa_sparse_attn_prefill_impl",
    "qsa_sparse_attn_decode_workspace", "qsa_sparse_attn_decode", "qsa_sparse_attn_decode_noalloc",
    "qsa_sparse_attn_decode_multi_workspace", "qsa_sparse_attn_decode_multi",
    "qsa_selftest_wait_timeout", "qsa_status_string",
    "qsa_read_device_error", "qsa_launch_count", "qsa_version",
]


class QsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class qsa_config(ctypes.Structure):
    _fields_ = [("r", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_dims", ctypes.c_int32), ("rope_base", ctypes.c_float), ("rmsnorm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("k_tokens", ctypes.c_int32)]


@dataclass
class Config:
    """Method parameters (see ``qsa_config`` in include/qsa.h)."""
    r: int = 4
    n_idx_heads: int = 4
    head_dim: int = 128
    rope_dims: int = 64
    rope_base: float = 10000.0
    rmsnorm: bool = False
    rms_eps: float = 1e-6
    k_tokens: int = 2048

    @property
    def k_b(self) -> int:
        """Selected blocks per token, as the library computes it (qsa_num_selected_blocks)."""
        c = self.c_struct()
        k_b = int(load_library().qsa_num_selected_blocks(ctypes.byref(c)))
        if k_b <= 0:
            raise ValueError(f"invalid QSA configuration: {self}")
        return k_b

    def c_struct(self) -> qsa_config:
        return qsa_config(self.r, self.n_idx_heads, self.head_dim, self.rope_dims, self.rope_base,
                          int(bool(self.rmsnorm)), self.rms_eps, self.k_tokens)


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libqsa.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with `python -m block_sparse_long_17_b300.build`")
    lib = ctypes.CDLL(path)
    P, I64, I32, SZ, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    C = ctypes.POINTER(qsa_config)
    sig = {
        "qsa_default_config": (None, [C]),
        "qsa_num_selected_blocks": (I32, [C]),
        "qsa_compress_keys": (ctypes.c_int, [C, P, I64, I64, I64, I64, P, I64, P]),
        "qsa_index_topk_workspace": (SZ, [C, I64, I64, I64]),
        "qsa_index_rows_per_wave": (ctypes.c_int, [C, ctypes.POINTER(I64)]),
        "qsa_index_topk": (ctypes.c_int, [C, P, P, I64, P, I64, I64, I64, P, P, P, SZ, P]),
        "qsa_index_topk_fallback_rows": (ctypes.c_int, [C, I64, I64, I64, P, SZ, ctypes.POINTER(I64), P]),
        "qsa_sparse_attn_prefill": (ctypes.c_int, [C, P, P, P, I64, P, P, P, I64, I64, I32, I32, F, P, P, P]),
        "qsa_sparse_attn_prefill_impl": (ctypes.c_int, [C, P, P, P, I64, P, P, P, I64, I64, I32, I32, F, P, P,
                                                        ctypes.c_int, P]),
        "qsa_sparse_attn_decode_workspace": (SZ, [C, I64, I32, I32]),
        "qsa_sparse_attn_decode": (ctypes.c_int, [C, P, P, P, I64, P, P, P, I64, I32, I32, F, P, P, P, SZ, P]),
        "qsa_sparse_attn_decode_multi_workspace": (SZ, [C, I64, I32, I32, I32]),
        "qsa_sparse_attn_decode_multi": (ctypes.c_int, [C, P, P, P, I64, P, P, P, I64, I32, I32, I32, F, P, P, P, SZ,
                                                        P]),
        "qsa_sparse_attn_decode_noalloc": (ctypes.c_int, [C, P, P, P, I64, P, P, P, I64, I32, I32, F, P, P, P]),
        "qsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "qsa_read_device_error": (ctypes.c_int, [P]),
        "qsa_selftest_wait_timeout": (ctypes.c_int, [I64, P]),
        "qsa_launch_count": (ctypes.c_uint64, []),
        "qsa_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != QSA_OK:
        raise QsaError(fn, status)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _bf16(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")


def _i64(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.int64 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int64 tensor")


# ----------------------------------------------------------------------------- entry points

def qsa_compress_keys(cfg: Config, k_idx: torch.Tensor, first_block: int, n_blocks: int,
                      kbar: torch.Tensor, stream=None) -> None:
    """k_idx [B, L, d] bf16 -> kbar[:, first_block:first_block+n_blocks] (kbar [B, N_cap, d])."""
    _bf16(k_idx, "k_idx"); _bf16(kbar, "kbar")
    lib = load_library()
    B = k_idx.shape[0]
    c = cfg.c_struct()
    _check("qsa_compress_keys", lib.qsa_compress_keys(
        ctypes.byref(c), _ptr(k_idx), k_idx.stride(0), B, first_block, n_blocks, _ptr(kbar),
        kbar.stride(0), _stream(stream)))


def qsa_index_topk_workspace(cfg: Config, B: int, n_q: int, n_blocks_max: int) -> int:
    c = cfg.c_struct()
    return int(load_library().qsa_index_topk_workspace(ctypes.byref(c), B, n_q, n_blocks_max))


def qsa_index_topk(cfg: Config, q_idx: torch.Tensor, kbar: torch.Tensor, q_pos: torch.Tensor,
                   n_blocks_max: int, idx: torch.Tensor, count: torch.Tensor, ws: torch.Tensor,
                   stream=None) -> None:
    """q_idx [B, n_q, n_idx_heads, d] bf16; kbar [B, N_cap, d] bf16; q_pos [B] int64 (device);
    idx [B, n_q, k_B] int32; count [B, n_q] int32; ws: uint8 workspace."""
    _bf16(q_idx, "q_idx"); _bf16(kbar, "kbar"); _i64(q_pos, "q_pos")
    for t, nm in ((idx, "idx"), (count, "count")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous CUDA int32 tensor")
    B, n_q = q_idx.shape[0], q_idx.shape[1]
    c = cfg.c_struct()
    _check("qsa_index_topk", load_library().qsa_index_topk(
        ctypes.byref(c), _ptr(q_idx), _ptr(kbar), kbar.stride(0), _ptr(q_pos), B, n_q, n_blocks_max,
        _ptr(idx), _ptr(count), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def qsa_index_rows_per_wave(cfg: Config) -> int:
    """Query rows one wave of the prefill indexer covers on the current device
    (a chunk-size hint for chunked prefill)."""
    c = cfg.c_struct()
    rows = ctypes.c_int64(0)
    _check("qsa_index_rows_per_wave", load_library().qsa_index_rows_per_wave(ctypes.byref(c), ctypes.byref(rows)))
    return int(rows.value)


def qsa_index_topk_fallback_rows(cfg: Config, B: int, n_q: int, n_blocks_max: int, ws: torch.Tensor,
                                 stream=None) -> int:
    """Rows of the last qsa_index_topk call on `ws` (same sizes) that its exact
    full-row fallback selected; waits for the stream."""
    c = cfg.c_struct()
    rows = ctypes.c_int64(0)
    _check("qsa_index_topk_fallback_rows", load_library().qsa_index_topk_fallback_rows(
        ctypes.byref(c), B, n_q, n_blocks_max, _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(rows),
        _stream(stream)))
    return int(rows.value)


# Kernel choice of qsa_sparse_attn_prefill_impl (qsa_attn_impl in include/qsa.h).
QSA_ATTN_AUTO, QSA_ATTN_TCGEN05, QSA_ATTN_MMA_SYNC = 0, 1, 2
ATTN_IMPLS = {"auto": QSA_ATTN_AUTO, "tcgen05": QSA_ATTN_TCGEN05, "mma_sync": QSA_ATTN_MMA_SYNC}


def qsa_sparse_attn_prefill(cfg: Config, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            q_pos: torch.Tensor, idx: torch.Tensor, count: torch.Tensor,
                            out: torch.Tensor, lse: torch.Tensor | None = None,
                            scale: float | None = None, stream=None, impl: str = "auto") -> None:
    """q [B, n_q, Hq, d]; k, v [B, Hkv, L_cap, d]; out like q; lse [B, n_q, Hq] fp32 or None.
    impl: "auto" (the library's choice), "tcgen05" or "mma_sync"."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _bf16(t, nm)
    _i64(q_pos, "q_pos")
    B, n_q, Hq, d = q.shape
    Hkv, L_cap = k.shape[1], k.shape[2]
    scale = 0.0 if scale is None else scale  # <= 0: the library's default 1/sqrt(head_dim)
    c = cfg.c_struct()
    _check("qsa_sparse_attn_prefill_impl", load_library().qsa_sparse_attn_prefill_impl(
        ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), L_cap, _ptr(q_pos), _ptr(idx), _ptr(count), B,
        n_q, Hq, Hkv, scale, _ptr(out), _ptr(lse), ATTN_IMPLS[impl], _stream(stream)))


def qsa_sparse_attn_decode_workspace(cfg: Config, B: int, Hq: int, Hkv: int) -> int:
    c = cfg.c_struct()
    return int(load_library().qsa_sparse_attn_decode_workspace(ctypes.byref(c), B, Hq, Hkv))


def qsa_sparse_attn_decode(cfg: Config, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, cache_len: torch.Tensor, idx: torch.Tensor,
                           count: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                           lse: torch.Tensor | None = None, scale: float | None = None,
                           stream=None) -> None:
    """q [B, Hq, d]; caches [B, Hkv, L_cap, d]; cache_len [B] int64 (device); idx [B, k_B]."""
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _bf16(t, nm)
    _i64(cache_len, "cache_len")
    B, Hq, d = q.shape
    Hkv, L_cap = k_cache.shape[1], k_cache.shape[2]
    scale = 0.0 if scale is None else scale  # <= 0: the library's default 1/sqrt(head_dim)
    c = cfg.c_struct()
    _check("qsa_sparse_attn_decode", load_library().qsa_sparse_attn_decode(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), L_cap, _ptr(cache_len), _ptr(idx),
        _ptr(count), B, Hq, Hkv, scale, _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def qsa_sparse_attn_decode_multi_workspace(cfg: Config, B: int, n_q: int, Hq: int, Hkv: int) -> int:
    c = cfg.c_struct()
    return int(load_library().qsa_sparse_attn_decode_multi_workspace(ctypes.byref(c), B, n_q, Hq, Hkv))


def qsa_sparse_attn_decode_multi(cfg: Config, q: torch.Tensor, k_cache: torch.Tensor,
                                 v_cache: torch.Tensor, cache_len: torch.Tensor, idx: torch.Tensor,
                                 count: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                                 lse: torch.Tensor | None = None, scale: float | None = None,
                                 stream=None) -> None:
    """q [B, n_q, Hq, d]; caches [B, Hkv, L_cap, d]; cache_len [B] int64 (device, includes
    the n_q new tokens); idx [B, n_q, k_B]; count [B, n_q]; out like q."""
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _bf16(t, nm)
    _i64(cache_len, "cache_len")
    B, n_q, Hq, d = q.shape
    Hkv, L_cap = k_cache.shape[1], k_cache.shape[2]
    scale = 0.0 if scale is None else scale  # <= 0: the library's default 1/sqrt(head_dim)
    c = cfg.c_struct()
    _check("qsa_sparse_attn_decode_multi", load_library().qsa_sparse_attn_decode_multi(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), L_cap, _ptr(cache_len), _ptr(idx),
        _ptr(count), B, n_q, Hq, Hkv, scale, _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 << 20  # QSA_NOALLOC_SCRATCH_BYTES in include/qsa.h


def qsa_sparse_attn_decode_noalloc(cfg: Config, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, cache_len: torch.Tensor, idx: torch.Tensor,
                                   count: torch.Tensor, out: torch.Tensor,
                                   lse: torch.Tensor | None = None, scale: float | None = None,
                                   stream=None) -> None:
    """qsa_sparse_attn_decode without a workspace: the library keeps the split
    partials in its own static device array, for callers that cannot allocate.
    Calls that may overlap on the GPU share that array and must be ordered."""
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _bf16(t, nm)
    _i64(cache_len, "cache_len")
    B, Hq, d = q.shape
    Hkv, L_cap = k_cache.shape[1], k_cache.shape[2]
    scale = 0.0 if scale is None else scale  # <= 0: the library's default 1/sqrt(head_dim)
    c = cfg.c_struct()
    _check("qsa_sparse_attn_decode_noalloc", load_library().qsa_sparse_attn_decode_noalloc(
        ctypes.byref(c), _ptr(q), _ptr(k_cache), _ptr(v_cache), L_cap, _ptr(cache_len), _ptr(idx),
        _ptr(count), B, Hq, Hkv, scale, _ptr(out), _ptr(lse), _stream(stream)))


def qsa_read_device_error(stream=None) -> int:
    return int(load_library().qsa_read_device_error(_stream(stream)))


def qsa_selftest_wait_timeout(limit_cycles: int, stream=None) -> None:
    """Diagnostic: a bounded device wait on a barrier nothing arrives on; the
    timeout then shows in qsa_read_device_error() as QSA_ERR_TIMEOUT."""
    _check("qsa_selftest_wait_timeout", load_library().qsa_selftest_wait_timeout(int(limit_cycles), _stream(stream)))


def qsa_launch_count() -> int:
    return int(load_library().qsa_launch_count())


def qsa_version() -> str:
    return load_library().qsa_version().decode()


# ----------------------------------------------------------------------------- whole path

class QsaPrefill:
    """One QSA layer's prefill over resident device tensors: compress keys, score +
    select blocks, sparse attention.  Buffers are allocated once (by torch) and
    reused across calls of the same shape."""

    def __init__(self, cfg: Config, B: int, n: int, Hq: int, Hkv: int, device="cuda"):
        self.cfg, self.B, self.n, self.Hq, self.Hkv = cfg, B, n, Hq, Hkv
        nb = n // cfg.r
        self.n_blocks = nb
        self.kbar = torch.empty((B, max(nb, 1), cfg.head_dim), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((B, n, cfg.k_b), dtype=torch.int32, device=device)
        self.count = torch.empty((B, n), dtype=torch.int32, device=device)
        self.q_pos = torch.zeros((B,), dtype=torch.int64, device=device)
        ws = qsa_index_topk_workspace(cfg, B, n, nb)
        self.ws = torch.empty((ws,), dtype=torch.uint8, device=device)
        self.out = torch.empty((B, n, Hq, cfg.head_dim), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, n, Hq), dtype=torch.float32, device=device)

    def __call__(self, q_idx, k_idx, q, k, v, stream=None, with_lse=True):
        qsa_compress_keys(self.cfg, k_idx, 0, self.n_blocks, self.kbar, stream)
        qsa_index_topk(self.cfg, q_idx, self.kbar, self.q_pos, self.n_blocks, self.idx, self.count,
                       self.ws, stream)
        qsa_sparse_attn_prefill(self.cfg, q, k, v, self.q_pos, self.idx, self.count, self.out,
                                self.lse if with_lse else None, stream=stream)
        return self.out

    def fallback_rows(self, stream=None) -> int:
        """Rows of the last call that the indexer's exact full-row fallback selected."""
        return qsa_index_topk_fallback_rows(self.cfg, self.B, self.n, self.n_blocks, self.ws, stream)


class QsaDecode:
    """One decode step for B sequences against a resident compressed-key cache and
    KV cache: score + select blocks for the new token, then sparse attention."""

    def __init__(self, cfg: Config, B: int, n_blocks_max: int, Hq: int, Hkv: int, device="cuda"):
        self.cfg, self.B, self.n_blocks_max = cfg, B, n_blocks_max
        self.idx = torch.empty((B, 1, cfg.k_b), dtype=torch.int32, device=device)
        self.count = torch.empty((B, 1), dtype=torch.int32, device=device)
        self.ws_idx = torch.empty((qsa_index_topk_workspace(cfg, B, 1, n_blocks_max),),
                                  dtype=torch.uint8, device=device)
        self.ws_attn = torch.empty((qsa_sparse_attn_decode_workspace(cfg, B, Hq, Hkv),),
                                   dtype=torch.uint8, device=device)
        self.out = torch.empty((B, Hq, cfg.head_dim), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=device)

    def __call__(self, q_idx, q, kbar, k_cache, v_cache, cache_len, stream=None, with_lse=True):
        """q_idx [B, 1, n_idx_heads, d]; q [B, Hq, d]; cache_len [B] int64 including the new token."""
        q_pos = cache_len - 1
        qsa_index_topk(self.cfg, q_idx, kbar, q_pos, self.n_blocks_max, self.idx, self.count,
                       self.ws_idx, stream)
        qsa_sparse_attn_decode(self.cfg, q, k_cache, v_cache, cache_len, self.idx.view(self.B, -1),
                               self.count.view(self.B), self.out, self.ws_attn,
                               self.lse if with_lse else None, stream=stream)
        return self.out
