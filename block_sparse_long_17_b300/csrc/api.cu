// C ABI of the QSA library: host-side argument checks, workspace layout and
// kernel dispatch.  The kernel sources are compiled into this one translation
// unit so that they share the device error word without relocatable device code.
#include <cmath>

#include "common.cuh"

#include "compress.cu"
#include "index_scan.cu"
#include "topk_select.cu"
#include "index_fused.cu"
#include "sparse_attn.cu"
#include "sparse_attn_tc.cu"

namespace qsa {
namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kScoreChunkBytes = int64_t(1) << 30;  // per-launch score rows, prefill path

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_config(const qsa_config* c) {
  if (c == nullptr) return false;
  if (c->r < 1 || c->r > 16 || (c->r & (c->r - 1)) != 0) return false;
  if (c->rope_dims < 0 || c->rope_dims > c->head_dim || (c->rope_dims & 1)) return false;
  if (!(c->rope_base > 0.f) || !std::isfinite(c->rope_base)) return false;
  if (c->rmsnorm != 0 && c->rmsnorm != 1) return false;
  if (c->rmsnorm && !(c->rms_eps > 0.f)) return false;
  if (c->k_tokens < 1) return false;
  return true;
}

// Shapes the kernels are built for (checked after valid_config).
bool supported_config(const qsa_config* c) {
  const int h = c->n_idx_heads;
  return (h == 1 || h == 2 || h == 4 || h == 8) && c->head_dim == kHeadDim;
}

qsa_status check_config(const qsa_config* c) {
  if (!valid_config(c)) return QSA_ERR_INVALID_ARG;
  if (!supported_config(c)) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

int k_blocks(const qsa_config* c) { return (c->k_tokens + c->r - 1) / c->r; }

// Longest K/V buffer the attention kernels take: they index its tokens with
// 32-bit integers.
constexpr int64_t kMaxLCap = 0x7fffffff;

// Softmax scale of the attention calls: a caller value <= 0 selects the usual
// 1 / sqrt(head_dim).
float softmax_scale(const qsa_config* c, float scale) {
  return scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)c->head_dim));
}

RopeParams rope_params(const qsa_config* c) {
  RopeParams p{};
  p.half = c->rope_dims / 2;
  for (int j = 0; j < p.half; ++j)
    p.theta[j] = std::pow((double)c->rope_base, -2.0 * (double)j / (double)c->rope_dims);
  return p;
}

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

struct IndexLayout {
  bool fused;
  size_t qt_off, s_off, total;
  int64_t s_stride, rows_per_launch;
};

// Workspace: rotated queries, then either the per-CTA selection buffers of the
// fused indexer (prefill) or one launch's worth of score rows (decode scan).
IndexLayout index_layout(int64_t B, int64_t n_q, int64_t n_blocks_max, int k_b, int H) {
  IndexLayout L{};
  const int64_t rows = B * n_q;
  L.fused = use_fused_indexer(n_q, k_b);
  L.qt_off = 0;
  L.s_off = align_up((size_t)rows * H * kHeadDim * sizeof(__nv_bfloat16));
  if (L.fused) {
    L.total = L.s_off + align_up(fused_layout(B, n_q, n_blocks_max, H).total);
    return L;
  }
  L.s_stride = (n_blocks_max + 3) / 4 * 4;
  if (L.s_stride < 4) L.s_stride = 4;
  int64_t per = kScoreChunkBytes / (L.s_stride * (int64_t)sizeof(float));
  if (per < 1) per = 1;
  L.rows_per_launch = rows < per ? rows : per;
  if (L.rows_per_launch < 1) L.rows_per_launch = 1;
  L.total = L.s_off + align_up((size_t)L.rows_per_launch * L.s_stride * sizeof(float));
  return L;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

void qsa_default_config(qsa_config* cfg) {
  if (cfg == nullptr) return;
  cfg->r = 4;
  cfg->n_idx_heads = 4;
  cfg->head_dim = 128;
  cfg->rope_dims = 64;
  cfg->rope_base = 10000.f;
  cfg->rmsnorm = 0;
  cfg->rms_eps = 1e-6f;
  cfg->k_tokens = 2048;
}

int32_t qsa_num_selected_blocks(const qsa_config* cfg) {
  if (!valid_config(cfg)) return 0;
  return k_blocks(cfg);
}

qsa_status qsa_compress_keys(const qsa_config* cfg, const void* k_idx, int64_t k_idx_stride_b,
                             int64_t B, int64_t first_block, int64_t n_blocks, void* kbar,
                             int64_t kbar_stride_b, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || first_block < 0 || n_blocks < 0) return QSA_ERR_INVALID_ARG;
  if (B == 0 || n_blocks == 0) return QSA_OK;
  if (k_idx == nullptr || kbar == nullptr || !aligned16(k_idx) || !aligned16(kbar)) return QSA_ERR_INVALID_ARG;
  if (B > 1 && (k_idx_stride_b < (first_block + n_blocks) * cfg->r * kHeadDim ||
                kbar_stride_b < (first_block + n_blocks) * kHeadDim))
    return QSA_ERR_INVALID_ARG;
  if ((k_idx_stride_b % 8) != 0 || (kbar_stride_b % 8) != 0) return QSA_ERR_INVALID_ARG;
  return from_cuda(launch_compress_keys(
      static_cast<const __nv_bfloat16*>(k_idx), k_idx_stride_b, B, first_block, n_blocks, cfg->r,
      cfg->rmsnorm, cfg->rms_eps, rope_params(cfg), static_cast<__nv_bfloat16*>(kbar),
      kbar_stride_b, reinterpret_cast<cudaStream_t>(stream)));
}

size_t qsa_index_topk_workspace(const qsa_config* cfg, int64_t B, int64_t n_q, int64_t n_blocks_max) {
  if (check_config(cfg) != QSA_OK || B < 0 || n_q < 0 || n_blocks_max < 0) return 0;
  return index_layout(B, n_q, n_blocks_max, k_blocks(cfg), cfg->n_idx_heads).total;
}

qsa_status qsa_index_rows_per_wave(const qsa_config* cfg, int64_t* rows) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (rows == nullptr) return QSA_ERR_INVALID_ARG;
  int sms = 0;
  if (current_sm_count(&sms) != cudaSuccess || sms <= 0) {
    cudaGetLastError();  // a failed query leaves no sticky error behind
    return QSA_ERR_CUDA;
  }
  *rows = (int64_t)fused_tile_tokens(cfg->n_idx_heads) * sms;
  return QSA_OK;
}

qsa_status qsa_index_topk(const qsa_config* cfg, const void* q_idx, const void* kbar,
                          int64_t kbar_stride_b, const int64_t* q_pos, int64_t B, int64_t n_q,
                          int64_t n_blocks_max, int32_t* idx, int32_t* count, void* ws,
                          size_t ws_bytes, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || n_q < 0 || n_blocks_max < 0) return QSA_ERR_INVALID_ARG;
  if (B == 0 || n_q == 0) return QSA_OK;
  if (q_idx == nullptr || q_pos == nullptr || idx == nullptr || count == nullptr) return QSA_ERR_INVALID_ARG;
  if (n_blocks_max > 0 && kbar == nullptr) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || (kbar != nullptr && !aligned16(kbar)) || (kbar_stride_b % 8) != 0)
    return QSA_ERR_INVALID_ARG;
  if (B > 1 && kbar_stride_b < n_blocks_max * kHeadDim) return QSA_ERR_INVALID_ARG;
  const IndexLayout L = index_layout(B, n_q, n_blocks_max, k_blocks(cfg), cfg->n_idx_heads);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return QSA_ERR_INVALID_ARG;
  if (ws_bytes < L.total) return QSA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  __nv_bfloat16* qt = reinterpret_cast<__nv_bfloat16*>(w + L.qt_off);
  float* S = reinterpret_cast<float*>(w + L.s_off);
  const int r = cfg->r, k_b = k_blocks(cfg), H = cfg->n_idx_heads;
  const auto* kb = static_cast<const __nv_bfloat16*>(kbar);
  cudaError_t e = launch_rotate_queries(static_cast<const __nv_bfloat16*>(q_idx), q_pos, B, n_q, r, H,
                                        rope_params(cfg), qt, st);
  if (e != cudaSuccess) return from_cuda(e);
  if (L.fused)
    return from_cuda(launch_index_fused(H, qt, kb, kbar_stride_b, q_pos, B, n_q, n_blocks_max, r, k_b, idx, count,
                                        w + L.s_off, st));
  const int64_t rows = B * n_q;
  if (n_q <= kDecodeMaxRows && rows <= L.rows_per_launch) {  // decode: one or a few query rows per sequence
    e = launch_decode_scan(H, qt, kb, kbar_stride_b, q_pos, B, (int)n_q, r, n_blocks_max, S, L.s_stride, st);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_topk_select_cluster(S, L.s_stride, q_pos, n_q, 0, rows, r, k_b, n_blocks_max, idx, count, st));
  }
  // Row ranges within one sequence at a time, as many rows as the score buffer holds.
  for (int64_t bb = 0; bb < B; ++bb) {
    for (int64_t j_lo = 0; j_lo < n_q; j_lo += L.rows_per_launch) {
      const int64_t nr = n_q - j_lo < L.rows_per_launch ? n_q - j_lo : L.rows_per_launch;
      e = launch_index_scan(H, qt, kb, kbar_stride_b, q_pos, bb, n_q, j_lo, nr, r, n_blocks_max, S, L.s_stride, st);
      if (e != cudaSuccess) return from_cuda(e);
      e = launch_topk_select(S, L.s_stride, q_pos, n_q, bb * n_q + j_lo, nr, r, k_b, n_blocks_max, idx, count, st);
      if (e != cudaSuccess) return from_cuda(e);
    }
  }
  return QSA_OK;
}

qsa_status qsa_index_topk_fallback_rows(const qsa_config* cfg, int64_t B, int64_t n_q, int64_t n_blocks_max,
                                        const void* ws, size_t ws_bytes, int64_t* rows, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || n_q < 0 || n_blocks_max < 0 || rows == nullptr) return QSA_ERR_INVALID_ARG;
  *rows = 0;
  if (B == 0 || n_q == 0) return QSA_OK;
  const IndexLayout L = index_layout(B, n_q, n_blocks_max, k_blocks(cfg), cfg->n_idx_heads);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return QSA_ERR_INVALID_ARG;
  if (ws_bytes < L.total) return QSA_ERR_WORKSPACE;
  if (!L.fused) return QSA_OK;  // the scan path selects every row exactly in one pass
  return from_cuda(read_fused_fallback_rows(static_cast<const char*>(ws) + L.s_off, B, n_q, n_blocks_max,
                                            cfg->n_idx_heads, rows, reinterpret_cast<cudaStream_t>(stream)));
}

qsa_status qsa_sparse_attn_prefill_impl(const qsa_config* cfg, const void* q, const void* k,
                                        const void* v, int64_t L_cap, const int64_t* q_pos,
                                        const int32_t* idx, const int32_t* count, int64_t B,
                                        int64_t n_q, int32_t Hq, int32_t Hkv, float scale, void* out,
                                        float* lse, qsa_attn_impl impl, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || n_q < 0 || L_cap < 0 || Hq < 1 || Hkv < 1 || !std::isfinite(scale)) return QSA_ERR_INVALID_ARG;
  if (impl != QSA_ATTN_AUTO && impl != QSA_ATTN_TCGEN05 && impl != QSA_ATTN_MMA_SYNC) return QSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || L_cap > kMaxLCap) return QSA_ERR_UNSUPPORTED;
  const bool tc_ok = tc_attention_supported(Hq, Hkv, cfg->r);
  if (impl == QSA_ATTN_TCGEN05 && !tc_ok) return QSA_ERR_UNSUPPORTED;
  if (B == 0 || n_q == 0) return QSA_OK;
  if (!q || !k || !v || !q_pos || !idx || !count || !out || L_cap < 1) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return QSA_ERR_INVALID_ARG;
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* ob = static_cast<__nv_bfloat16*>(out);
  const float sc = softmax_scale(cfg, scale);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // AUTO takes the mma.sync kernel: on B300 it gathers at about 18.6 TB/s
  // against 6.8 TB/s for the TMA-fed tcgen05 kernel at every supported r.
  if (impl == QSA_ATTN_TCGEN05)
    return from_cuda(launch_sparse_attn_tc(qb, kb, vb, L_cap, q_pos, idx, count, B, n_q, Hq, Hkv, cfg->r,
                                           k_blocks(cfg), sc, ob, lse, st));
  return from_cuda(launch_sparse_attn_prefill(qb, kb, vb, L_cap, q_pos, idx, count, B, n_q, Hq, Hkv, cfg->r,
                                              k_blocks(cfg), sc, ob, lse, st));
}

qsa_status qsa_sparse_attn_prefill(const qsa_config* cfg, const void* q, const void* k,
                                   const void* v, int64_t L_cap, const int64_t* q_pos,
                                   const int32_t* idx, const int32_t* count, int64_t B,
                                   int64_t n_q, int32_t Hq, int32_t Hkv, float scale, void* out,
                                   float* lse, qsa_stream_t stream) {
  return qsa_sparse_attn_prefill_impl(cfg, q, k, v, L_cap, q_pos, idx, count, B, n_q, Hq, Hkv, scale, out, lse,
                                      QSA_ATTN_AUTO, stream);
}

size_t qsa_sparse_attn_decode_workspace(const qsa_config* cfg, int64_t B, int32_t Hq, int32_t Hkv) {
  if (check_config(cfg) != QSA_OK || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return 0;
  return align_up(decode_workspace_bytes(B, Hq, Hkv, k_blocks(cfg), cfg->r));
}

qsa_status qsa_sparse_attn_decode(const qsa_config* cfg, const void* q, const void* k_cache,
                                  const void* v_cache, int64_t L_cap, const int64_t* cache_len,
                                  const int32_t* idx, const int32_t* count, int64_t B, int32_t Hq,
                                  int32_t Hkv, float scale, void* out, float* lse, void* ws,
                                  size_t ws_bytes, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || L_cap < 0 || Hq < 1 || Hkv < 1 || !std::isfinite(scale)) return QSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || L_cap > kMaxLCap) return QSA_ERR_UNSUPPORTED;
  if (B == 0) return QSA_OK;
  if (!q || !k_cache || !v_cache || !cache_len || !idx || !count || !out || L_cap < 1)
    return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return QSA_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return QSA_ERR_INVALID_ARG;
  if (ws_bytes < qsa_sparse_attn_decode_workspace(cfg, B, Hq, Hkv)) return QSA_ERR_WORKSPACE;
  return from_cuda(launch_sparse_attn_decode(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_cache),
      static_cast<const __nv_bfloat16*>(v_cache), L_cap, cache_len, idx, count, B, 1, Hq, Hkv,
      cfg->r, k_blocks(cfg), softmax_scale(cfg, scale), static_cast<__nv_bfloat16*>(out), lse, ws,
      reinterpret_cast<cudaStream_t>(stream)));
}

size_t qsa_sparse_attn_decode_multi_workspace(const qsa_config* cfg, int64_t B, int32_t n_q, int32_t Hq,
                                              int32_t Hkv) {
  if (check_config(cfg) != QSA_OK || B < 0 || n_q < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return 0;
  return align_up(decode_workspace_bytes(B * n_q, Hq, Hkv, k_blocks(cfg), cfg->r));
}

qsa_status qsa_sparse_attn_decode_multi(const qsa_config* cfg, const void* q, const void* k_cache,
                                        const void* v_cache, int64_t L_cap, const int64_t* cache_len,
                                        const int32_t* idx, const int32_t* count, int64_t B, int32_t n_q,
                                        int32_t Hq, int32_t Hkv, float scale, void* out, float* lse, void* ws,
                                        size_t ws_bytes, qsa_stream_t stream) {
  qsa_status s = check_config(cfg);
  if (s != QSA_OK) return s;
  if (B < 0 || n_q < 1 || L_cap < 0 || Hq < 1 || Hkv < 1 || !std::isfinite(scale)) return QSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || L_cap > kMaxLCap) return QSA_ERR_UNSUPPORTED;
  if (B == 0) return QSA_OK;
  if (!q || !k_cache || !v_cache || !cache_len || !idx || !count || !out || L_cap < 1)
    return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return QSA_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return QSA_ERR_INVALID_ARG;
  if (ws_bytes < qsa_sparse_attn_decode_multi_workspace(cfg, B, n_q, Hq, Hkv)) return QSA_ERR_WORKSPACE;
  return from_cuda(launch_sparse_attn_decode(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_cache),
      static_cast<const __nv_bfloat16*>(v_cache), L_cap, cache_len, idx, count, B, n_q, Hq, Hkv,
      cfg->r, k_blocks(cfg), softmax_scale(cfg, scale), static_cast<__nv_bfloat16*>(out), lse, ws,
      reinterpret_cast<cudaStream_t>(stream)));
}

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_WORKSPACE: return "QSA_ERR_WORKSPACE";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
    case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
  }
  return "QSA_ERR_UNKNOWN";
}

qsa_status qsa_read_device_error(qsa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  unsigned int code = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&code, g_device_error, sizeof(code));
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
  if (e != cudaSuccess) return from_cuda(e);
  switch (code) {
    case 0: return QSA_OK;
    case kDevErrTimeout: return QSA_ERR_TIMEOUT;
    default: return QSA_ERR_INVALID_ARG;
  }
}

uint64_t qsa_launch_count(void) { return __atomic_load_n(&launch_counter(), __ATOMIC_RELAXED); }

const char* qsa_version(void) { return "qsa-b300 0.1 sm_103a"; }

}  // extern "C"

// Decode entry point with library-owned static scratch (no allocation).
#include "decode_noalloc.cu"

// Diagnostic entry point for the bounded-wait path.
#include "selftest.cu"
