/*
 * qsa.h -- C ABI of the Qwen Sparse Attention (QSA) library for B300 (sm_103a).
 *
 * Method: "On the Design of Qwen3.8-Next Architecture" (arXiv:2608.30320), as
 * restated by
 *   [KI]  research-hub notes, "Key ideas", QSA compressed-indexer bullet: an MQA
 *         indexer with 4 query heads and 1 shared 128-dim key head; keys are
 *         average-pooled into blocks of r tokens and get partial RoPE on 64 of the
 *         128 dims after pooling; block score I_ib = sum_h ReLU(<q_i^h, kbar_b>);
 *         each query keeps the top k_B = ceil(K / r) blocks plus the tail of its
 *         current block (K = 2048, r = 4 there).
 *   [QSA] paperglide reader, section "Qwen Sparse Attention", toy walk-through
 *         steps 1-5 and Fig. 3: pooling, block-causal scoring, top-k selection,
 *         expansion of the selected blocks to tokens, the tokens of the incomplete
 *         final block, then "sparse core attention" over that token set.
 *   [F6]  paperglide reader, Fig. 6 caption: prefill (chunked) and decode are the
 *         two timed modes.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     never allocates device memory; scratch space is the caller's workspace
 *     (`ws`, `ws_bytes`), whose required size the matching *_workspace() call
 *     returns.  Workspace pointers must be 256-byte aligned.
 *   - Every call is ordered on `stream` and returns without synchronising,
 *     except the two that read a value back to the host
 *     (qsa_index_topk_fallback_rows, qsa_read_device_error), which synchronise
 *     `stream` first.
 *   - Arguments are checked on the host before any launch.  A bad argument
 *     returns QSA_ERR_INVALID_ARG and launches nothing; a shape outside what the
 *     kernels are built for returns QSA_ERR_UNSUPPORTED; a launch failure returns
 *     QSA_ERR_CUDA.  Nothing aborts the process.
 *   - bf16 tensors are row-major with the innermost dimension contiguous; the
 *     head dimension d is 128.
 *   - Positions: token i of a sequence sees the compressed blocks b with
 *     b*r + r - 1 <= i, i.e. c_i = floor((i + 1) / r) blocks; its tail is the
 *     tokens [c_i * r, i] (empty when token i closes its own block).
 *   - Selection is shared by every attention head of a token (one MQA indexer
 *     per token [KI]).
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qsa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned or too-small buffer */
  QSA_ERR_UNSUPPORTED = 2,  /* shape the kernels are not built for (d != 128, Hq % Hkv != 0, ...) */
  QSA_ERR_WORKSPACE = 3,    /* ws_bytes below the size the *_workspace() call reports */
  QSA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  QSA_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (see qsa_read_device_error) */
} qsa_status;

/*
 * Method parameters.  Fields the pages fix: n_idx_heads = 4, head_dim = 128,
 * rope_dims = 64, r and k_tokens (K) [KI]; the paperglide reader's Fig. 5(b)
 * varies the number of indexer query heads and Fig. 5(a) / 6(a,b) the
 * micro-block size r, so both are runtime parameters here.  Fields the pages
 * leave open and this library states explicitly:
 *   rope_base  -- RoPE base (10000 in every workload here).
 *   rmsnorm    -- 1 = unit-weight RMSNorm between pooling and RoPE (the [QSA]
 *                 toy mentions it, [KI] does not); 0 = off (default).
 *   rms_eps    -- epsilon of that RMSNorm.
 * RoPE pairs dims (j, j + rope_dims/2) for j < rope_dims/2 with angle
 * pos * rope_base^(-2j/rope_dims); compressed key b sits at position b and query
 * token i at position floor(i / r), both on the block-index scale.
 */
typedef struct {
  int32_t r;            /* tokens per micro-block (1..16, power of two) */
  int32_t n_idx_heads;  /* indexer query heads: 1, 2, 4 or 8 (4 in [KI]) */
  int32_t head_dim;     /* must be 128 */
  int32_t rope_dims;    /* rotated dims, even, <= head_dim (64) */
  float rope_base;      /* > 0 */
  int32_t rmsnorm;      /* 0 or 1 */
  float rms_eps;        /* > 0 when rmsnorm = 1 */
  int32_t k_tokens;     /* K; k_B = ceil(K / r) selected blocks per token */
} qsa_config;

/* Fills `cfg` with the configuration of [KI]: r = 4, 4 indexer heads, d = 128,
 * 64 rotated dims, base 10000, no RMSNorm, K = 2048.  An n_idx_heads outside
 * {1, 2, 4, 8} or a head_dim other than 128 makes every call return
 * QSA_ERR_UNSUPPORTED. */
void qsa_default_config(qsa_config* cfg);

/* k_B = ceil(K / r) for `cfg` (0 on a null or invalid cfg). */
int32_t qsa_num_selected_blocks(const qsa_config* cfg);

/*
 * Key compression [KI] (pool into blocks of r, partial RoPE after pooling) and
 * [QSA] step 2 (average pooling; optional RMSNorm):
 *   kbar[bb, b] = bf16( RoPE_b( [RMSNorm]( (1/r) * sum_{t<r} k_idx[bb, b*r + t] ) ) )
 * for b in [first_block, first_block + n_blocks) and every sequence bb < B.
 *   k_idx  bf16 [B][*][head_dim]: indexer keys; sequence bb starts at
 *          k_idx + bb * k_idx_stride_b elements; block b reads tokens
 *          [b*r, b*r + r), which the caller guarantees exist.
 *   kbar   bf16 [B][*][head_dim]: sequence bb starts at kbar + bb * kbar_stride_b
 *          elements; rows outside the block range are not touched.
 * Decode appends one block with first_block = (cache_len / r) - 1, n_blocks = 1.
 * Pooling and rotation run in fp32 (angles in fp64); the result is rounded to
 * bf16 once, round-to-nearest-even.
 */
qsa_status qsa_compress_keys(const qsa_config* cfg, const void* k_idx, int64_t k_idx_stride_b,
                             int64_t B, int64_t first_block, int64_t n_blocks, void* kbar,
                             int64_t kbar_stride_b, qsa_stream_t stream);

/*
 * Workspace for qsa_index_topk with the same (cfg, B, n_q, n_blocks_max).
 * Returns 0 when the arguments are invalid.
 */
size_t qsa_index_topk_workspace(const qsa_config* cfg, int64_t B, int64_t n_q,
                                int64_t n_blocks_max);

/*
 * Query rows that one wave of the prefill indexer covers on the current device:
 * its tile rows (48; 24 with 8 indexer heads) times the device's SM count.  A
 * qsa_index_topk call over n_q rows of one sequence runs ceil(n_q / tile rows)
 * tiles, at most one per SM at a time, so chunked prefill [QSA] ("chunked
 * prefill" of the decode/prefill panels) with chunk sizes that are multiples of
 * this number keeps every SM busy to the end of each indexer launch.  A
 * sizing hint only: every chunk size gives the same result.
 *   rows  host int64 out.
 * Returns QSA_ERR_INVALID_ARG for a null cfg or rows, QSA_ERR_UNSUPPORTED for
 * an unsupported cfg, QSA_ERR_CUDA when the device cannot be queried (no GPU).
 */
qsa_status qsa_index_rows_per_wave(const qsa_config* cfg, int64_t* rows);

/*
 * Indexer scoring and top-k_B block selection [KI], [QSA] steps 3-4:
 *   I_ib = sum_{h < H} ReLU(<qt_i^h, kbar_b>)   for b < c_i,  H = n_idx_heads,
 * where qt_i^h = bf16(RoPE_{floor(i/r)}(q_idx[i, h])).  For each row, if
 * c_i <= k_B every visible block is kept; otherwise the k_B blocks with the
 * largest I_ib, an equal score going to the lower block id.
 *   q_idx   bf16 [B][n_q][H][head_dim], un-rotated indexer queries.
 *   kbar    bf16 compressed keys as written by qsa_compress_keys; sequence bb
 *           at kbar + bb * kbar_stride_b elements, holding >= c_i rows for its
 *           last query row.
 *   q_pos   device int64 [B]: absolute position of row 0 of sequence bb; row j
 *           is token q_pos[bb] + j.  Decode passes n_q = 1, q_pos = cache_len - 1.
 *   n_blocks_max  host upper bound of c_i over all rows (sizes the work).
 *   idx     int32 [B][n_q][k_B]: selected block ids in ascending order, -1 past
 *           count.
 *   count   int32 [B][n_q]: min(c_i, k_B).
 * Scores accumulate in fp32 from the bf16 operands; the score matrix is never
 * stored whole.
 */
qsa_status qsa_index_topk(const qsa_config* cfg, const void* q_idx, const void* kbar,
                          int64_t kbar_stride_b, const int64_t* q_pos, int64_t B, int64_t n_q,
                          int64_t n_blocks_max, int32_t* idx, int32_t* count, void* ws,
                          size_t ws_bytes, qsa_stream_t stream);

/*
 * Diagnostic for the prefill indexer: how many rows of the last qsa_index_topk
 * call on `ws` (made with the same cfg, B, n_q, n_blocks_max) were selected by
 * its exact full-row fallback.  The threshold pass collects the entries at or
 * above a per-row threshold taken from a pilot sample; a row whose collection
 * held fewer than k_B entries or more than its buffer (2.5 k_B) is scored again
 * in full.  Its selection is exact either way; only its cost differs.  0 when
 * that call took the one-pass scan path (fewer than 64 rows per sequence, or
 * k_B > 512).  Waits for `stream` and copies one int to the host.
 *   rows   host int64, written.
 * QSA_ERR_INVALID_ARG for a NULL `rows` or workspace, QSA_ERR_WORKSPACE when
 * ws_bytes is below qsa_index_topk_workspace for these sizes.
 */
qsa_status qsa_index_topk_fallback_rows(const qsa_config* cfg, int64_t B, int64_t n_q,
                                        int64_t n_blocks_max, const void* ws, size_t ws_bytes,
                                        int64_t* rows, qsa_stream_t stream);

/*
 * Sparse core attention, prefill [QSA] step 5 and Fig. 3: for query row j of
 * sequence bb (token i = q_pos[bb] + j) and head h with kv head g = h / (Hq/Hkv),
 *   T_i   = union over selected b of [b*r, b*r + r)  plus the tail [c_i*r, i],
 *   o[h]  = sum_{t in T_i} softmax_t(scale * <q[h], k[g, t]>) v[g, t],
 *   lse[h]= log sum_{t in T_i} exp(scale * <q[h], k[g, t]>).
 *   q      bf16 [B][n_q][Hq][head_dim]   (already position-encoded by the caller)
 *   k, v   bf16 [B][Hkv][L_cap][head_dim]; every token of T_i must be < L_cap.
 *          L_cap above 2^31 - 1 returns QSA_ERR_UNSUPPORTED (the kernels index
 *          tokens with 32-bit integers); the same holds for every attention
 *          call below.
 *   q_pos  device int64 [B] as for qsa_index_topk (chunked prefill = q_pos > 0).
 *   idx, count  as written by qsa_index_topk.
 *   scale  softmax scale; a value <= 0 selects 1 / sqrt(head_dim).  Not finite:
 *          QSA_ERR_INVALID_ARG.  (The same holds for every attention call below.)
 *   out    bf16 [B][n_q][Hq][head_dim];  lse  fp32 [B][n_q][Hq] or NULL.
 * Softmax runs in fp32 with a running maximum; QK^T and PV accumulate in fp32.
 */
qsa_status qsa_sparse_attn_prefill(const qsa_config* cfg, const void* q, const void* k,
                                   const void* v, int64_t L_cap, const int64_t* q_pos,
                                   const int32_t* idx, const int32_t* count, int64_t B,
                                   int64_t n_q, int32_t Hq, int32_t Hkv, float scale, void* out,
                                   float* lse, qsa_stream_t stream);

/* Kernel choice for qsa_sparse_attn_prefill_impl. */
typedef enum {
  QSA_ATTN_AUTO = 0,     /* the faster kernel for the shape (what qsa_sparse_attn_prefill does):
                            the mma.sync kernel, measured faster on B300 for every r */
  QSA_ATTN_TCGEN05 = 1,  /* TMA-staged micro-blocks, tcgen05 MMAs with TMEM accumulators; needs
                            Hq = 8 Hkv and r in {4, 8, 16}, else QSA_ERR_UNSUPPORTED */
  QSA_ATTN_MMA_SYNC = 2  /* per-warp cp.async gathers and m16n8k16 MMAs; any Hq % Hkv == 0, any r */
} qsa_attn_impl;

/*
 * qsa_sparse_attn_prefill with an explicit kernel: the same arguments, results
 * and errors, plus `impl` (QSA_ERR_INVALID_ARG for a value outside the enum).
 * Both kernels compute the same function; they differ in rounding order only
 * (fp32 accumulation in both, P rounded to bf16 before the PV product in both).
 */
qsa_status qsa_sparse_attn_prefill_impl(const qsa_config* cfg, const void* q, const void* k,
                                        const void* v, int64_t L_cap, const int64_t* q_pos,
                                        const int32_t* idx, const int32_t* count, int64_t B,
                                        int64_t n_q, int32_t Hq, int32_t Hkv, float scale, void* out,
                                        float* lse, qsa_attn_impl impl, qsa_stream_t stream);

/* Workspace for qsa_sparse_attn_decode with the same (cfg, B, Hq, Hkv). */
size_t qsa_sparse_attn_decode_workspace(const qsa_config* cfg, int64_t B, int32_t Hq,
                                        int32_t Hkv);

/*
 * Sparse core attention for one new token per sequence ([F6] decode mode).
 * The same arithmetic as qsa_sparse_attn_prefill for the single row
 * i = cache_len[bb] - 1, split over the selected tokens and combined with
 * log-sum-exp weights.
 *   q          bf16 [B][Hq][head_dim]
 *   k_cache, v_cache  bf16 [B][Hkv][L_cap][head_dim]
 *   cache_len  device int64 [B]: valid tokens including the new one (<= L_cap).
 *   idx, count int32 [B][k_B], [B] from qsa_index_topk with n_q = 1.
 *   out        bf16 [B][Hq][head_dim];  lse fp32 [B][Hq] or NULL.
 */
qsa_status qsa_sparse_attn_decode(const qsa_config* cfg, const void* q, const void* k_cache,
                                  const void* v_cache, int64_t L_cap, const int64_t* cache_len,
                                  const int32_t* idx, const int32_t* count, int64_t B, int32_t Hq,
                                  int32_t Hkv, float scale, void* out, float* lse, void* ws,
                                  size_t ws_bytes, qsa_stream_t stream);

/* Workspace for qsa_sparse_attn_decode_multi with the same (cfg, B, n_q, Hq, Hkv). */
size_t qsa_sparse_attn_decode_multi_workspace(const qsa_config* cfg, int64_t B, int32_t n_q,
                                              int32_t Hq, int32_t Hkv);

/*
 * Multi-token decode: n_q new tokens per sequence in one step ([F6] decode
 * mode with next_n = 4, i.e. the query token plus three MTP draft tokens).
 * Row j of sequence bb is token i = cache_len[bb] - n_q + j; each row attends
 * over its own selection and tail exactly as qsa_sparse_attn_prefill does for
 * that row, split over the selected tokens and combined with log-sum-exp
 * weights.  Select the rows with qsa_index_topk(n_q, q_pos = cache_len - n_q):
 * for n_q <= 4 it scores all rows of a sequence in one pass over kbar.
 *   q          bf16 [B][n_q][Hq][head_dim]
 *   k_cache, v_cache  bf16 [B][Hkv][L_cap][head_dim]
 *   cache_len  device int64 [B]: valid tokens including the n_q new ones (<= L_cap).
 *   idx, count int32 [B][n_q][k_B], [B][n_q] from qsa_index_topk.
 *   out        bf16 [B][n_q][Hq][head_dim];  lse fp32 [B][n_q][Hq] or NULL.
 *   n_q >= 1; with n_q = 1 this is qsa_sparse_attn_decode.
 */
qsa_status qsa_sparse_attn_decode_multi(const qsa_config* cfg, const void* q, const void* k_cache,
                                        const void* v_cache, int64_t L_cap, const int64_t* cache_len,
                                        const int32_t* idx, const int32_t* count, int64_t B,
                                        int32_t n_q, int32_t Hq, int32_t Hkv, float scale, void* out,
                                        float* lse, void* ws, size_t ws_bytes, qsa_stream_t stream);

/*
 * Size of the static scratch array behind qsa_sparse_attn_decode_noalloc.
 * Every device that loads the library holds this much device memory for it
 * until the process exits.
 */
#define QSA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * qsa_sparse_attn_decode without a workspace argument, for callers that cannot
 * allocate device memory: code inside a host framework or plugin that owns
 * every allocation, paths that must not call cudaMalloc or a pool allocator,
 * or small C hosts with no allocator of their own.  The paper has no
 * counterpart of this entry point; it only changes where the partial results
 * of the split decode live.
 *   Arguments, results and errors are those of qsa_sparse_attn_decode.
 *   Scratch: a fixed QSA_NOALLOC_SCRATCH_BYTES array of static device memory
 *     inside the library (32 MiB: 64 sequences x 2 kv heads at K = 2048,
 *     r = 4 fit).  A call whose qsa_sparse_attn_decode_workspace() size is
 *     larger returns QSA_ERR_WORKSPACE and launches nothing.
 *   No allocation: the call makes no cudaMalloc, cudaFree or other allocating
 *     call.  Its first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on that device.
 *   Devices: the scratch array exists once per device, so the current device
 *     must own `stream` and the tensors on every call; a stream or query tensor
 *     of another device returns QSA_ERR_INVALID_ARG.
 *   Sharing: every call on a device uses the same array, which keeps whatever
 *     the last call left in it.  Nothing in it has to start at zero: each call
 *     writes the maximum and sum of every split it combines, and the combine
 *     skips the partial output of a split whose maximum is -inf (an empty
 *     split), so stale values, even Inf or NaN, never reach a result.  Calls
 *     whose kernels can overlap on the GPU (different streams without ordering
 *     between them) race on the array and give wrong results; order them.
 */
qsa_status qsa_sparse_attn_decode_noalloc(const qsa_config* cfg, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          int64_t L_cap, const int64_t* cache_len,
                                          const int32_t* idx, const int32_t* count, int64_t B,
                                          int32_t Hq, int32_t Hkv, float scale, void* out,
                                          float* lse, qsa_stream_t stream);

/* Human-readable name of a status. */
const char* qsa_status_string(qsa_status s);

/*
 * Diagnostic (not part of the method): launches one CTA whose thread waits,
 * with the library's bounded mbarrier wait, on a barrier that nothing arrives
 * on.  The wait gives up after limit_cycles SM cycles (1000 .. 4e9), records a
 * timeout in the device error word exactly as a stalled qsa_index_topk pipeline
 * would, and the kernel returns normally; qsa_read_device_error then reports
 * QSA_ERR_TIMEOUT.  Lets a host exercise its timeout handling with no device
 * fault.  Returns QSA_ERR_INVALID_ARG for a limit outside the range, else the
 * launch status.
 */
qsa_status qsa_selftest_wait_timeout(int64_t limit_cycles, qsa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error word
 * on the current device (set by a bounded wait that gave up).  Returns QSA_OK,
 * QSA_ERR_TIMEOUT or QSA_ERR_CUDA.
 */
qsa_status qsa_read_device_error(qsa_stream_t stream);

/* Number of kernels this library has launched in this process (all devices,
 * all streams; a host-side counter, incremented at each successful launch). */
uint64_t qsa_launch_count(void);

/* Library version, e.g. "qsa-b300 0.1 sm_103a". */
const char* qsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
