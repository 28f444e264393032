// Indexer block scores I_ib = sum_h ReLU(<qt_i^h, kbar_b>) written out per row,
// for rows whose score vector is short enough to keep (decode: one query per
// sequence, c_i <= 2^18 blocks; prefill: a bounded chunk of rows at a time).
//
// "On the Design of Qwen3.8-Next Architecture", research-hub notes, Key ideas,
// QSA compressed-indexer bullet (the formula and the 4-query-head / 1-key-head
// MQA layout); paperglide reader, "Qwen Sparse Attention" step 3 (block-causal
// mask: row i scores only the c_i completed blocks).
//
// Decode reads 256 B of kbar per candidate block and does 1 KFLOP with it, so
// the scan is HBM-bound.  Each warp streams kbar rows straight into the A
// fragments of m16n8k16 tensor-core MMAs (16 blocks x 16 dims per step), with the
// 8 B columns holding two query rows x four indexer heads.  Head dims are
// visited in a permuted order in which every lane reads 64 contiguous bytes of
// each row it touches (4 x 16-byte loads); the permutation is applied to both
// operands, so the dot products are unchanged.
#include "common.cuh"

namespace qsa {

constexpr int kScanWarps = 8;
constexpr int kScanChunk = 256;  // blocks per warp work item

// qt     [rows][4][128] bf16, rows = B * n_q, rotated queries
// kbar   sequence bb at kbar + bb * kbar_stride_b
// S      [rows][s_stride] fp32; entry b written for b < c_row only
// row_lo first row handled by this launch (prefill chunks), n_rows rows
__global__ void __launch_bounds__(kScanWarps * 32)
index_scan_kernel(const __nv_bfloat16* __restrict__ qt, const __nv_bfloat16* __restrict__ kbar,
                  int64_t kbar_stride_b, const int64_t* __restrict__ q_pos, int64_t n_q,
                  int64_t row_lo, int64_t n_rows, int r, int64_t c_cap, int64_t n_chunks,
                  float* __restrict__ S, int64_t s_stride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t item = (int64_t)blockIdx.x * kScanWarps + warp;
  const int64_t n_pairs = (n_rows + 1) >> 1;
  if (item >= n_pairs * n_chunks) return;
  const int64_t pair = item % n_pairs;
  const int64_t chunk = item / n_pairs;

  // The two rows of the pair (the second may be past the end, or in another
  // sequence: each row carries its own sequence, position and c).
  int64_t row[2], bb[2], c[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    int64_t rr = row_lo + 2 * pair + p;
    const bool ok = (2 * pair + p) < n_rows;
    rr = ok ? rr : row_lo + 2 * pair;
    row[p] = rr;
    bb[p] = rr / n_q;
    const int64_t pos = q_pos[bb[p]] + rr % n_q;
    c[p] = ok ? (pos + 1) / r : 0;
    if (c[p] > c_cap) {  // position past the caller's bound: clamp and report
      if (chunk == 0 && (lane == 0)) flag_device_error(kDevErrPosition);
      c[p] = c_cap;
    }
  }
  const int64_t b_begin = chunk * kScanChunk;
  const int64_t c_max = c[0] > c[1] ? c[0] : c[1];
  if (b_begin >= c_max) return;
  // Rows of a pair share kbar only when they are in the same sequence.
  const bool same_seq = bb[0] == bb[1];

  // B fragment: column n = gid -> (row in pair gid / 4, head gid % 4); lane t
  // holds permuted dims 32t .. 32t+31 of that head.
  uint32_t qf[16];
  {
    const int p = gid >> 2, h = gid & 3;
    const bool valid = c[p] > 0;
    const uint4* src = reinterpret_cast<const uint4*>(qt + (row[p] * kIdxHeads + h) * kHeadDim + 32 * t);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint4 v = valid ? src[u] : make_uint4(0, 0, 0, 0);
      qf[4 * u + 0] = v.x; qf[4 * u + 1] = v.y; qf[4 * u + 2] = v.z; qf[4 * u + 3] = v.w;
    }
  }

  const int64_t b_end = (b_begin + kScanChunk < c_max) ? b_begin + kScanChunk : c_max;
  // Each pair is processed once per sequence it spans (normally once).
  for (int pass = 0; pass < (same_seq ? 1 : 2); ++pass) {
    const __nv_bfloat16* kb = kbar + bb[pass] * kbar_stride_b;
    // Never read past the blocks this sequence is known to hold.
    const int64_t e = same_seq ? b_end : (b_end < c[pass] ? b_end : c[pass]);
    for (int64_t b0 = b_begin; b0 < e; b0 += 16) {
      const int64_t ra = b0 + gid, rb = b0 + gid + 8;
      const int64_t ra_c = ra < e ? ra : e - 1;
      const int64_t rb_c = rb < e ? rb : e - 1;
      uint32_t ka[16], kb16[16];
      const uint4* pa = reinterpret_cast<const uint4*>(kb + ra_c * kHeadDim + 32 * t);
      const uint4* pb = reinterpret_cast<const uint4*>(kb + rb_c * kHeadDim + 32 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 x = ldg_stream(pa + u), y = ldg_stream(pb + u);
        ka[4 * u] = x.x; ka[4 * u + 1] = x.y; ka[4 * u + 2] = x.z; ka[4 * u + 3] = x.w;
        kb16[4 * u] = y.x; kb16[4 * u + 1] = y.y; kb16[4 * u + 2] = y.z; kb16[4 * u + 3] = y.w;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a[4] = {ka[2 * ks], kb16[2 * ks], ka[2 * ks + 1], kb16[2 * ks + 1]};
        const uint32_t b[2] = {qf[2 * ks], qf[2 * ks + 1]};
        mma_bf16_16816(acc, a, b);
      }
      // acc: (block ra, col 2t), (ra, 2t+1), (rb, 2t), (rb, 2t+1); col -> row
      // in pair t/2, heads 2(t%2), 2(t%2)+1.  ReLU, then sum the head pair held
      // by lane t^1.
      float sa = fmaxf(acc[0], 0.f) + fmaxf(acc[1], 0.f);
      float sb = fmaxf(acc[2], 0.f) + fmaxf(acc[3], 0.f);
      sa += __shfl_xor_sync(0xffffffffu, sa, 1);
      sb += __shfl_xor_sync(0xffffffffu, sb, 1);
      const int p = t >> 1;
      if (same_seq || p == pass) {
        const int64_t rblk = (t & 1) ? rb : ra;
        const float val = (t & 1) ? sb : sa;
        if (rblk < c[p]) S[(row[p] - row_lo) * s_stride + rblk] = val;
      }
    }
  }
}

cudaError_t launch_index_scan(const __nv_bfloat16* qt, const __nv_bfloat16* kbar,
                              int64_t kbar_stride_b, const int64_t* q_pos, int64_t n_q,
                              int64_t row_lo, int64_t n_rows, int r, int64_t c_max, float* S,
                              int64_t s_stride, cudaStream_t st) {
  // c_max is also the clamp for every row's visible-block count.
  if (n_rows <= 0 || c_max <= 0) return cudaSuccess;
  const int64_t n_chunks = (c_max + kScanChunk - 1) / kScanChunk;
  const int64_t items = ((n_rows + 1) / 2) * n_chunks;
  const int64_t grid = (items + kScanWarps - 1) / kScanWarps;
  index_scan_kernel<<<(unsigned)grid, kScanWarps * 32, 0, st>>>(
      qt, kbar, kbar_stride_b, q_pos, n_q, row_lo, n_rows, r, c_max, n_chunks, S, s_stride);
  return count_launch(cudaGetLastError());
}


// Decode scan: up to 4 query rows per sequence (one new token, or the n_q
// tokens of a multi-token step), all scored in the same pass over k-bar.  A
// persistent grid of warps splits the (sequence, 16-block tile) space into
// equal contiguous ranges, so every warp streams the same number of k-bar rows
// and none is left for a tail wave.  Within a range the 16-block tiles are
// double-buffered in registers (the next tile's 8 loads per lane are in flight
// while the current tile's MMAs run).  MMA n-tile j holds query rows 2j and
// 2j + 1 (4 heads each; a missing row is zero).  Every row is scored up to the
// sequence's largest visible block; the selection applies each row's own range.
template <int NT>
__global__ void __launch_bounds__(kScanWarps * 32)
decode_scan_kernel(const __nv_bfloat16* __restrict__ qt, const __nv_bfloat16* __restrict__ kbar,
                   int64_t kbar_stride_b, const int64_t* __restrict__ q_pos, int64_t B, int n_q, int r,
                   int64_t c_cap, int64_t tiles_per_seq, int64_t tiles_per_warp, float* __restrict__ S,
                   int64_t s_stride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t wid = (int64_t)blockIdx.x * kScanWarps + warp;
  const int64_t total = B * tiles_per_seq;
  int64_t t0 = wid * tiles_per_warp;
  const int64_t t1 = t0 + tiles_per_warp < total ? t0 + tiles_per_warp : total;
  while (t0 < t1) {
    const int64_t bb = t0 / tiles_per_seq;
    const int64_t seg_end = (bb + 1) * tiles_per_seq < t1 ? (bb + 1) * tiles_per_seq : t1;
    int64_t c = (q_pos[bb] + n_q) / r;  // blocks the sequence's last row sees
    if (c > c_cap) {
      if (lane == 0 && t0 == bb * tiles_per_seq) flag_device_error(kDevErrPosition);
      c = c_cap;
    }
    const int64_t b_begin = (t0 - bb * tiles_per_seq) * 16;
    const int64_t b_lim = (seg_end - bb * tiles_per_seq) * 16;
    const int64_t b_end = b_lim < c ? b_lim : c;
    t0 = seg_end;
    if (b_begin >= b_end) continue;
    uint32_t qf[NT][16];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int qrow = 2 * j + (gid >> 2);
      const uint4* src =
          reinterpret_cast<const uint4*>(qt + ((bb * n_q + qrow) * kIdxHeads + (gid & 3)) * kHeadDim + 32 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = qrow < n_q ? src[u] : make_uint4(0, 0, 0, 0);
        qf[j][4 * u + 0] = v.x; qf[j][4 * u + 1] = v.y; qf[j][4 * u + 2] = v.z; qf[j][4 * u + 3] = v.w;
      }
    }
    const __nv_bfloat16* kb = kbar + bb * kbar_stride_b;
    auto load_tile = [&](int64_t b0, uint32_t (&ka)[16], uint32_t (&kx)[16]) {
      const int64_t ra = b0 + gid < b_end ? b0 + gid : b_end - 1;
      const int64_t rb = b0 + gid + 8 < b_end ? b0 + gid + 8 : b_end - 1;
      const uint4* pa = reinterpret_cast<const uint4*>(kb + ra * kHeadDim + 32 * t);
      const uint4* pb = reinterpret_cast<const uint4*>(kb + rb * kHeadDim + 32 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 x = ldg_stream(pa + u), y = ldg_stream(pb + u);
        ka[4 * u] = x.x; ka[4 * u + 1] = x.y; ka[4 * u + 2] = x.z; ka[4 * u + 3] = x.w;
        kx[4 * u] = y.x; kx[4 * u + 1] = y.y; kx[4 * u + 2] = y.z; kx[4 * u + 3] = y.w;
      }
    };
    uint32_t ka[16], kx[16], na[16], nx[16];
    load_tile(b_begin, ka, kx);
    for (int64_t b0 = b_begin; b0 < b_end; b0 += 16) {
      const bool more = b0 + 16 < b_end;
      if (more) load_tile(b0 + 16, na, nx);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a[4] = {ka[2 * ks], kx[2 * ks], ka[2 * ks + 1], kx[2 * ks + 1]};
          const uint32_t bq[2] = {qf[j][2 * ks], qf[j][2 * ks + 1]};
          mma_bf16_16816(acc, a, bq);
        }
        // acc: (block b0+gid, columns 2t, 2t+1), (b0+gid+8, 2t, 2t+1); column
        // 4 q' + h is head h of query row 2j + q'.
        float sa = fmaxf(acc[0], 0.f) + fmaxf(acc[1], 0.f);
        float sb = fmaxf(acc[2], 0.f) + fmaxf(acc[3], 0.f);
        sa += __shfl_xor_sync(0xffffffffu, sa, 1);
        sb += __shfl_xor_sync(0xffffffffu, sb, 1);
        const int qrow = 2 * j + (t >> 1);
        if ((t & 1) == 0 && qrow < n_q) {
          float* srow = S + (bb * n_q + qrow) * s_stride;
          if (b0 + gid < b_end) srow[b0 + gid] = sa;
          if (b0 + gid + 8 < b_end) srow[b0 + gid + 8] = sb;
        }
      }
      if (more) {
#pragma unroll
        for (int u = 0; u < 16; ++u) { ka[u] = na[u]; kx[u] = nx[u]; }
      }
    }
  }
}

template <int NT>
static cudaError_t launch_decode_scan_nt(const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                                         const int64_t* q_pos, int64_t B, int n_q, int r, int64_t c_max, float* S,
                                         int64_t s_stride, cudaStream_t st) {
  int blocks_per_sm = 0, sms = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, decode_scan_kernel<NT>,
                                                                kScanWarps * 32, 0);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm < 1) blocks_per_sm = 1;
  e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int64_t tiles_per_seq = (c_max + 15) / 16;
  const int64_t total = B * tiles_per_seq;
  int64_t warps = (int64_t)sms * blocks_per_sm * kScanWarps;
  const int64_t tiles_per_warp = (total + warps - 1) / warps;
  warps = (total + tiles_per_warp - 1) / tiles_per_warp;
  const int64_t grid = (warps + kScanWarps - 1) / kScanWarps;
  decode_scan_kernel<NT><<<(unsigned)grid, kScanWarps * 32, 0, st>>>(qt, kbar, kbar_stride_b, q_pos, B, n_q, r, c_max,
                                                                     tiles_per_seq, tiles_per_warp, S, s_stride);
  return count_launch(cudaGetLastError());
}

// Scores of the n_q <= kDecodeMaxRows query rows of each sequence in one pass
// over k-bar; rows bb * n_q + j of S.
constexpr int kDecodeMaxRows = 4;

cudaError_t launch_decode_scan(const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                               const int64_t* q_pos, int64_t B, int n_q, int r, int64_t c_max, float* S,
                               int64_t s_stride, cudaStream_t st) {
  if (B <= 0 || c_max <= 0 || n_q <= 0) return cudaSuccess;
  if (n_q > kDecodeMaxRows) return cudaErrorInvalidValue;
  return n_q <= 2 ? launch_decode_scan_nt<1>(qt, kbar, kbar_stride_b, q_pos, B, n_q, r, c_max, S, s_stride, st)
                  : launch_decode_scan_nt<2>(qt, kbar, kbar_stride_b, q_pos, B, n_q, r, c_max, S, s_stride, st);
}

}  // namespace qsa
