// Indexer block scores I_ib = sum_h ReLU(<qt_i^h, kbar_b>) written out per row,
// for rows whose score vector is short enough to keep (decode: a few queries
// per sequence; prefill: a bounded range of rows at a time).
//
// "On the Design of Qwen3.8-Next Architecture", research-hub notes, Key ideas,
// QSA compressed-indexer bullet (the formula; an MQA indexer whose H query
// heads share one key head, H = 4 there); paperglide reader, "Qwen Sparse
// Attention" step 3 (block-causal mask: row i scores only the c_i completed
// blocks).
//
// Decode reads 256 B of kbar per candidate block and does 2 H 128 flops per
// query row with it, so the scan is HBM-bound.  Each warp streams kbar rows
// straight into the A fragments of m16n8k16 tensor-core MMAs (16 blocks x 16
// dims per step), with the 8 B columns holding 8 / H query rows x H indexer
// heads.  Head dims are visited in a permuted order in which every lane reads
// 64 contiguous bytes of each row it touches (4 x 16-byte loads); the
// permutation is applied to both operands, so the dot products are unchanged.
#include "common.cuh"

namespace qsa {

constexpr int kScanWarps = 8;
constexpr int kScanChunk = 256;  // blocks per warp work item

// Scores of the MMA columns of one 16-block step: column n = (row n / H, head
// n % H).  acc[0..1] are columns 2t, 2t + 1 of block ra, acc[2..3] of block rb.
// Returns, for the lane's first column's row, the head sums of blocks ra and rb
// (valid where `writes` is set: the lane holding head 0 of a row).
template <int H>
__device__ __forceinline__ void head_sums(const float acc[4], int t, float& sa, float& sb, float& sa2, float& sb2,
                                          bool& writes) {
  if (H == 1) {  // columns 2t and 2t + 1 are two rows
    sa = fmaxf(acc[0], 0.f);
    sa2 = fmaxf(acc[1], 0.f);
    sb = fmaxf(acc[2], 0.f);
    sb2 = fmaxf(acc[3], 0.f);
    writes = true;
    return;
  }
  sa = fmaxf(acc[0], 0.f) + fmaxf(acc[1], 0.f);
  sb = fmaxf(acc[2], 0.f) + fmaxf(acc[3], 0.f);
  if (H >= 4) {
    sa += __shfl_xor_sync(0xffffffffu, sa, 1);
    sb += __shfl_xor_sync(0xffffffffu, sb, 1);
  }
  if (H >= 8) {
    sa += __shfl_xor_sync(0xffffffffu, sa, 2);
    sb += __shfl_xor_sync(0xffffffffu, sb, 2);
  }
  sa2 = sb2 = 0.f;
  writes = ((2 * t) % H) == 0;
}

// Prefill rows j_lo .. j_lo + n_rows - 1 of sequence bb, in groups of R = 8 / H
// rows (one MMA N tile).  qt [B * n_q][H][128] bf16 rotated queries; S row
// (j - j_lo) of the launch, entry b written for b < c_row.
template <int H>
__global__ void __launch_bounds__(kScanWarps * 32)
index_scan_kernel(const __nv_bfloat16* __restrict__ qt, const __nv_bfloat16* __restrict__ kbar,
                  int64_t kbar_stride_b, const int64_t* __restrict__ q_pos, int64_t bb, int64_t n_q,
                  int64_t j_lo, int64_t n_rows, int r, int64_t c_cap, int64_t n_chunks,
                  float* __restrict__ S, int64_t s_stride) {
  constexpr int R = 8 / H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t item = (int64_t)blockIdx.x * kScanWarps + warp;
  const int64_t n_groups = (n_rows + R - 1) / R;
  if (item >= n_groups * n_chunks) return;
  const int64_t grp = item % n_groups;
  const int64_t chunk = item / n_groups;
  // Rows of the group (one sequence): row k is j_lo + R grp + k; c = 0 past the range.
  int64_t c[R];
  int64_t c_max = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int64_t jj = R * grp + k;
    c[k] = 0;
    if (jj < n_rows) {
      c[k] = (q_pos[bb] + j_lo + jj + 1) / r;
      if (c[k] > c_cap) {  // position past the caller's bound: clamp and report
        if (chunk == 0 && lane == 0) flag_device_error(kDevErrPosition);
        c[k] = c_cap;
      }
    }
    c_max = c[k] > c_max ? c[k] : c_max;
  }
  const int64_t b_begin = chunk * kScanChunk;
  if (b_begin >= c_max) return;

  // B fragment: column n = gid -> (row gid / H, head gid % H); lane t holds
  // permuted dims 32t .. 32t+31 of that head.
  uint32_t qf[16];
  {
    const int k = gid / H, h = gid % H;
    const int64_t jj = R * grp + k;
    const bool valid = jj < n_rows;
    const uint4* src =
        reinterpret_cast<const uint4*>(qt + ((bb * n_q + j_lo + (valid ? jj : 0)) * H + h) * kHeadDim + 32 * t);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint4 v = valid ? src[u] : make_uint4(0, 0, 0, 0);
      qf[4 * u + 0] = v.x; qf[4 * u + 1] = v.y; qf[4 * u + 2] = v.z; qf[4 * u + 3] = v.w;
    }
  }
  // c of the rows this lane's columns belong to (no dynamic register indexing).
  const int k0 = (2 * t) / H, k1 = (2 * t + 1) / H;
  int64_t c0 = 0, c1 = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    if (k == k0) c0 = c[k];
    if (k == k1) c1 = c[k];
  }

  const int64_t e = (b_begin + kScanChunk < c_max) ? b_begin + kScanChunk : c_max;
  const __nv_bfloat16* kb = kbar + bb * kbar_stride_b;
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
    float sa, sb, sa2, sb2;
    bool writes;
    head_sums<H>(acc, t, sa, sb, sa2, sb2, writes);
    if (writes) {
      float* s0 = S + (R * grp + k0) * s_stride;
      if (ra < c0) s0[ra] = sa;
      if (rb < c0) s0[rb] = sb;
      if (H == 1) {
        float* s1 = S + (R * grp + k1) * s_stride;
        if (ra < c1) s1[ra] = sa2;
        if (rb < c1) s1[rb] = sb2;
      }
    }
  }
}

cudaError_t launch_index_scan(int H, const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                              const int64_t* q_pos, int64_t bb, int64_t n_q, int64_t j_lo, int64_t n_rows, int r,
                              int64_t c_max, float* S, int64_t s_stride, cudaStream_t st) {
  // c_max is also the clamp for every row's visible-block count.
  if (n_rows <= 0 || c_max <= 0) return cudaSuccess;
  const int R = 8 / H;
  const int64_t n_chunks = (c_max + kScanChunk - 1) / kScanChunk;
  const int64_t items = ((n_rows + R - 1) / R) * n_chunks;
  const int64_t grid = (items + kScanWarps - 1) / kScanWarps;
#define QSA_SCAN_CASE(HH)                                                                                  \
  case HH:                                                                                                 \
    index_scan_kernel<HH><<<(unsigned)grid, kScanWarps * 32, 0, st>>>(qt, kbar, kbar_stride_b, q_pos, bb, \
                                                                      n_q, j_lo, n_rows, r, c_max,         \
                                                                      n_chunks, S, s_stride);              \
    break;
  switch (H) {
    QSA_SCAN_CASE(1)
    QSA_SCAN_CASE(2)
    QSA_SCAN_CASE(4)
    QSA_SCAN_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef QSA_SCAN_CASE
  return count_launch(cudaGetLastError());
}


// Decode scan: up to 4 query rows per sequence (one new token, or the n_q
// tokens of a multi-token step), all scored in the same pass over k-bar.  A
// persistent grid of warps splits the (sequence, 16-block tile) space into
// equal contiguous ranges, so every warp streams the same number of k-bar rows
// and none is left for a tail wave.  Within a range the 16-block tiles are
// double-buffered in registers (the next tile's 8 loads per lane are in flight
// while the current tile's MMAs run).  MMA n-tile j holds query rows R j ..
// R j + R - 1, R = 8 / H (H heads each; a missing row is zero).  Every row is
// scored up to the sequence's largest visible block; the selection applies
// each row's own range.
template <int H, int NT>
__global__ void __launch_bounds__(kScanWarps * 32)
decode_scan_kernel(const __nv_bfloat16* __restrict__ qt, const __nv_bfloat16* __restrict__ kbar,
                   int64_t kbar_stride_b, const int64_t* __restrict__ q_pos, int64_t B, int n_q, int r,
                   int64_t c_cap, int64_t tiles_per_seq, int64_t tiles_per_warp, float* __restrict__ S,
                   int64_t s_stride) {
  constexpr int R = 8 / H;
  griddep_wait();  // the rotated queries come from the previous kernel
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
      const int qrow = R * j + gid / H;
      const uint4* src =
          reinterpret_cast<const uint4*>(qt + ((bb * n_q + (qrow < n_q ? qrow : 0)) * H + gid % H) * kHeadDim + 32 * t);
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
        float sa, sb, sa2, sb2;
        bool writes;
        head_sums<H>(acc, t, sa, sb, sa2, sb2, writes);
        const int q0 = R * j + (2 * t) / H, q1 = R * j + (2 * t + 1) / H;
        if (writes && q0 < n_q) {
          float* srow = S + (bb * n_q + q0) * s_stride;
          if (b0 + gid < b_end) srow[b0 + gid] = sa;
          if (b0 + gid + 8 < b_end) srow[b0 + gid + 8] = sb;
        }
        if (H == 1 && q1 < n_q) {
          float* srow = S + (bb * n_q + q1) * s_stride;
          if (b0 + gid < b_end) srow[b0 + gid] = sa2;
          if (b0 + gid + 8 < b_end) srow[b0 + gid + 8] = sb2;
        }
      }
      if (more) {
#pragma unroll
        for (int u = 0; u < 16; ++u) { ka[u] = na[u]; kx[u] = nx[u]; }
      }
    }
  }
}

template <int H, int NT>
static cudaError_t launch_decode_scan_nt(const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                                         const int64_t* q_pos, int64_t B, int n_q, int r, int64_t c_max, float* S,
                                         int64_t s_stride, cudaStream_t st) {
  int blocks_per_sm = 0, sms = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, decode_scan_kernel<H, NT>,
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
  return count_launch(launch_dependent(decode_scan_kernel<H, NT>, dim3((unsigned)grid), dim3(kScanWarps * 32), 0, st,
                                      qt, kbar, kbar_stride_b, q_pos, B, n_q, r, c_max, tiles_per_seq,
                                      tiles_per_warp, S, s_stride));
}

// Scores of the n_q <= kDecodeMaxRows query rows of each sequence in one pass
// over k-bar; rows bb * n_q + j of S.
constexpr int kDecodeMaxRows = 4;

cudaError_t launch_decode_scan(int H, const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                               const int64_t* q_pos, int64_t B, int n_q, int r, int64_t c_max, float* S,
                               int64_t s_stride, cudaStream_t st) {
  if (B <= 0 || c_max <= 0 || n_q <= 0) return cudaSuccess;
  if (n_q > kDecodeMaxRows) return cudaErrorInvalidValue;
  const int nt = (n_q * H + 7) / 8;  // MMA n-tiles of 8 columns
#define QSA_DS(HH, NN) launch_decode_scan_nt<HH, NN>(qt, kbar, kbar_stride_b, q_pos, B, n_q, r, c_max, S, s_stride, st)
  switch (H) {
    case 1: return QSA_DS(1, 1);
    case 2: return QSA_DS(2, 1);
    case 4: return nt <= 1 ? QSA_DS(4, 1) : QSA_DS(4, 2);
    case 8: return nt <= 1 ? QSA_DS(8, 1) : (nt <= 2 ? QSA_DS(8, 2) : QSA_DS(8, 4));
    default: return cudaErrorInvalidValue;
  }
#undef QSA_DS
}

}  // namespace qsa
