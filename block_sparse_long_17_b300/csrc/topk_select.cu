// Exact top-k_B block selection over a stored score row.
//
// "On the Design of Qwen3.8-Next Architecture", research-hub notes, Key ideas,
// QSA compressed-indexer bullet: each query keeps the top k_B = ceil(K / r)
// blocks; paperglide reader, "Qwen Sparse Attention" step 4 (top-K_B per query,
// expanded back to token indices).  Equal scores go to the lower block id.
//
// One CTA per row.  Scores are ReLU sums, so their fp32 bit patterns (sign
// cleared) order exactly like the values.  A radix descent narrows the range
// [lo, hi] of bit patterns that holds the k_B-th largest score: each pass builds
// a 2048-bin histogram of the patterns inside the range and keeps the bin where
// the running count from the top crosses the number still needed.  It ends when
// that bin holds exactly the number needed, or when it is a single value (an
// exact tie, resolved by taking the lowest block ids first).  A final ordered
// compaction writes the winners in ascending block order.
#include <cooperative_groups.h>

#include "common.cuh"

namespace qsa {

constexpr int kSelThreads = 512;
constexpr int kSelBins = 2048;
constexpr int kSelBinsPerThread = kSelBins / kSelThreads;

__device__ __forceinline__ uint32_t score_key(float s) { return __float_as_uint(s) & 0x7fffffffu; }

// Exclusive scan of `v` across the CTA (blockDim = kSelThreads); returns the
// prefix and stores the total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelThreads / 32 ? warp_sums[lane] : 0;
    int inc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane < kSelThreads / 32) warp_sums[lane] = inc - w;
    if (lane == 31) *total = inc;
  }
  __syncthreads();
  const int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

struct SelectSmem {
  int hist[kSelBins];
  int warp_sums[32];
  int total;
  uint32_t lo, hi;
  int need, done;
};

// Exact top-k_b of the scores s[0 .. c) (c > k_b) by one CTA of kSelThreads
// threads: writes the k_b winners to out[] in ascending block order.
__device__ void cta_select_row(const float* __restrict__ s, int64_t c, int k_b, int32_t* __restrict__ out,
                               SelectSmem& sm) {
  // done = 1: winners are key > hi plus every key in [lo, hi];
  // done = 2: lo == hi, winners are key > hi plus the first `need` keys == lo.
  uint32_t lo = 0, hi = 0x7fffffffu;
  int need = k_b, done = 0;
  for (int guard = 0; !done && guard < 6; ++guard) {  // the range shrinks 2^11-fold per round
    const uint32_t width = hi - lo;
    const int nbits = 32 - __clz(width);
    const int shift = nbits > 11 ? nbits - 11 : 0;
    for (int j = threadIdx.x; j < kSelBins; j += kSelThreads) sm.hist[j] = 0;
    __syncthreads();
    // 16-byte loads (score rows are 16-byte aligned), scalar tail.
    const int64_t c4 = c & ~int64_t(3);
#pragma unroll 4
    for (int64_t e = 4 * (int64_t)threadIdx.x; e < c4; e += 4 * kSelThreads) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(s + e));
      const uint32_t u0 = score_key(x.x), u1 = score_key(x.y), u2 = score_key(x.z), u3 = score_key(x.w);
      if (u0 >= lo && u0 <= hi) atomicAdd(&sm.hist[(u0 - lo) >> shift], 1);
      if (u1 >= lo && u1 <= hi) atomicAdd(&sm.hist[(u1 - lo) >> shift], 1);
      if (u2 >= lo && u2 <= hi) atomicAdd(&sm.hist[(u2 - lo) >> shift], 1);
      if (u3 >= lo && u3 <= hi) atomicAdd(&sm.hist[(u3 - lo) >> shift], 1);
    }
    for (int64_t e = c4 + threadIdx.x; e < c; e += kSelThreads) {
      const uint32_t u = score_key(__ldcg(s + e));
      if (u >= lo && u <= hi) atomicAdd(&sm.hist[(u - lo) >> shift], 1);
    }
    __syncthreads();
    // Counts from the top: thread j owns bins [4(T-1-j), 4(T-1-j)+4) so that the
    // exclusive scan over threads is a suffix sum over bins.
    const int base_bin = (kSelThreads - 1 - threadIdx.x) * kSelBinsPerThread;
    int loc[kSelBinsPerThread];
    int sum = 0;
#pragma unroll
    for (int q = 0; q < kSelBinsPerThread; ++q) {
      loc[q] = sm.hist[base_bin + kSelBinsPerThread - 1 - q];  // descending bins
      sum += loc[q];
    }
    const int above0 = block_exclusive_scan(sum, sm.warp_sums, &sm.total);
    if (above0 < need && above0 + sum >= need) {
      int above = above0;
#pragma unroll
      for (int q = 0; q < kSelBinsPerThread; ++q) {
        if (above + loc[q] >= need) {
          const int bin = base_bin + kSelBinsPerThread - 1 - q;
          const uint32_t nlo = lo + ((uint32_t)bin << shift);
          const uint32_t span = shift >= 32 ? 0xffffffffu : ((1u << shift) - 1u);
          const uint32_t nhi = (hi - nlo) < span ? hi : nlo + span;
          const int nneed = need - above;
          sm.lo = nlo;
          sm.hi = nhi;
          sm.need = nneed;
          sm.done = (loc[q] == nneed) ? 1 : (nlo == nhi ? 2 : 0);
          break;
        }
        above += loc[q];
      }
    }
    __syncthreads();
    lo = sm.lo;
    hi = sm.hi;
    need = sm.need;
    done = sm.done;
    __syncthreads();
  }

  // Ordered compaction: each thread takes 4 consecutive blocks per round.
  int written = 0, ties_taken = 0;
  for (int64_t e0 = 0; e0 < c; e0 += 4 * kSelThreads) {
    const int64_t e = e0 + 4 * threadIdx.x;
    uint32_t win = 0, tie = 0;
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e + 3 < c) x4 = __ldcg(reinterpret_cast<const float4*>(s + e));
    const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e + q < c) {
        const uint32_t u = score_key(e + 3 < c ? xs[q] : __ldcg(s + e + q));
        if (u > hi || (done == 1 && u >= lo)) win |= 1u << q;
        else if (done == 2 && u == lo) tie |= 1u << q;
      }
    }
    const int n_tie = __popc(tie);
    const int tie_before = ties_taken + block_exclusive_scan(n_tie, sm.warp_sums, &sm.total);
    const int tie_total = sm.total;
    // Ties are taken in block order while the quota lasts.
#pragma unroll
    for (int q = 0, k = 0; q < 4; ++q) {
      if (tie & (1u << q)) {
        if (tie_before + k < need) win |= 1u << q;
        ++k;
      }
    }
    ties_taken += tie_total;
    const int n_win = __popc(win);
    const int before = written + block_exclusive_scan(n_win, sm.warp_sums, &sm.total);
    const int win_total = sm.total;
#pragma unroll
    for (int q = 0, k = 0; q < 4; ++q) {
      if (win & (1u << q)) {
        if (before + k < k_b) out[before + k] = (int32_t)(e + q);  // exactly k_b winners exist
        ++k;
      }
    }
    written += win_total;
  }
}

// S: [n_rows][s_stride] fp32 (row j of this launch is global row row_lo + j);
// idx: [rows][k_b]; count: [rows].
__global__ void __launch_bounds__(kSelThreads)
topk_select_kernel(const float* __restrict__ S, int64_t s_stride, const int64_t* __restrict__ q_pos,
                   int64_t n_q, int64_t row_lo, int r, int k_b, int64_t c_cap,
                   int32_t* __restrict__ idx, int32_t* __restrict__ count) {
  __shared__ SelectSmem sm;
  const int64_t row = row_lo + blockIdx.x;
  const int64_t bb = row / n_q;
  const int64_t pos = q_pos[bb] + row % n_q;
  int64_t c = (pos + 1) / r;
  if (c > c_cap) c = c_cap;  // reported by the scan kernel
  int32_t* out = idx + row * (int64_t)k_b;
  if (c <= k_b) {
    for (int j = threadIdx.x; j < k_b; j += kSelThreads) out[j] = j < c ? j : -1;
    if (threadIdx.x == 0) count[row] = (int32_t)c;
    return;
  }
  cta_select_row(S + (int64_t)blockIdx.x * s_stride, c, k_b, out, sm);
  if (threadIdx.x == 0) count[row] = k_b;
}

cudaError_t launch_topk_select(const float* S, int64_t s_stride, const int64_t* q_pos, int64_t n_q,
                               int64_t row_lo, int64_t n_rows, int r, int k_b, int64_t c_cap,
                               int32_t* idx, int32_t* count, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  topk_select_kernel<<<(unsigned)n_rows, kSelThreads, 0, st>>>(S, s_stride, q_pos, n_q, row_lo, r,
                                                               k_b, c_cap, idx, count);
  return count_launch(cudaGetLastError());
}


// ---------------------------------------------------------------------------------------------
// Two-pass selection for long rows: one pass for a histogram of 1/32-octave
// bins (first_bin, below), one ordered pass that copies every entry at or above the boundary bin
// into shared memory (at most kSelCand entries, in block order); the remaining
// refinement and the emission run on that copy.  Rows whose boundary bin is
// too full fall back to cta_select_row.
constexpr int kSelCand = 4096;

struct SelectFastSmem {
  SelectSmem base;
  uint32_t cu[kSelCand];
  int32_t cb[kSelCand];
};

// Refinement and ordered emission on a candidate copy: sm.cu / sm.cb hold, in
// block order, the ncand entries whose pattern is >= lo; `need` of those in
// [lo, hi] win besides every entry above hi.
__device__ void select_from_candidates(SelectFastSmem& sm, int ncand, uint32_t lo, uint32_t hi, int need, int k_b,
                                       int32_t* __restrict__ out) {
  const int base_bin = (kSelThreads - 1 - threadIdx.x) * kSelBinsPerThread;
  int loc[kSelBinsPerThread];
  int sum = 0;
  // Refine [lo, hi] on the copy (entries > hi are all winners).
  int done = 0;
  for (int guard = 0; !done && guard < 6; ++guard) {
    const uint32_t width = hi - lo;
    const int nbits = 32 - __clz(width);
    const int shift = nbits > 11 ? nbits - 11 : 0;
    for (int j = threadIdx.x; j < kSelBins; j += kSelThreads) sm.base.hist[j] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < ncand; e += kSelThreads) {
      const uint32_t u = sm.cu[e];
      if (u >= lo && u <= hi) atomicAdd(&sm.base.hist[(u - lo) >> shift], 1);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kSelBinsPerThread; ++q) loc[q] = sm.base.hist[base_bin + kSelBinsPerThread - 1 - q];
    sum = loc[0] + loc[1] + loc[2] + loc[3];
    const int ab0 = block_exclusive_scan(sum, sm.base.warp_sums, &sm.base.total);
    if (ab0 < need && ab0 + sum >= need) {
      int above = ab0;
#pragma unroll
      for (int q = 0; q < kSelBinsPerThread; ++q) {
        if (above + loc[q] >= need) {
          const int bin = base_bin + kSelBinsPerThread - 1 - q;
          const uint32_t nlo = lo + ((uint32_t)bin << shift);
          const uint32_t span = (1u << shift) - 1u;
          const uint32_t nhi = (hi - nlo) < span ? hi : nlo + span;
          const int nneed = need - above;
          sm.base.lo = nlo;
          sm.base.hi = nhi;
          sm.base.need = nneed;
          sm.base.done = (loc[q] == nneed) ? 1 : (nlo == nhi ? 2 : 0);
          break;
        }
        above += loc[q];
      }
    }
    __syncthreads();
    lo = sm.base.lo;
    hi = sm.base.hi;
    need = sm.base.need;
    done = sm.base.done;
    __syncthreads();
  }
  // Ordered emission from the copy (already in block order).
  int wr = 0, ties_taken = 0;
  for (int e0 = 0; e0 < ncand; e0 += 4 * kSelThreads) {
    const int e = e0 + 4 * threadIdx.x;
    uint32_t win = 0, tie = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e + q < ncand) {
        const uint32_t u = sm.cu[e + q];
        if (u > hi || (done == 1 && u >= lo)) win |= 1u << q;
        else if (done == 2 && u == lo) tie |= 1u << q;
      }
    }
    const int tie_before = ties_taken + block_exclusive_scan(__popc(tie), sm.base.warp_sums, &sm.base.total);
    const int tie_total = sm.base.total;
#pragma unroll
    for (int q = 0, k = 0; q < 4; ++q) {
      if (tie & (1u << q)) {
        if (tie_before + k < need) win |= 1u << q;
        ++k;
      }
    }
    ties_taken += tie_total;
    const int before = wr + block_exclusive_scan(__popc(win), sm.base.warp_sums, &sm.base.total);
    const int wtot = sm.base.total;
#pragma unroll
    for (int q = 0, k = 0; q < 4; ++q) {
      if (win & (1u << q)) {
        if (before + k < k_b) out[before + k] = sm.cb[e + q];
        ++k;
      }
    }
    wr += wtot;
  }
}

// ---------------------------------------------------------------------------------------------
// The same selection with each row split over a cluster of kSelCluster CTAs
// (decode: few rows, long rows).  Every CTA takes a share of the row: local
// histograms of 1/32-octave bins (first_bin), merged by the first CTA through
// distributed shared memory; ordered copies of the entries at or above the
// boundary bin, gathered into the first CTA's candidate arrays in rank (=
// block) order; that CTA refines and emits.
//
// First-pass bins: 32 per octave of the fp32 score over the 64 octaves
// [2^-30, 2^34), clamped at both ends (bin 0 also holds 0 and everything below
// 2^-30; the last bin everything above).  The top 11 bits of the pattern would
// give 4 bins per octave, so that a row's scores, which span a few octaves,
// fall into about a dozen bins: the shared-memory atomics of the histogram
// then serialise on those bins, and the boundary bin holds several times more
// candidates.
constexpr int kFirstShift = 18;               // 23 - 5 mantissa bits: 32 bins per octave
constexpr int kFirstBase = 97 << 5;           // (biased exponent of 2^-30) x 32
__device__ __forceinline__ int first_bin(uint32_t u) {
  const int b = (int)(u >> kFirstShift) - kFirstBase;
  return b < 0 ? 0 : (b > kSelBins - 1 ? kSelBins - 1 : b);
}
__device__ __forceinline__ uint32_t first_bin_lo(int b) {
  return b == 0 ? 0u : (uint32_t)(b + kFirstBase) << kFirstShift;
}
__device__ __forceinline__ uint32_t first_bin_hi(int b) {
  return b == kSelBins - 1 ? 0x7fffffffu : ((uint32_t)(b + kFirstBase + 1) << kFirstShift) - 1u;
}

template <int kSelCluster>
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads)
topk_select_cluster_kernel(const float* __restrict__ S, int64_t s_stride, const int64_t* __restrict__ q_pos,
                           int64_t n_q, int64_t row_lo, int r, int k_b, int64_t c_cap,
                           int32_t* __restrict__ idx, int32_t* __restrict__ count) {
  namespace cg = cooperative_groups;
  __shared__ SelectFastSmem sm;
  __shared__ int n_local;
  griddep_wait();  // the scores come from the previous kernel
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int64_t lrow = blockIdx.x / kSelCluster;
  const int64_t row = row_lo + lrow;
  const int64_t bb = row / n_q;
  const int64_t pos = q_pos[bb] + row % n_q;
  int64_t c = (pos + 1) / r;
  if (c > c_cap) c = c_cap;
  int32_t* out = idx + row * (int64_t)k_b;
  if (c <= k_b) {  // the same for the whole cluster: nobody touches another CTA's memory
    if (rank == 0) {
      for (int j = threadIdx.x; j < k_b; j += kSelThreads) out[j] = j < c ? j : -1;
      if (threadIdx.x == 0) count[row] = (int32_t)c;
    }
    return;
  }
  const float* s = S + lrow * s_stride;
  // This CTA's part of the row, in batches of kSelThreads x 32 scores; thread
  // t owns the 32 consecutive scores at 32 t of each batch (8 float4 loads in
  // flight, one line per thread).
  const int64_t part = ((c + 32 * kSelCluster - 1) / (32 * kSelCluster)) * 32;
  const int64_t e_lo = c < rank * part ? c : rank * part;
  const int64_t e_hi = c < e_lo + part ? c : e_lo + part;
  auto load_batch = [&](int64_t b0, uint32_t (&u)[32]) {
    const int64_t e = b0 + 32 * (int64_t)threadIdx.x;
    if (e + 32 <= e_hi) {
      float4 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = reinterpret_cast<const float4*>(s + e)[j];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        u[4 * j] = score_key(x[j].x); u[4 * j + 1] = score_key(x[j].y);
        u[4 * j + 2] = score_key(x[j].z); u[4 * j + 3] = score_key(x[j].w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) u[j] = e + j < e_hi ? score_key(s[e + j]) : 0xffffffffu;  // past the end: no bin
    }
  };
  // Pass 1: local histogram of this CTA's part.
  for (int j = threadIdx.x; j < kSelBins; j += kSelThreads) sm.base.hist[j] = 0;
  __syncthreads();
  for (int64_t b0 = e_lo; b0 < e_hi; b0 += 32 * kSelThreads) {
    uint32_t u[32];
    load_batch(b0, u);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (u[j] != 0xffffffffu) atomicAdd(&sm.base.hist[first_bin(u[j])], 1);
  }
  cluster.sync();
  // The first CTA merges the histograms (this thread's bins summed over the
  // cluster), finds the boundary bin and hands it to the other CTAs; they wait
  // at the cluster barrier instead of all reading each other's histograms.
  if (rank == 0) {
    const int base_bin = (kSelThreads - 1 - threadIdx.x) * kSelBinsPerThread;
    int loc[kSelBinsPerThread];
#pragma unroll
    for (int j = 0; j < kSelBinsPerThread; ++j) loc[j] = 0;
#pragma unroll
    for (int q = 0; q < kSelCluster; ++q) {
      const int* h = cluster.map_shared_rank(sm.base.hist, q);
#pragma unroll
      for (int j = 0; j < kSelBinsPerThread; ++j) loc[j] += h[base_bin + kSelBinsPerThread - 1 - j];
    }
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kSelBinsPerThread; ++j) sum += loc[j];
    const int above0 = block_exclusive_scan(sum, sm.base.warp_sums, &sm.base.total);
    if (above0 < k_b && above0 + sum >= k_b) {
      int above = above0;
#pragma unroll
      for (int j = 0; j < kSelBinsPerThread; ++j) {
        if (above + loc[j] >= k_b) {
          const int bin = base_bin + kSelBinsPerThread - 1 - j;
          sm.base.lo = first_bin_lo(bin);
          sm.base.hi = first_bin_hi(bin);
          sm.base.need = k_b - above;
          sm.base.done = above + loc[j];  // entries at or above the bin, whole row
          break;
        }
        above += loc[j];
      }
    }
    __syncthreads();
    if (threadIdx.x > 0 && threadIdx.x < kSelCluster) {  // thread q writes CTA q's copy
      SelectSmem* dst = cluster.map_shared_rank(&sm.base, (int)threadIdx.x);
      dst->lo = sm.base.lo;
      dst->hi = sm.base.hi;
      dst->need = sm.base.need;
      dst->done = sm.base.done;
    }
  }
  cluster.sync();  // the boundary is in every CTA's shared memory; the histograms are no longer read
  const uint32_t lo = sm.base.lo, hi = sm.base.hi;
  const int need = sm.base.need;
  const int ncand = sm.base.done;
  if (ncand > kSelCand) {  // boundary bin too full for the copy: the first CTA takes the whole row
    if (rank == 0) {
      __syncthreads();
      cta_select_row(s, c, k_b, out, sm.base);
      if (threadIdx.x == 0) count[row] = k_b;
    }
    return;
  }
  // Pass 2: ordered copy of this part's entries with pattern >= lo.
  int written = 0;
  for (int64_t b0 = e_lo; b0 < e_hi; b0 += 32 * kSelThreads) {
    uint32_t u[32], take = 0;
    load_batch(b0, u);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (u[j] != 0xffffffffu && u[j] >= lo) take |= 1u << j;
    const int before = written + block_exclusive_scan(__popc(take), sm.base.warp_sums, &sm.base.total);
    const int tot = sm.base.total;
    const int64_t e = b0 + 32 * (int64_t)threadIdx.x;
    int k = before;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if ((take >> j) & 1u) {
        if (k < kSelCand) {
          sm.cu[k] = u[j];
          sm.cb[k] = (int32_t)(e + j);
        }
        ++k;
      }
    }
    written += tot;
  }
  if (threadIdx.x == 0) n_local = written;
  cluster.sync();
  // Append this part's candidates to the first CTA's arrays after the lower ranks'.
  int offset = 0;
  for (int q = 0; q < rank; ++q) offset += *cluster.map_shared_rank(&n_local, q);
  if (rank > 0) {
    uint32_t* du = cluster.map_shared_rank(sm.cu, 0);
    int32_t* db = cluster.map_shared_rank(sm.cb, 0);
    const int n_mine = min(written, kSelCand);
    for (int j = threadIdx.x; j < n_mine; j += kSelThreads) {
      if (offset + j < kSelCand) {
        du[offset + j] = sm.cu[j];
        db[offset + j] = sm.cb[j];
      }
    }
  }
  cluster.sync();  // the first CTA's arrays are complete; the others are done
  if (rank != 0) return;
  select_from_candidates(sm, ncand, lo, hi, need, k_b, out);
  if (threadIdx.x == 0) count[row] = k_b;
}

// Clusters of 4 CTAs per row, or of 8 when fewer than 64 rows share the GPU
// (a multi-token decode step of a few long sequences).
cudaError_t launch_topk_select_cluster(const float* S, int64_t s_stride, const int64_t* q_pos, int64_t n_q,
                                       int64_t row_lo, int64_t n_rows, int r, int k_b, int64_t c_cap,
                                       int32_t* idx, int32_t* count, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (n_rows < 64)
    return count_launch(launch_dependent(topk_select_cluster_kernel<8>, dim3((unsigned)(n_rows * 8)),
                                         dim3(kSelThreads), 0, st, S, s_stride, q_pos, n_q, row_lo, r, k_b, c_cap,
                                         idx, count));
  return count_launch(launch_dependent(topk_select_cluster_kernel<4>, dim3((unsigned)(n_rows * 4)),
                                       dim3(kSelThreads), 0, st, S, s_stride, q_pos, n_q, row_lo, r, k_b, c_cap, idx,
                                       count));
}


}  // namespace qsa
