// Fused QSA indexer for prefill: block scores on the tcgen05 tensor cores and an
// exact top-k_B per query row, without storing the score matrix.
//
// "On the Design of Qwen3.8-Next Architecture", research-hub notes, Key ideas,
// QSA compressed-indexer bullet: I_ib = sum_h ReLU(<q_i^h, kbar_b>) over the 4
// indexer heads, top k_B = ceil(K / r) blocks per query; paperglide reader,
// "Qwen Sparse Attention" step 3 (block-causal mask) and step 4 (top-K_B).
//
// Layout of the work.  A persistent CTA takes tiles of 48 consecutive query
// tokens of one sequence.  A chunk is 128 compressed blocks: 8 tcgen05 MMAs
// (16 head dims each) compute D[row][token * 4 + head] = <kbar_block(row),
// qt_token^head>: M = 128 rows (A = the kbar chunk, streamed through a 3-stage
// TMA ring), N = 192 (B = the tile's 48 x 4 rotated query rows, loaded once per
// tile), fp32 accumulators in TMEM (two buffers, 256 columns apart).  The tile's
// visible blocks are split into 4 consecutive regions of R = 32 x nchunks
// blocks; rows 32 q .. 32 q + 31 of chunk x hold blocks q R + 32 x .. + 31, so
// TMEM lane quarter q walks region q in order.  A TMEM lane holds the four
// heads of each token in adjacent columns: a thread finishes two scores with
// 8 adds x + |x| (= 2 ReLU(x)) and 3 packed two-lane fp32 adds.
//
// Exact selection in one pass over the blocks.
//   1. Pilot: a strided sample of the tile's blocks (every 16th block, in one
//      or more phases) is scored first and binned per token into 512 bins of
//      1/16 octave of the fp32 score (16-bit counters, two per word).  From it
//      each token takes a threshold tau above which about sqrt(k_B kFCap) of
//      its scores are expected (interpolated inside the bin where the count is
//      reached).
//   2. Collect: every chunk is scored; each (token, block) with score >= tau is
//      appended (bit pattern u of 2 x score, block id) to the token's buffer in
//      global memory: one segment per TMEM lane quarter, so that no two warps
//      share a counter.  Segment q lists region q in ascending block order, so
//      the 4 segments read in turn are in block order.  Counts are stored when
//      the tile is done.
//   3. Finalize (a separate kernel, one warp per row): if the buffer holds
//      between k_B and kFCap entries it contains the whole top-k_B; a radix
//      descent on u finds the k_B-th value, equal values go to the lower block
//      ids, and the winners, compacted in entry order, come out sorted by block
//      id.  Rows whose buffer fell outside that range are queued for the exact
//      fallback kernel (score the whole row, radix-select it), so the result is
//      always exact.
// Twelve score warps (three per TMEM lane quarter, 16 tokens each) read the
// accumulators; the host launches the kernel over ranges of at most
// kTilesPerLaunch tiles so that the entry buffers stay bounded.
//
// Every wait is a bounded mbarrier wait; on timeout the CTA raises its abort
// flag, every role leaves its loop, in-flight copies and MMAs are waited for
// (bounded), TMEM is freed and the device error word reports the timeout.
#include <cudaTypedefs.h>

#include <cmath>

#include "common.cuh"
#include "sm100.cuh"

namespace qsa {

constexpr int kTT = 48;                  // query tokens per tile (most; 24 with 8 indexer heads)
constexpr int kNRows = 192;              // largest MMA N (token, head rows) of a tile
constexpr int kMB = 128;                 // blocks per chunk: MMA M
constexpr int kAStages = 3;              // kbar TMA ring depth
constexpr int kEpiWarps = 12;            // 3 per TMEM lane quarter, 16 tokens each
constexpr int kFThreads = 32 * (2 + kEpiWarps);              // 448: 128 registers per thread
constexpr uint32_t kAccCols = 256;                           // TMEM columns between the two accumulators
constexpr uint32_t kTmemCols = 2 * kAccCols;                 // 512
constexpr int kPBins = 512;              // pilot bins (1/16 octave), packed 2 per word
constexpr int kPShift = 19;              // bits below the bin index
constexpr int kPBase = 1920;             // (bits of 2^-7) >> 19: bins of 2 x score start at 2^-7
constexpr int kFinRegs = 40;             // entries per lane in finalize
constexpr int kFCap = 32 * kFinRegs;     // 1280 (2.5 k_B at k_B = 512): most entries a token may collect
constexpr int kSeg = kFCap;              // entries per (token, TMEM lane quarter) segment: a
                                         // quarter may hold all of a row's entries
constexpr int kFMaxKb = 512;             // largest k_B the fused path handles
constexpr int kFMaxCtas = 160;           // >= SM count; sizes the buffers
constexpr int kFMinRows = 64;            // fewer query rows per sequence: scan path
constexpr int kFbCtas = 148;             // fallback kernel CTAs (one row each at a time)
constexpr int kTilesPerLaunch = 1024;    // tiles per fused launch (bounds the row buffers: 1.9 GiB each)
constexpr uint32_t kABytes = kMB * 128 * 2;     // 32 KB

// Tile shape for H indexer heads: TT query tokens, NR = TT H MMA columns
// (token-major, the H heads of a token adjacent), TPW tokens and CPW = TPW H
// accumulator columns per score warp (three warps per TMEM lane quarter).
template <int H>
struct FusedShape {
  static constexpr int TT = H == 8 ? 24 : 48;
  static constexpr int NR = TT * H;
  static constexpr int TPW = TT / 3;
  static constexpr int CPW = TPW * H;
  static constexpr uint32_t BBytes = NR * 128 * 2;
  static_assert(NR % 16 == 0 && NR <= kNRows && TPW % 4 == 0, "tile shape");
};

// Tokens per tile for H indexer heads (host and device).
__host__ __device__ constexpr int fused_tile_tokens(int H) { return H == 8 ? 24 : 48; }

struct FusedSmem {
  uint8_t a[kAStages][2][kMB * 128];   // kbar chunk, dims 0-63 | 64-127 (SW128)
  uint8_t b[2][kNRows * 128];          // rotated queries of the tile, same split
  uint32_t phist[kTT][kPBins / 2];     // pilot counts, two 16-bit bins per word
  uint32_t tau[kTT];
  uint64_t a_full[kAStages], a_empty[kAStages];
  uint64_t tfull[2], tempty[2];
  uint64_t b_full, b_empty, pilot_bar, tau_bar, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kFusedSmemBytes = sizeof(FusedSmem) + 1024;  // + alignment slack

struct TileMeta {
  int64_t bb, tok0, i0;
  int nvalid;
  int nchunks;   // chunks of kMB blocks covering the last row's visible blocks
  int ngroups;   // complete 16-block groups visible to the last row
  int mc;        // pilot chunks per phase: ceil(ngroups / kMB)
  int nphase;    // pilot phases p: blocks 16 m + p are sampled
  int npilot;    // nphase * mc pilot chunks
  bool mma;
};

constexpr int kPilotStride = 16;   // the pilot samples every 16th block (per phase)
// At least this many pilot samples per row when possible: with the aim below
// about 50 samples are expected above a row's threshold at every context
// length (one phase of every 16th block gives c / 16 samples, and aim / 16 of
// them above).  Measured at 128K and 32K: 1024 took 1% and 5% longer (more
// phases for rows below 16384 visible blocks); 384 or 256 sent one or two of
// the 32K rows to the exact fallback, whose full-row scoring cost more than
// the pilot saved; 2048 spent 15% of the 128K chunks on the pilot.
constexpr int kPilotMin = 512;
// tau aims at sqrt(k_B kFCap) entries per row, the middle in ratio of the
// accepted [k_B, kFCap]: 1.6 k_B at k_B = 512, 3.2 k_B at k_B = 128, where the
// quantile sought lies further in the tail and the pilot's estimate of it is
// noisier (never below 1.6 k_B).  Aims of 0.92 and 0.85 times this sent 49
// and 620 of the 128K rows to the exact fallback (4% and 18% slower).
inline int pilot_aim(int k_b) {
  const double g = std::sqrt((double)k_b * kFCap), lo = 1.6 * k_b;
  return (int)((g > lo ? g : lo) + 0.5);
}

template <int TT>
__device__ __forceinline__ TileMeta tile_meta(int64_t t, int64_t tiles_per_seq, int64_t n_q,
                                              const int64_t* q_pos, int rshift, int k_b, int64_t c_cap) {
  TileMeta m;
  m.bb = t / tiles_per_seq;
  m.tok0 = (t % tiles_per_seq) * TT;
  const int64_t rem = n_q - m.tok0;
  m.nvalid = rem < TT ? (int)rem : TT;
  m.i0 = q_pos[m.bb] + m.tok0;
  int64_t c = (m.i0 + m.nvalid) >> rshift;
  if (c > c_cap) c = c_cap;
  m.mma = c > k_b;
  m.nchunks = (int)((c + kMB - 1) / kMB);
  m.ngroups = (int)(c / kPilotStride);
  m.mc = (m.ngroups + kMB - 1) / kMB;
  if (m.ngroups == 0) {
    m.nphase = 0;
  } else {
    int np = (kPilotMin + m.ngroups - 1) / m.ngroups;
    m.nphase = np < 1 ? 1 : (np > kPilotStride ? kPilotStride : np);
  }
  m.npilot = m.nphase * m.mc;
  return m;
}

__device__ __forceinline__ int64_t token_c(const TileMeta& m, int t, int rshift, int64_t c_cap) {
  int64_t c = (m.i0 + t + 1) >> rshift;
  return c > c_cap ? c_cap : c;
}

// Bounded wait executed by every lane of a warp; the outcome is made uniform so
// that a warp never splits across a collective (TMEM loads, shuffles).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned sleep_ns = 0) {
  const bool w = sm100::mbar_wait(bar, parity, abort_flag, sm100::kWaitCycles, sleep_ns);
  return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ int range_shift(uint32_t lo, uint32_t hi) {
  const int nb = 32 - __clz(hi - lo);
  return nb > 9 ? nb - 9 : 0;
}

// One refinement round: `hist` holds the 512-bin histogram of the entries in
// [lo, hi]; keep the bin where the count from the top reaches `need`.  mode
// becomes 1 (every entry of the new range wins), 2 (single value: `need` of its
// entries win) or stays 0.
__device__ __forceinline__ void refine_round(uint32_t* hist, uint32_t& lo, uint32_t& hi, int& need,
                                             int& mode, int shift) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const int base_bin = (31 - lane) * 16;  // lane owns 16 bins, scanned from the top
  int loc[16], sum = 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    loc[q] = (int)hist[base_bin + 15 - q];
    sum += loc[q];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int above0 = incl - sum;
  const bool cross = above0 < need && above0 + sum >= need;
  const unsigned who = __ballot_sync(0xffffffffu, cross);
  uint32_t nlo = 0, nhi = 0;
  int nneed = 0, nmode = 0;
  if (cross) {
    int above = above0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (above + loc[q] >= need) {
        const int bin = base_bin + 15 - q;
        const uint32_t l = lo + ((uint32_t)bin << shift);
        const uint32_t span = (1u << shift) - 1u;
        nlo = l;
        nhi = (hi - l) < span ? hi : l + span;
        nneed = need - above;
        nmode = (loc[q] == nneed) ? 1 : (nlo == nhi ? 2 : 0);
        break;
      }
      above += loc[q];
    }
  }
  const int src = who ? __ffs(who) - 1 : 0;
  lo = __shfl_sync(0xffffffffu, nlo, src);
  hi = __shfl_sync(0xffffffffu, nhi, src);
  need = __shfl_sync(0xffffffffu, nneed, src);
  mode = who ? __shfl_sync(0xffffffffu, nmode, src) : 1;  // cannot happen; stop safely
  __syncwarp();
}

// Entry e of a token's buffer: its 4 segments (one per TMEM lane quarter,
// kSeg entries apart) holding n0, p2 - p1, p3 - p2, ... entries, read as one list.
__device__ __forceinline__ const uint2* entry_ptr(const uint2* seg, int e, int p1, int p2, int p3) {
  const int q = (e >= p1) + (e >= p2) + (e >= p3);
  const int off = e - (q == 0 ? 0 : (q == 1 ? p1 : (q == 2 ? p2 : p3)));
  return seg + q * kSeg + off;
}

// Exact top-k_b of a token's buffer (n entries, k_b <= n <= kFCap): the k_b
// largest patterns, equal patterns going to the lower block ids; the winners
// are written to out[] sorted by block id.  One warp.  The patterns stay in
// registers (entry e = lane + 32 j in slot j), the block ids in ids[e].  Each
// segment lists its quarter's blocks in ascending order and the quarters cover
// consecutive block ranges, so entry order is block order.
__device__ __forceinline__ void finalize_row(const uint2* __restrict__ seg, int p1, int p2, int p3, int n,
                                             int k_b, uint32_t* __restrict__ hist,
                                             int32_t* __restrict__ ids, int32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  uint32_t ru[kFinRegs];
#pragma unroll
  for (int j0 = 0; j0 < kFinRegs; j0 += 16) {  // up to 16 loads in flight per lane
    uint2 xs[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int e = lane + 32 * (j0 + jj);
      xs[jj] = (j0 + jj < kFinRegs && e < n) ? __ldcs(entry_ptr(seg, e, p1, p2, p3)) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      if (j0 + jj < kFinRegs) {  // resolved at compile time
        const int e = lane + 32 * (j0 + jj);
        ru[j0 + jj] = xs[jj].x;
        if (e < n) ids[e] = (int32_t)xs[jj].y;
      }
    }
  }
  // Start from the buffer's own pattern range, so the first round's bins are
  // spread over the entries (they all lie within a few octaves of tau).
  uint32_t lo = 0xffffffffu, hi = 0;
#pragma unroll
  for (int j = 0; j < kFinRegs; ++j) {
    if (lane + 32 * j < n) {
      lo = min(lo, ru[j]);
      hi = max(hi, ru[j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  int need = k_b, mode = (lo == hi) ? 2 : 0;
  for (int guard = 0; mode == 0 && guard < 6; ++guard) {  // the range shrinks 2^9-fold per round
    const int shift = range_shift(lo, hi);
#pragma unroll
    for (int j = 0; j < 4; ++j) reinterpret_cast<uint4*>(hist)[lane + 32 * j] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kFinRegs; ++j)
      if (lane + 32 * j < n && ru[j] >= lo && ru[j] <= hi) atomicAdd(&hist[(ru[j] - lo) >> shift], 1u);
    refine_round(hist, lo, hi, need, mode, shift);
  }
  __syncwarp();
  // Ties at a single value: keep the `need` lowest block ids among them.
  uint32_t tie_cut = 0xffffffffu;  // tied entries with block id < tie_cut win
  if (mode == 2) {
    int nt = 0;
#pragma unroll
    for (int j = 0; j < kFinRegs; ++j) nt += (lane + 32 * j < n && ru[j] == lo) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o);
    if (nt > need) {
      // Radix descent on 0x7fffffff - id (ids are distinct), so the largest
      // keys are the smallest ids.
      uint32_t blo = 0, bhi = 0x7fffffffu;
      int bneed = need, bmode = 0;
      for (int guard = 0; bmode == 0 && guard < 6; ++guard) {
        const int shift = range_shift(blo, bhi);
        for (int j = lane; j < 512; j += 32) hist[j] = 0;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kFinRegs; ++j) {
          const int e = lane + 32 * j;
          if (e < n && ru[j] == lo) {
            const uint32_t key = 0x7fffffffu - (uint32_t)ids[e];
            if (key >= blo && key <= bhi) atomicAdd(&hist[(key - blo) >> shift], 1u);
          }
        }
        refine_round(hist, blo, bhi, bneed, bmode, shift);
      }
      // With distinct keys the descent ends with every key of [blo, bhi]
      // winning: key >= blo  <=>  id <= 0x7fffffff - blo.
      tie_cut = 0x7fffffffu - blo + 1u;
    }
  }
  // Entry order is block order, so compacting the k_b winners in entry order
  // lists them sorted.
  int written = 0;
#pragma unroll
  for (int j = 0; j < kFinRegs; ++j) {
    if (32 * j >= n) break;
    const int e = lane + 32 * j;
    bool win = false;
    if (e < n) {
      win = ru[j] > hi || (mode == 1 && ru[j] >= lo);
      if (!win && mode == 2 && ru[j] == lo) win = (uint32_t)ids[e] < tie_cut;
    }
    const unsigned wm = __ballot_sync(0xffffffffu, win);
    const int pos = written + __popc(wm & ((1u << lane) - 1u));
    if (win && pos < k_b) out[pos] = ids[e];
    written += __popc(wm);
  }
  for (int i = (written < k_b ? written : k_b) + lane; i < k_b; i += 32) out[i] = -1;
  __syncwarp();
}

// ---------------------------------------------------------------------------------------------
// Threshold of one token from its pilot histogram (one warp).  want =
// ceil(aim P / c) of the P samples should lie at or above
// tau: the bin where the count from the top reaches want is found, and tau is
// placed inside it by linear interpolation, as if its samples were spread
// evenly over its value range (the bins are 1/16 octave wide, and in the far
// tail of a row's scores one bin can hold as many samples as all the bins above
// it).  tau is 0 when the bottom bin is reached or the row has no samples,
// which collects every visible block.  The histogram is cleared for the next
// tile.  Lane L owns bins 16 (31 - L) .. + 15.
__device__ __forceinline__ uint32_t pilot_tau(uint32_t* __restrict__ hist, int64_t c, int aim) {
  const int lane = threadIdx.x & 31;
  uint4* const w4 = reinterpret_cast<uint4*>(hist + 8 * (31 - lane));
  const uint4 lo4 = w4[0], hi4 = w4[1];
  const uint32_t wd[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
  w4[0] = make_uint4(0, 0, 0, 0);
  w4[1] = make_uint4(0, 0, 0, 0);
  int loc[16], sum = 0;  // loc[q]: bin 16 (31 - lane) + 15 - q
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int j = 15 - q;
    loc[q] = (int)((j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xffffu));
    sum += loc[q];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int64_t P = __shfl_sync(0xffffffffu, incl, 31);
  int64_t want = ((int64_t)aim * P + c - 1) / c;
  if (want < 1) want = 1;
  const int above0 = incl - sum;
  const bool cross = above0 < want && incl >= want;
  uint32_t tau = 0;
  if (cross) {
    // The first of the lane's bins (from the top) where the count reaches want:
    // its index, the count above it and its own count (no early exit, so that
    // loc[] stays in registers).
    int above = above0, bin = -1, b_above = 0, b_cnt = 1;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (bin < 0 && above + loc[q] >= want) {
        bin = 16 * (31 - lane) + 15 - q;
        b_above = above;
        b_cnt = loc[q];
      }
      above += loc[q];
    }
    if (bin > 0) {
      tau = (uint32_t)(kPBase + bin) << kPShift;  // lower edge
      if (bin < kPBins - 1) {  // the top bin is open above: keep its lower edge
        const float lo = __uint_as_float(tau);
        const float hi = __uint_as_float((uint32_t)(kPBase + bin + 1) << kPShift);
        const float f = (float)(want - b_above) / (float)b_cnt;  // in (0, 1]
        tau = __float_as_uint(hi - f * (hi - lo));                // in [lo, hi]
      }
    }
  }
  const unsigned who = __ballot_sync(0xffffffffu, cross);
  return who ? __shfl_sync(0xffffffffu, tau, __ffs(who) - 1) : 0u;
}

// Tile order of a CTA: the k-th tile it takes is round k of a snake over the
// launch's tiles, heaviest (latest positions) first, so that the per-CTA sums
// of the (position-proportional) tile costs stay level.  -1: no tile.
__device__ __forceinline__ int64_t tile_order(int64_t k, int64_t t_count) {
  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t kk = k * G + ((k & 1) ? G - 1 - b : b);
  return kk < t_count ? t_count - 1 - kk : -1;
}

template <int H>
__global__ void __launch_bounds__(kFThreads, 1)
index_topk_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_kp, const int64_t* __restrict__ q_pos,
                        int64_t n_q, int64_t tiles_per_seq, int64_t t_begin, int64_t t_count, int rshift,
                        int k_b, int aim, int64_t c_cap, uint2* __restrict__ buf, int* __restrict__ cnt) {
  using namespace sm100;
  using Sh = FusedShape<H>;
  constexpr int TT = Sh::TT, TPW = Sh::TPW, CPW = Sh::CPW;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* const smem_base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  FusedSmem& S = *reinterpret_cast<FusedSmem*>(smem_base);
  // The finalize of the previous launch's range is launched dependent on this
  // kernel: it may start now, on the registers and shared memory this CTA
  // leaves free on its SM.  It reads only the other entry buffer.
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.abort_flag;
  const int64_t rounds = (t_count + gridDim.x - 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&S.a_full[s], 1);
      mbar_init(&S.a_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S.tfull[a], 1);
      mbar_init(&S.tempty[a], kEpiWarps);
    }
    mbar_init(&S.b_full, 1);
    mbar_init(&S.b_empty, 1);
    mbar_init(&S.pilot_bar, kEpiWarps);
    mbar_init(&S.tau_bar, kEpiWarps);
    mbar_init(&S.mma_done, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  for (int j = threadIdx.x; j < TT * (kPBins / 2); j += kFThreads) (&S.phist[0][0])[j] = 0;
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_kp);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, b_uses = 0;
      bool ok = true;
      for (int64_t k = 0; ok && k < rounds; ++k) {
        const int64_t lt = tile_order(k, t_count);
        if (lt < 0) continue;
        const TileMeta m = tile_meta<TT>(t_begin + lt, tiles_per_seq, n_q, q_pos, rshift, k_b, c_cap);
        if (!m.mma) continue;
        if (!mbar_wait(&S.b_empty, (b_uses & 1) ^ 1, abort_flag, kWaitCycles, 128)) { ok = false; break; }
        ++b_uses;
        mbar_arrive_expect_tx(&S.b_full, Sh::BBytes);
        const int qrow = (int)((m.bb * n_q + m.tok0) * H);
        tma_load_2d(S.b[0], &tm_q, &S.b_full, 0, qrow);
        tma_load_2d(S.b[1], &tm_q, &S.b_full, 64, qrow);
        const int total = m.npilot + m.nchunks;
        int pph = 0, pkc = 0;  // phase and column of the next pilot chunk
        for (int x = 0; x < total; ++x, ++it) {
          const int st = it % kAStages;
          if (!mbar_wait(&S.a_empty[st], ((it / kAStages) & 1) ^ 1, abort_flag, kWaitCycles, 64)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.a_full[st], kABytes);
          if (x < m.npilot) {  // blocks 16 (kMB kc + row) + ph
            const int ph = pph, kc = pkc;
            if (++pkc == m.mc) {
              pkc = 0;
              ++pph;
            }
            tma_load_4d(S.a[st][0], &tm_kp, &S.a_full[st], 0, ph, kc * kMB, (int)m.bb);
            tma_load_4d(S.a[st][1], &tm_kp, &S.a_full[st], 64, ph, kc * kMB, (int)m.bb);
          } else {
            // Rows 32 q .. 32 q + 31 of the chunk: blocks q R + 32 ch + j of region q.
            const int ch = x - m.npilot, R = m.nchunks * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              tma_load_3d(S.a[st][0] + q * 4096, &tm_k, &S.a_full[st], 0, q * R + ch * 32, (int)m.bb);
              tma_load_3d(S.a[st][1] + q * 4096, &tm_k, &S.a_full[st], 64, q * R + ch * 32, (int)m.bb);
            }
          }
        }
      }
      if (!ok) {
        volatile int never = 0;  // wait (bounded) for copies still in flight
        for (uint32_t j = (it > kAStages ? it - kAStages : 0); j < it; ++j)
          mbar_wait(&S.a_full[j % kAStages], (j / kAStages) & 1, &never, 100000000LL);
        if (b_uses > 0) mbar_wait(&S.b_full, (b_uses - 1) & 1, &never, 100000000LL);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kMB, Sh::NR);
      uint32_t it = 0, ct = 0, b_uses = 0;
      bool ok = true;
      const uint32_t b0 = smem_u32(S.b[0]), b1 = smem_u32(S.b[1]);
      for (int64_t k = 0; ok && k < rounds; ++k) {
        const int64_t lt = tile_order(k, t_count);
        if (lt < 0) continue;
        const TileMeta m = tile_meta<TT>(t_begin + lt, tiles_per_seq, n_q, q_pos, rshift, k_b, c_cap);
        if (!m.mma) continue;
        if (!mbar_wait(&S.b_full, b_uses & 1, abort_flag, kWaitCycles, 64)) { ok = false; break; }
        ++b_uses;
        tc_fence_after();
        const int total = m.npilot + m.nchunks;
        for (int x = 0; x < total; ++x, ++it, ++ct) {
          const int st = it % kAStages;
          const int acc = ct & 1;
          if (!mbar_wait(&S.a_full[st], (it / kAStages) & 1, abort_flag, kWaitCycles, 32)) { ok = false; break; }
          if (!mbar_wait(&S.tempty[acc], ((ct >> 1) & 1) ^ 1, abort_flag, kWaitCycles, 32)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(S.a[st][0]), a1 = smem_u32(S.a[st][1]);
          const uint32_t d = tmem + (uint32_t)acc * kAccCols;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk < 4 ? a0 : a1) + (uint32_t)((kk & 3) * 32);
            const uint32_t boff = (kk < 4 ? b0 : b1) + (uint32_t)((kk & 3) * 32);
            umma_bf16(d, desc_kmajor_sw128(aoff), desc_kmajor_sw128(boff), idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&S.a_empty[st]);
          umma_commit(&S.tfull[acc]);
        }
        if (ok) umma_commit(&S.b_empty);
      }
      umma_commit(&S.mma_done);  // every MMA completes before TMEM is released
      volatile int never = 0;
      mbar_wait(&S.mma_done, 0, &never, 100000000LL);
    }
  } else {
    // ------------------------------------------------------------ score warps
    const int ew = warp - 2;            // 0..11
    const int q4 = warp & 3;            // TMEM lane quarter: blocks 32 q4 .. 32 q4 + 31 of a chunk
    const int h = ew >> 2;              // tokens TPW h .. TPW h + TPW - 1 (TMEM columns CPW h ..)
    const int cap32 = (int)(c_cap < 0x7fffffff ? c_cap : 0x7fffffff);
    uint32_t ct = 0, pilot_n = 0;
    bool ok = true;
    for (int64_t k = 0; ok && k < rounds; ++k) {
      const int64_t lt = tile_order(k, t_count);
      if (lt < 0) continue;
      const TileMeta m = tile_meta<TT>(t_begin + lt, tiles_per_seq, n_q, q_pos, rshift, k_b, c_cap);
      if (!m.mma) continue;
      // Token TPW h + j sits at position posw + j.
      const int posw = (int)(m.i0 + TPW * h);
      const int cminw = min((posw + 1) >> rshift, cap32);  // smallest c of the warp's tokens
      // Segment of (token TPW h + j, this warp's lane quarter): seg0 + j * 4 kSeg.
      uint2* const seg0 = buf + ((lt * TT + TPW * h) * 4 + q4) * kSeg;
      // Thresholds and entry counts of the warp's tokens (the same in every lane).
      uint32_t tauw[TPW];
      int cntw[TPW];
#pragma unroll
      for (int k2 = 0; k2 < TPW; ++k2) {
        tauw[k2] = 0xffffffffu;
        cntw[k2] = 0;
      }
      const int total = m.npilot + m.nchunks;
      int pph = 0, pkc = 0;  // phase and column of the next pilot chunk
      for (int x = 0; x < total; ++x, ++ct) {
        const bool pilot = x < m.npilot;
        if (x == m.npilot) {
          // ---- pilot done: thresholds of tokens ew, ew + kEpiWarps, ...
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.pilot_bar);
          if (!warp_wait(&S.pilot_bar, pilot_n & 1, abort_flag)) { ok = false; break; }
#pragma unroll 1
          for (int t = ew; t < TT; t += kEpiWarps) {
            const int64_t c = token_c(m, t, rshift, c_cap);
            // Rows that do not select (past the end, or c <= k_B) collect nothing.
            const uint32_t tau = pilot_tau(S.phist[t], c, aim);
            if (lane == 0) S.tau[t] = (t < m.nvalid && c > k_b) ? tau : 0xffffffffu;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.tau_bar);
          if (!warp_wait(&S.tau_bar, pilot_n & 1, abort_flag)) { ok = false; break; }
#pragma unroll
          for (int k4 = 0; k4 < TPW / 4; ++k4) {
            const uint4 t4 = *reinterpret_cast<const uint4*>(&S.tau[TPW * h + 4 * k4]);
            tauw[4 * k4] = t4.x;
            tauw[4 * k4 + 1] = t4.y;
            tauw[4 * k4 + 2] = t4.z;
            tauw[4 * k4 + 3] = t4.w;
          }
          ++pilot_n;
        }
        const int acc = ct & 1;
        if (!warp_wait(&S.tfull[acc], (ct >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();

        // The CPW accumulator columns of this warp's TPW tokens are reduced to
        // TPW scores in registers, and the accumulator is handed back to the
        // MMA warp at once.  x + |x| is 2 ReLU(x) exactly and doubling
        // commutes with the rounding of the sums, so the bit patterns of
        // 2 x score order exactly as the scores do.
        uint32_t uw[TPW];
        {
          const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)acc * kAccCols + (uint32_t)(CPW * h);
          if constexpr (H == 4) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              uint32_t v[32];
              tmem_ld32(taddr + (uint32_t)(32 * g), v);
              tmem_ld_wait();
#pragma unroll
              for (int kk = 0; kk < 8; kk += 2) {  // two tokens at a time: packed fp32 pair adds
                float rr[2][4];
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                  for (int hh = 0; hh < 4; ++hh) {
                    const float a = __uint_as_float(v[4 * (kk + e) + hh]);
                    rr[e][hh] = a + fabsf(a);
                  }
                const float2 s01 = __fadd2_rn(make_float2(rr[0][0], rr[1][0]), make_float2(rr[0][1], rr[1][1]));
                const float2 s23 = __fadd2_rn(make_float2(rr[0][2], rr[1][2]), make_float2(rr[0][3], rr[1][3]));
                const float2 tot = __fadd2_rn(s01, s23);
                uw[8 * g + kk] = __float_as_uint(tot.x);
                uw[8 * g + kk + 1] = __float_as_uint(tot.y);
              }
            }
          } else if constexpr (CPW == 16) {  // one head: 16 columns, one per token
            uint32_t v[16];
            tmem_ld16(taddr, v);
            tmem_ld_wait();
#pragma unroll
            for (int k2 = 0; k2 < TPW; ++k2) {
              const float a = __uint_as_float(v[k2]);
              uw[k2] = __float_as_uint(a + fabsf(a));
            }
          } else {  // 32 columns per load: 32 / H tokens of H heads, summed in head order
#pragma unroll
            for (int g = 0; g < CPW / 32; ++g) {
              uint32_t v[32];
              tmem_ld32(taddr + (uint32_t)(32 * g), v);
              tmem_ld_wait();
#pragma unroll
              for (int kk = 0; kk < 32 / H; ++kk) {
                float sum = 0.f;
#pragma unroll
                for (int hh = 0; hh < H; ++hh) {
                  const float a = __uint_as_float(v[H * kk + hh]);
                  sum += a + fabsf(a);
                }
                uw[(32 / H) * g + kk] = __float_as_uint(sum);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.tempty[acc]);
        }
        // Blocks of this warp's lanes: main chunk ch holds blocks gbase + lane,
        // gbase = q4 R + 32 ch (the quarter's own region of R = 32 nchunks
        // blocks); pilot chunks hold blocks 16 (gbase + lane) + ph, gbase = kMB kc + 32 q4.
        const int ph = pilot ? pph : 0;
        const int gbase = pilot ? pkc * kMB + 32 * q4 : q4 * (m.nchunks * 32) + (x - m.npilot) * 32;
        if (pilot && ++pkc == m.mc) {  // pilot chunk x is phase x / mc, column x % mc
          pkc = 0;
          ++pph;
        }
        const int bi = pilot ? (gbase + lane) * kPilotStride + ph : gbase + lane;
        // Every block of the warp is visible to all its tokens when they end
        // below the first token's visible range.
        const int warp_last = pilot ? (m.mc * kMB) * kPilotStride : gbase + 32;
        const bool chunk_all_visible = warp_last <= cminw;
        // Lanes (blocks) token TPW h + k2 sees in a main chunk: a prefix of the
        // warp, as block ids grow with the lane.  Tokens that do not select are
        // excluded by their threshold.
        auto vis_mask = [&](int k2) -> unsigned {
          if (chunk_all_visible) return 0xffffffffu;
          int c = (posw + k2 + 1) >> rshift;
          c = c < cap32 ? c : cap32;
          const int lim = c - gbase;
          return lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : (1u << lim) - 1u);
        };
        if (pilot) {
          // The sample is every sampled block the tile's last row sees: the
          // visible ranges of the tile's rows differ by at most 12 blocks, and
          // tau only sets the fraction of a row's scores to collect.  The
          // collect pass applies each row's exact range.
          if (gbase + lane < m.ngroups) {
#pragma unroll
            for (int k2 = 0; k2 < TPW; ++k2) {
              int bin = (int)(uw[k2] >> kPShift) - kPBase;
              bin = bin < 0 ? 0 : (bin > kPBins - 1 ? kPBins - 1 : bin);
              atomicAdd(&S.phist[TPW * h + k2][bin >> 1], (bin & 1) ? 65536u : 1u);
            }
          }
        } else {
          {  // nearly every chunk has some pair above tau, so no pre-check
            const unsigned lt_mask = (1u << lane) - 1u;
            if (chunk_all_visible) {
#pragma unroll
              for (int k2 = 0; k2 < TPW; ++k2) {
                const bool mine = uw[k2] >= tauw[k2];
                const unsigned tmk = __ballot_sync(0xffffffffu, mine);
                // An overflowing segment writes its last slot; its count keeps
                // growing, and the finalize sends such a row to the fallback.
                const int pos = min(cntw[k2] + __popc(tmk & lt_mask), kSeg - 1);
                if (mine) seg0[k2 * 4 * kSeg + pos] = make_uint2(uw[k2], (uint32_t)bi);
                cntw[k2] += __popc(tmk);
              }
            } else {
#pragma unroll
              for (int k2 = 0; k2 < TPW; ++k2) {
                const unsigned tmk = __ballot_sync(0xffffffffu, uw[k2] >= tauw[k2]) & vis_mask(k2);
                const int pos = min(cntw[k2] + __popc(tmk & lt_mask), kSeg - 1);
                if ((tmk >> lane) & 1u) seg0[k2 * 4 * kSeg + pos] = make_uint2(uw[k2], (uint32_t)bi);
                cntw[k2] += __popc(tmk);
              }
            }
          }
        }
      }
      if (!ok) break;
      // ---- tile done: this warp's entry counts go to the finalize kernel
      if (lane == 0) {
        int4* const dst = reinterpret_cast<int4*>(cnt + (lt * 4 + q4) * TT + TPW * h);
#pragma unroll
        for (int k4 = 0; k4 < TPW / 4; ++k4)
          dst[k4] = make_int4(cntw[4 * k4], cntw[4 * k4 + 1], cntw[4 * k4 + 2], cntw[4 * k4 + 3]);
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Selection of every query row of a launch's tiles, one warp per row: rows that
// see at most k_B blocks keep all of them (-1 padding); the others take the
// exact top-k_B of the entries their tile collected (finalize_row), or are
// queued for the exact fallback kernel when their buffer fell outside
// [k_B, kFCap] entries or a segment overflowed.
// W warps per CTA: 4 (four CTAs per SM) for a finalize that has the GPU to
// itself; 2 (8192 registers) for one that runs beside a fused launch, whose CTA
// leaves exactly that many registers of its SM free.
template <int TT, int W>
__global__ void __launch_bounds__(32 * W, 16 / W)
index_finalize_kernel(const uint2* __restrict__ buf, const int* __restrict__ cnt, const int64_t* __restrict__ q_pos,
                      int64_t n_q, int tiles_per_seq, int t_begin, int t_count, int rshift, int k_b,
                      int64_t c_cap, int32_t* __restrict__ idx, int32_t* __restrict__ count,
                      int64_t* __restrict__ fb_rows, int* __restrict__ fb_count) {
  constexpr int tt = TT;
  __shared__ __align__(16) uint32_t hist[W][512];
  __shared__ int32_t ids[W][kFCap];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = t_count * tt;  // tt: tokens per tile; 32-bit row and tile indices
  for (int rr = blockIdx.x * W + w; rr < rows; rr += gridDim.x * W) {
    const int lt = rr / tt;
    const int t = rr - lt * tt;
    const int tile = t_begin + lt;
    const int bbi = tile / tiles_per_seq;
    const int64_t bb = bbi;
    const int64_t tok = (int64_t)(tile - bbi * tiles_per_seq) * tt + t;
    if (tok >= n_q) continue;
    int64_t c = (q_pos[bb] + tok + 1) >> rshift;
    if (c > c_cap) c = c_cap;
    const int64_t grow = bb * n_q + tok;
    int32_t* const out = idx + grow * (int64_t)k_b;
    if (c <= k_b) {
      for (int j = lane; j < k_b; j += 32) out[j] = j < c ? j : -1;
      if (lane == 0) count[grow] = (int32_t)c;
      continue;
    }
    const int* const cr = cnt + lt * 4 * tt + t;
    const int n0 = cr[0], n1 = cr[tt], n2 = cr[2 * tt], n3 = cr[3 * tt];
    const int n = n0 + n1 + n2 + n3;
    const bool seg_ok = n0 <= kSeg && n1 <= kSeg && n2 <= kSeg && n3 <= kSeg;
    if (seg_ok && n >= k_b && n <= kFCap) {
      finalize_row(buf + (lt * tt + t) * 4 * kSeg, n0, n0 + n1, n0 + n1 + n2, n, k_b, hist[w], ids[w], out);
      if (lane == 0) count[grow] = k_b;
    } else if (lane == 0) {
      fb_rows[atomicAdd(fb_count, 1)] = grow;  // the exact fallback kernel takes it
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Exact fallback for rows whose threshold missed: one CTA scores the whole row
// (m16n8k16 MMAs on kbar rows read straight from memory, the n_heads indexer
// heads in the MMA columns) into its scratch row, then runs the CTA radix
// selection on it.
__global__ void __launch_bounds__(kSelThreads)
index_fallback_kernel(const __nv_bfloat16* __restrict__ qt, const __nv_bfloat16* __restrict__ kbar,
                      int64_t kbar_stride_b, const int64_t* __restrict__ q_pos, int64_t n_q, int r, int k_b,
                      int n_heads, int64_t c_cap, const int64_t* __restrict__ fb_rows, const int* __restrict__ fb_count,
                      float* __restrict__ scratch, int64_t scratch_stride, int32_t* __restrict__ idx,
                      int32_t* __restrict__ count) {
  __shared__ SelectSmem sm;
  const int n_fb = *fb_count;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t = lane & 3;
  float* s = scratch + (int64_t)blockIdx.x * scratch_stride;
  for (int f = blockIdx.x; f < n_fb; f += gridDim.x) {
    const int64_t row = fb_rows[f];
    const int64_t bb = row / n_q;
    int64_t c = (q_pos[bb] + row % n_q + 1) / r;
    if (c > c_cap) c = c_cap;
    // B fragment: columns gid < n_heads are the heads, the others zero.
    uint32_t qf[16];
    {
      const int hh = gid < n_heads ? gid : 0;
      const uint4* src = reinterpret_cast<const uint4*>(qt + (row * n_heads + hh) * kHeadDim + 32 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = gid < n_heads ? src[u] : make_uint4(0, 0, 0, 0);
        qf[4 * u] = v.x; qf[4 * u + 1] = v.y; qf[4 * u + 2] = v.z; qf[4 * u + 3] = v.w;
      }
    }
    const __nv_bfloat16* kb = kbar + bb * kbar_stride_b;
    for (int64_t b0 = 16 * warp; b0 < c; b0 += 16 * (kSelThreads / 32)) {
      const int64_t ra = b0 + gid < c ? b0 + gid : c - 1;
      const int64_t rb2 = b0 + gid + 8 < c ? b0 + gid + 8 : c - 1;
      uint32_t ka[16], kx[16];
      const uint4* pa = reinterpret_cast<const uint4*>(kb + ra * kHeadDim + 32 * t);
      const uint4* pb = reinterpret_cast<const uint4*>(kb + rb2 * kHeadDim + 32 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 x = pa[u], y = pb[u];
        ka[4 * u] = x.x; ka[4 * u + 1] = x.y; ka[4 * u + 2] = x.z; ka[4 * u + 3] = x.w;
        kx[4 * u] = y.x; kx[4 * u + 1] = y.y; kx[4 * u + 2] = y.z; kx[4 * u + 3] = y.w;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a[4] = {ka[2 * ks], kx[2 * ks], ka[2 * ks + 1], kx[2 * ks + 1]};
        const uint32_t bq[2] = {qf[2 * ks], qf[2 * ks + 1]};
        mma_bf16_16816(acc, a, bq);
      }
      // acc: (block b0+gid, heads 2t, 2t+1), (b0+gid+8, heads 2t, 2t+1); heads >=
      // n_heads are zero, so the sum over all 8 columns is the sum over the heads.
      float sa = fmaxf(acc[0], 0.f) + fmaxf(acc[1], 0.f);
      float sb = fmaxf(acc[2], 0.f) + fmaxf(acc[3], 0.f);
      sa += __shfl_xor_sync(0xffffffffu, sa, 1);
      sb += __shfl_xor_sync(0xffffffffu, sb, 1);
      sa += __shfl_xor_sync(0xffffffffu, sa, 2);
      sb += __shfl_xor_sync(0xffffffffu, sb, 2);
      if (t == 0 && b0 + gid < c) s[b0 + gid] = sa;
      if (t == 0 && b0 + gid + 8 < c) s[b0 + gid + 8] = sb;
    }
    __syncthreads();
    cta_select_row(s, c, k_b, idx + row * (int64_t)k_b, sm);
    if (threadIdx.x == 0) count[row] = k_b;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------------
// Host side

struct FusedLayout {
  int64_t tiles_per_seq, n_tiles, tiles_per_launch;
  int nbuf;                   // entry buffers: 2 when there is more than one launch
  int64_t buf_elems, cnt_elems;  // per buffer
  size_t buf_off, cnt_off, fb_rows_off, fb_count_off, scratch_off, total;
  int64_t scratch_stride;
};

// Workspace of the fused path (after the rotated queries): the entry buffers of
// one launch's tiles (48 or 24 tokens x 4 segments x kSeg entries per tile) and their
// counts, twice when the tiles take several launches (launch j fills buffer
// j % 2 while the finalize of launch j - 1 reads the other), the fallback row
// list and counter, and the fallback kernel's score rows.
inline FusedLayout fused_layout(int64_t B, int64_t n_q, int64_t n_blocks_max, int H) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const int tt = fused_tile_tokens(H);
  FusedLayout L;
  L.tiles_per_seq = (n_q + tt - 1) / tt;
  L.n_tiles = B * L.tiles_per_seq;
  L.tiles_per_launch = L.n_tiles < kTilesPerLaunch ? L.n_tiles : kTilesPerLaunch;
  L.nbuf = L.n_tiles > L.tiles_per_launch ? 2 : 1;
  L.buf_elems = L.tiles_per_launch * tt * 4 * kSeg;
  L.cnt_elems = L.tiles_per_launch * 4 * tt;
  L.buf_off = 0;
  L.cnt_off = al(L.buf_off + (size_t)L.nbuf * L.buf_elems * sizeof(uint2));
  L.fb_rows_off = al(L.cnt_off + (size_t)L.nbuf * L.cnt_elems * sizeof(int));
  L.fb_count_off = al(L.fb_rows_off + (size_t)B * n_q * sizeof(int64_t));
  L.scratch_off = al(L.fb_count_off + sizeof(int));
  L.scratch_stride = (n_blocks_max + 63) / 64 * 64;
  L.total = al(L.scratch_off + (size_t)kFbCtas * L.scratch_stride * sizeof(float));
  return L;
}

inline bool use_fused_indexer(int64_t n_q, int k_b) { return n_q >= kFMinRows && k_b <= kFMaxKb; }

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// One finalize launch over tiles [t_begin, t_begin + t_count) (tile and row
// indices of a launch fit 32 bits: at most kTilesPerLaunch tiles).  dependent:
// launched with launch_dependent() behind the next range's fused launch (the
// kernel does not wait for that launch: what it reads was written by the one
// before, which the stream order has finished).
template <int TT, int W>
static cudaError_t launch_finalize(bool dependent, const uint2* buf, const int* cnt, const int64_t* q_pos,
                                   int64_t n_q, int64_t tiles_per_seq, int64_t t_begin, int64_t t_count, int rshift,
                                   int k_b, int64_t c_cap, int32_t* idx, int32_t* count, int64_t* fb_rows,
                                   int* fb_count, cudaStream_t st) {
  const unsigned grid = (unsigned)((t_count * TT + W - 1) / W);
  if (!dependent) {
    index_finalize_kernel<TT, W><<<grid, 32 * W, 0, st>>>(buf, cnt, q_pos, n_q, (int)tiles_per_seq, (int)t_begin,
                                                          (int)t_count, rshift, k_b, c_cap, idx, count, fb_rows,
                                                          fb_count);
    return count_launch(cudaGetLastError());
  }
  // All of the SM's unified storage as shared memory, as the fused CTA beside it has set.
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(index_finalize_kernel<TT, W>), 0);
  if (e != cudaSuccess) return e;
  return count_launch(launch_dependent(index_finalize_kernel<TT, W>, dim3(grid), dim3(32 * W), 0, st, buf, cnt,
                                       q_pos, n_q, (int)tiles_per_seq, (int)t_begin, (int)t_count, rshift, k_b,
                                       c_cap, idx, count, fb_rows, fb_count));
}

cudaError_t launch_index_fused(int H, const __nv_bfloat16* qt, const __nv_bfloat16* kbar, int64_t kbar_stride_b,
                               const int64_t* q_pos, int64_t B, int64_t n_q, int64_t n_blocks_max, int r,
                               int k_b, int32_t* idx, int32_t* count, void* ws, cudaStream_t st) {
  if (H != 1 && H != 2 && H != 4 && H != 8) return cudaErrorInvalidValue;
  const FusedLayout L = fused_layout(B, n_q, n_blocks_max, H);
  const int tt = fused_tile_tokens(H);
  const int aim = pilot_aim(k_b);
  if (L.n_tiles == 0) return cudaSuccess;
  if (L.n_tiles > 0x7fffffff) return cudaErrorInvalidValue;  // the finalize indexes tiles with 32 bits
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  char* w = static_cast<char*>(ws);
  CUtensorMap tm_q, tm_k;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(B * n_q * H)};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(tt * H)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(qt), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const int64_t nb = n_blocks_max > 0 ? n_blocks_max : 1;
    int64_t sb = kbar_stride_b;
    if (B == 1 || sb < nb * kHeadDim) sb = nb * kHeadDim;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)nb, (cuuint64_t)B};
    const cuuint64_t strides[2] = {kHeadDim * 2, (cuuint64_t)sb * 2};
    const cuuint32_t box[3] = {64, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(kbar), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap tm_kp;
  {
    // The same rows viewed as [B][groups][16][128]: a box of 128 groups at one
    // phase p loads blocks 16 m + p.  Only complete groups are addressable.
    const int64_t nb = n_blocks_max > 0 ? n_blocks_max : 1;
    int64_t sb = kbar_stride_b;
    if (B == 1 || sb < nb * kHeadDim) sb = nb * kHeadDim;
    const int64_t groups = nb / kPilotStride > 0 ? nb / kPilotStride : 1;
    const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kPilotStride, (cuuint64_t)groups, (cuuint64_t)B};
    const cuuint64_t strides[3] = {kHeadDim * 2, (cuuint64_t)kPilotStride * kHeadDim * 2, (cuuint64_t)sb * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kMB, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(&tm_kp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<__nv_bfloat16*>(kbar), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const void* kern = H == 1   ? reinterpret_cast<const void*>(index_topk_fused_kernel<1>)
                       : H == 2 ? reinterpret_cast<const void*>(index_topk_fused_kernel<2>)
                       : H == 4 ? reinterpret_cast<const void*>(index_topk_fused_kernel<4>)
                                : reinterpret_cast<const void*>(index_topk_fused_kernel<8>);
    cudaError_t e = ensure_dyn_smem(kern, (int)kFusedSmemBytes);
    if (e != cudaSuccess) return e;
  }
  int* fb_count = reinterpret_cast<int*>(w + L.fb_count_off);
  int64_t* fb_rows = reinterpret_cast<int64_t*>(w + L.fb_rows_off);
  uint2* buf = reinterpret_cast<uint2*>(w + L.buf_off);
  int* cnt = reinterpret_cast<int*>(w + L.cnt_off);
  cudaError_t e = cudaMemsetAsync(fb_count, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  int rshift = 0;  // r is a power of two
  while ((1 << rshift) < r) ++rshift;
  // Launches over ranges of tiles, the last (heaviest) range first.  The
  // finalize of range j is launched after the fused launch of range j + 1,
  // dependent on it, and runs beside it (two-warp CTAs on the registers the
  // fused CTAs leave free, then on whole SMs once that launch drains); the
  // fused launch of range j + 2 waits for both.  The finalize of the last
  // range follows it alone, in four-warp CTAs.
  int64_t p_begin = 0, p_count = 0;  // range waiting for its finalize
  int p_half = 0, half = 0;
  for (int64_t t_end = L.n_tiles; t_end > 0; t_end -= L.tiles_per_launch, half ^= 1) {
    const int64_t t_begin = t_end > L.tiles_per_launch ? t_end - L.tiles_per_launch : 0;
    const int64_t t_count = t_end - t_begin;
    int64_t grid = sms < kFMaxCtas ? sms : kFMaxCtas;
    if (grid > t_count) grid = t_count;
    uint2* const hbuf = buf + half * L.buf_elems;
    int* const hcnt = cnt + half * L.cnt_elems;
#define QSA_FUSED_LAUNCH(HH)                                                                                 \
  index_topk_fused_kernel<HH><<<(unsigned)grid, kFThreads, kFusedSmemBytes, st>>>(                           \
      tm_q, tm_k, tm_kp, q_pos, n_q, L.tiles_per_seq, t_begin, t_count, rshift, k_b, aim, n_blocks_max, hbuf, hcnt)
    switch (H) {
      case 1: QSA_FUSED_LAUNCH(1); break;
      case 2: QSA_FUSED_LAUNCH(2); break;
      case 4: QSA_FUSED_LAUNCH(4); break;
      default: QSA_FUSED_LAUNCH(8); break;
    }
#undef QSA_FUSED_LAUNCH
    e = count_launch(cudaGetLastError());
    if (e != cudaSuccess) return e;
    if (p_count > 0) {
      e = tt == 48 ? launch_finalize<48, 2>(true, buf + p_half * L.buf_elems, cnt + p_half * L.cnt_elems, q_pos,
                                            n_q, L.tiles_per_seq, p_begin, p_count, rshift, k_b, n_blocks_max, idx,
                                            count, fb_rows, fb_count, st)
                   : launch_finalize<24, 2>(true, buf + p_half * L.buf_elems, cnt + p_half * L.cnt_elems, q_pos,
                                            n_q, L.tiles_per_seq, p_begin, p_count, rshift, k_b, n_blocks_max, idx,
                                            count, fb_rows, fb_count, st);
      if (e != cudaSuccess) return e;
    }
    p_begin = t_begin;
    p_count = t_count;
    p_half = half;
  }
  if (p_count > 0) {
    e = tt == 48 ? launch_finalize<48, 4>(false, buf + p_half * L.buf_elems, cnt + p_half * L.cnt_elems, q_pos, n_q,
                                          L.tiles_per_seq, p_begin, p_count, rshift, k_b, n_blocks_max, idx, count,
                                          fb_rows, fb_count, st)
                 : launch_finalize<24, 4>(false, buf + p_half * L.buf_elems, cnt + p_half * L.cnt_elems, q_pos, n_q,
                                          L.tiles_per_seq, p_begin, p_count, rshift, k_b, n_blocks_max, idx, count,
                                          fb_rows, fb_count, st);
    if (e != cudaSuccess) return e;
  }
  index_fallback_kernel<<<kFbCtas, kSelThreads, 0, st>>>(
      qt, kbar, kbar_stride_b, q_pos, n_q, r, k_b, H, n_blocks_max, fb_rows, fb_count,
      reinterpret_cast<float*>(w + L.scratch_off), L.scratch_stride, idx, count);
  return count_launch(cudaGetLastError());
}


// Rows of the last fused-indexer call on workspace `ws` (its fused part) that
// went to the exact fallback kernel.  Waits for `st`.
inline cudaError_t read_fused_fallback_rows(const void* ws, int64_t B, int64_t n_q, int64_t n_blocks_max, int H,
                                            int64_t* rows, cudaStream_t st) {
  const FusedLayout L = fused_layout(B, n_q, n_blocks_max, H);
  int n = 0;
  cudaError_t e = cudaMemcpyAsync(&n, static_cast<const char*>(ws) + L.fb_count_off, sizeof(int),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *rows = n;
  return e;
}

}  // namespace qsa
