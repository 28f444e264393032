// Sparse core attention for prefill on the Blackwell tensor cores: the selected
// micro-blocks and the current-block tail of one query token are staged by TMA
// and contracted by tcgen05 MMAs with accumulators in TMEM.
//
// "On the Design of Qwen3.8-Next Architecture", paperglide reader, "Qwen Sparse
// Attention" steps 4-5 and Fig. 3: the selected block ids are expanded back to
// their tokens (a micro-block sparse mask), joined with the tokens of the
// incomplete final block, and softmax attention runs over that set only.  The
// attention is grouped-query: the 8 query heads of one kv head share its K/V.
//
// Unit of work = (query token, kv head): its 8 query heads against the token's
// set T_i.  A stage is 64 gathered tokens (16 slots of r = 4 tokens).
//
//   Staging.  One TMA box per slot loads a whole micro-block of K (and one of V)
//   through a 4-D view of the [B*Hkv][L][128] cache as (dim within half, half,
//   token, head): the box (64, 2, r, 1) lands as 2r rows of 128 bytes, row
//   2t + h holding half h (dims 64h .. 64h + 63) of token t, 128-byte
//   swizzled, one 1024-byte atom per 4 tokens.  A selected block is the box at
//   token b r; the tail is the box that ends at token i (its tokens before the
//   tail are masked), which never reads past the query token.
//   Scores.  S^T = Kstage . Q'^T with M = 128 stage rows and N = 16, Q' = the 8
//   heads' dims 0-63 (columns 0-7) stacked on their dims 64-127 (columns 8-15),
//   K = 64 per row: row (t, h) holds in column n + 8h the half-h product of
//   token t with head n, and the two lanes of a token add their halves.
//   PV.  O^T += Vstage^T . P'^T with Vstage read MN-major (M = 64 dims of a
//   row, K = the 128 stage rows) and N = 16: P'[n][(t, 0)] = P[t][n] and
//   P'[8 + n][(t, 1)] = P[t][n], zero elsewhere, so column n of the result is
//   head n's dims 0-63 and column 8 + n its dims 64-127.
//   Softmax.  fp32, in the log2 domain with the scale folded in.  All four
//   epilogue warps use one running maximum per head; it is raised (and the
//   partial results rescaled) only when some score of a stage exceeds it by
//   more than 2^8, decided by one barrier-reduction vote, so most stages need no
//   exchange.  P is rounded to bf16 for the MMA; the sums use the fp32 values.
//   O is kept in registers: each stage's PV lands in a fresh TMEM buffer and is
//   folded in with that stage's rescale factor.
//
// Warp roles (256 threads, two CTAs per SM).  Warps 0-2 issue the TMA loads:
// a TMA copy takes its issuing warp about a hundred cycles, so one issuing
// warp caps the gather rate, and each of the three issues a third of every
// stage's slots.  K of a stage is loaded as soon as its ring slot frees after
// that stage's scores MMA, V one stage later, as its slot frees only after
// the PV MMA.  Warp 3 issues the MMAs; warps 4-7 read TMEM (one 32-lane
// quarter each) and run the softmax.  Two CTAs of 8 warps at up to 128
// registers fit an SM (each of its four schedulers holds 16K registers).
// Every wait is bounded; on a timeout the CTA raises its abort flag, the
// roles drain without further work, in-flight copies and MMAs are waited for
// and TMEM is freed, and the device error word reports the timeout.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace qsa {

constexpr int kTcStages = 3;                         // K/V ring depth
constexpr int kTcProducers = 3;                      // TMA-issuing warps (each a third of a stage's slots)
constexpr int kTcEpiWarps = 4;
constexpr int kTcMmaWarp = kTcProducers;             // warp 3
constexpr int kTcThreads = 32 * (kTcProducers + 1 + kTcEpiWarps);  // 256
constexpr int kTcStageBytes = 128 * 128;             // 128 rows of 128 B: 64 tokens
constexpr int kTcGroup = 8;                          // query heads per kv head
constexpr uint32_t kTcTmemCols = 64;                 // S: 2 x 16 columns, O: 2 x 16 columns
constexpr float kTcRescale = 8.f;                    // log2 headroom of the running maximum
constexpr int kTcBar = 1;                            // named barrier of the epilogue warps

struct TcSmem {
  uint8_t k[kTcStages][kTcStageBytes];
  uint8_t v[kTcStages][kTcStageBytes];
  uint8_t q[2][2048];   // Q' of two units: rows 0-7 dims 0-63, rows 8-15 dims 64-127
  uint8_t p[2][4096];   // P' of two stages: 16 rows x 128 stage rows, two 64-row slabs
  float red[2][kTcEpiWarps][8];
  float lred[kTcEpiWarps][8];
  uint64_t k_full[kTcStages], v_full[kTcStages], k_empty[kTcStages], v_empty[kTcStages];
  uint64_t q_full[2], q_empty[2], s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kTcSmemBytes = sizeof(TcSmem) + 1024;  // + alignment slack

// One unit's geometry, computed identically by every role.
struct TcUnit {
  int64_t row;     // query row bb * n_q + j
  int64_t i;       // its token position
  int64_t c;       // completed blocks visible
  int head;        // bb * Hkv + g: the K/V head of the 4-D view
  int g;           // kv head
  int cnt;         // selected blocks
  int tail;        // tail tokens [c r, i]
  int n_slots;     // cnt + (tail > 0)
  int n_stages;
  bool skip;       // position outside the K/V buffers
};

__device__ __forceinline__ TcUnit tc_unit(int64_t u, int64_t rows, int64_t n_q, int Hkv, const int64_t* q_pos,
                                          const int32_t* count, int64_t L_cap, int r, int k_b, int sps, bool report) {
  TcUnit U;
  U.g = (int)(u / rows);
  U.row = u % rows;
  const int64_t bb = U.row / n_q;
  U.head = (int)(bb * Hkv + U.g);
  U.i = q_pos[bb] + U.row % n_q;
  U.skip = U.i < 0 || U.i >= L_cap;
  U.c = U.skip ? 0 : (U.i + 1) / r;
  U.tail = U.skip ? 0 : (int)(U.i + 1 - U.c * r);
  int cnt = U.skip ? 0 : count[U.row];
  const int64_t cmax = U.c < k_b ? U.c : k_b;
  if (cnt < 0 || cnt > cmax) {  // count inconsistent with the position: clamp, report
    if (report) flag_device_error(kDevErrBlockId);
    cnt = cnt < 0 ? 0 : (int)cmax;
  }
  if (U.skip && report) flag_device_error(kDevErrPosition);
  U.cnt = cnt;
  U.n_slots = cnt + (U.tail > 0 ? 1 : 0);
  U.n_stages = (U.n_slots + sps - 1) / sps;
  return U;
}

// Slots loaded in stage s: the live ones, rounded up to whole MMA K-steps of
// 16 rows (`spk` slots); the extra slot re-loads the tail box and is masked.
__device__ __forceinline__ int tc_loaded_slots(const TcUnit& U, int s, int sps, int spk) {
  int n = U.n_slots - s * sps;
  n = n < sps ? n : sps;
  n = (n + spk - 1) / spk * spk;
  return n < sps ? n : sps;
}

// Slot `slot`'s selected block id, or -1 for the tail (and any padding slot):
// a plain load, so that it can be issued a stage before its use.
__device__ __forceinline__ int tc_slot_block(const TcUnit& U, const int32_t* __restrict__ sel, int slot) {
  return slot < U.cnt ? __ldg(sel + slot) : -1;
}

// First token of a slot's box: block b's first token, or for b = -1 the box
// ending at i (the tail, and any padding slot).
__device__ __forceinline__ int tc_slot_start(const TcUnit& U, int b, int r) {
  if (b < 0) return (int)(U.i - r + 1);
  if ((int64_t)b >= U.c) {  // malformed selection: read block 0, report
    flag_device_error(kDevErrBlockId);
    b = 0;
  }
  return b * r;
}

// Bounded wait by every lane of a warp.  After a timeout (abort flag raised)
// it returns at once, so the epilogue warps run out their loops, and their
// named barriers, in step without further waiting.
__device__ __forceinline__ void warp_wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  sm100::mbar_wait(bar, parity, abort_flag, sm100::kWaitCycles, 0);
  __syncwarp();
}

// Folds the PV result of global stage g (TMEM columns 32 + 16 (g & 1) of this
// warp's lane quarter at taddr) into O: O = O * alpha[head] + PV.
__device__ __forceinline__ void tc_fold(TcSmem& S, uint32_t taddr, uint32_t g, const float (&alpha)[8], float (&O)[16],
                                        volatile int* abort_flag) {
  using namespace sm100;
  const uint32_t b2 = g & 1;
  warp_wait_all(&S.o_full[b2], (g >> 1) & 1, abort_flag);
  tc_fence_after();
  uint32_t ov[16];
  tmem_ld16(taddr + 32 + b2 * 16, ov);
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.o_empty[b2]);
#pragma unroll
  for (int c = 0; c < 16; ++c) O[c] = fmaf(O[c], alpha[c & 7], __uint_as_float(ov[c]));
}

__device__ __forceinline__ void st_global_cs_b16(__nv_bfloat16* p, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  asm volatile("st.global.cs.b16 [%0], %1;" ::"l"(p), "h"(*reinterpret_cast<const unsigned short*>(&h)) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 2)
sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, int64_t L_cap, const int64_t* __restrict__ q_pos,
                      const int32_t* __restrict__ idx, const int32_t* __restrict__ count, int64_t B, int64_t n_q,
                      int Hq, int Hkv, int r, int k_b, float scale_log2, __nv_bfloat16* __restrict__ out,
                      float* __restrict__ lse) {
  using namespace sm100;
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* const base = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  TcSmem& S = *reinterpret_cast<TcSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.abort_flag;
  const int64_t rows = B * n_q;
  const int64_t units = rows * Hkv;
  const int sps = 64 / r;                // slots per stage
  const int spk = r >= 8 ? 1 : 8 / r;    // slots per 16-row MMA K-step
  const int box = 256 * r;               // bytes per slot box

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&S.k_full[s], kTcProducers);
      mbar_init(&S.v_full[s], kTcProducers);
      mbar_init(&S.k_empty[s], 1);
      mbar_init(&S.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.q_full[b], 1);
      mbar_init(&S.q_empty[b], 1);
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_empty[b], kTcEpiWarps);
      mbar_init(&S.p_full[b], kTcEpiWarps);
      mbar_init(&S.p_empty[b], 1);
      mbar_init(&S.o_full[b], 1);
      mbar_init(&S.o_empty[b], kTcEpiWarps);
    }
    mbar_init(&S.mma_done, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(&S.tmem_base, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp < kTcProducers) {
    // ------------------------------------------------------------ TMA producers
    const uint64_t pol_stream = policy_evict_first();
    // This warp's slots of every stage: [my0, my1).
    const int my0 = warp * sps / kTcProducers, my1 = (warp + 1) * sps / kTcProducers;
    const int qs = my1 - my0;
    uint32_t gst = 0, gu = 0, v_issued = 0;
    bool ok = true;
    // V of global stage g: this warp's `mine` slots, lane l's box at token
    // `ts` of head `head` (the same boxes as that stage's K).
    int pv_mine = 0, pv_ts = 0, pv_head = 0;
    auto issue_v = [&](uint32_t g, int mine, int ts, int head) -> bool {
      const int st = (int)(g % kTcStages);
      bool w = true;
      if (lane == 0) w = mbar_wait(&S.v_empty[st], ((g / kTcStages) & 1) ^ 1, abort_flag, kWaitCycles, 64);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) return false;
      if (lane == 0) mbar_arrive_expect_tx(&S.v_full[st], (uint32_t)(mine * box));
      __syncwarp();
      if (lane < mine) tma_load_4d(S.v[st] + (my0 + lane) * box, &tm_v, &S.v_full[st], 0, 0, ts, head);
      v_issued = g + 1;
      return true;
    };
    for (int64_t u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const TcUnit U = tc_unit(u, rows, n_q, Hkv, q_pos, count, L_cap, r, k_b, sps, false);
      if (U.skip || U.n_stages == 0) continue;
      const uint32_t qb = gu & 1;
      if (warp == 0 && lane == 0) {
        ok = mbar_wait(&S.q_empty[qb], ((gu >> 1) & 1) ^ 1, abort_flag, kWaitCycles, 64);
        if (ok) {
          mbar_arrive_expect_tx(&S.q_full[qb], 2048);
          const int qrow = (int)(U.row * Hq + U.g * kTcGroup);
          tma_load_2d_hint(S.q[qb], &tm_q, &S.q_full[qb], 0, qrow, pol_stream);
          tma_load_2d_hint(S.q[qb] + 1024, &tm_q, &S.q_full[qb], 64, qrow, pol_stream);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++gu;
      const int32_t* sel = idx + U.row * (int64_t)k_b;
      // Block ids are loaded one stage ahead of their use.
      int blk = lane < qs ? tc_slot_block(U, sel, my0 + lane) : -1;
      for (int s = 0; s < U.n_stages; ++s, ++gst) {
        const int blk_next = (lane < qs && s + 1 < U.n_stages) ? tc_slot_block(U, sel, (s + 1) * sps + my0 + lane) : -1;
        // K of this stage (its slot frees as soon as the scores MMA is done) ...
        const int st = (int)(gst % kTcStages);
        if (lane == 0) ok = mbar_wait(&S.k_empty[st], ((gst / kTcStages) & 1) ^ 1, abort_flag, kWaitCycles, 64);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int n_ld = tc_loaded_slots(U, s, sps, spk);
        int mine = n_ld - my0;  // this warp's loaded slots: [my0, my0 + mine)
        mine = mine < 0 ? 0 : (mine > qs ? qs : mine);
        if (lane == 0) mbar_arrive_expect_tx(&S.k_full[st], (uint32_t)(mine * box));
        __syncwarp();
        const int ts = lane < mine ? tc_slot_start(U, blk, r) : 0;
        blk = blk_next;
        if (lane < mine) tma_load_4d(S.k[st] + (my0 + lane) * box, &tm_k, &S.k_full[st], 0, 0, ts, U.head);
        // ... then V of the previous stage, whose slot frees only after its PV.
        if (gst > 0 && !issue_v(gst - 1, pv_mine, pv_ts, pv_head)) { ok = false; break; }
        pv_mine = mine;
        pv_ts = ts;
        pv_head = U.head;
      }
    }
    if (ok && gst > 0) ok = issue_v(gst - 1, pv_mine, pv_ts, pv_head);
    if (!ok && lane == 0) {
      volatile int never = 0;  // wait (bounded) for copies still in flight
      for (uint32_t j = (gst > kTcStages ? gst - kTcStages : 0); j < gst; ++j)
        mbar_wait(&S.k_full[j % kTcStages], (j / kTcStages) & 1, &never, 100000000LL);
      for (uint32_t j = (v_issued > kTcStages ? v_issued - kTcStages : 0); j < v_issued; ++j)
        mbar_wait(&S.v_full[j % kTcStages], (j / kTcStages) & 1, &never, 100000000LL);
      if (warp == 0 && gu > 0) mbar_wait(&S.q_full[(gu - 1) & 1], ((gu - 1) >> 1) & 1, &never, 100000000LL);
    }
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16);
      constexpr uint32_t idesc_pv = idesc_bf16_f32_amn(64, 16);
      uint32_t gst = 0, gu = 0;
      bool ok = true, pend = false;
      uint32_t pend_g = 0;
      int pend_kk = 0;
      // PV of global stage g over its first nkk 16-row K-steps.
      auto issue_pv = [&](uint32_t g, int nkk) -> bool {
        const int st = (int)(g % kTcStages);
        const uint32_t b2 = g & 1, ph2 = (g >> 1) & 1;
        if (!mbar_wait(&S.v_full[st], (g / kTcStages) & 1, abort_flag, kWaitCycles, 32)) return false;
        if (!mbar_wait(&S.p_full[b2], ph2, abort_flag, kWaitCycles, 32)) return false;
        if (!mbar_wait(&S.o_empty[b2], ph2 ^ 1, abort_flag, kWaitCycles, 32)) return false;
        tc_fence_after();
        const uint32_t a0 = smem_u32(S.v[st]), b0 = smem_u32(S.p[b2]);
        const uint32_t d = tmem + 32 + b2 * 16;
        for (int kk = 0; kk < nkk; ++kk)
          umma_bf16(d, desc_mnmajor_sw128(a0 + (uint32_t)kk * 2048),
                    desc_kmajor_sw128(b0 + (uint32_t)(kk >> 2) * 2048 + (uint32_t)(kk & 3) * 32), idesc_pv,
                    kk > 0 ? 1u : 0u);
        umma_commit(&S.v_empty[st]);
        umma_commit(&S.p_empty[b2]);
        umma_commit(&S.o_full[b2]);
        return true;
      };
      for (int64_t u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const TcUnit U = tc_unit(u, rows, n_q, Hkv, q_pos, count, L_cap, r, k_b, sps, false);
        if (U.skip || U.n_stages == 0) continue;
        const uint32_t qb = gu & 1;
        if (!mbar_wait(&S.q_full[qb], (gu >> 1) & 1, abort_flag, kWaitCycles, 32)) { ok = false; break; }
        ++gu;
        const uint32_t qa = smem_u32(S.q[qb]);
        for (int s = 0; s < U.n_stages; ++s, ++gst) {
          const int st = (int)(gst % kTcStages);
          const uint32_t b2 = gst & 1;
          if (!mbar_wait(&S.k_full[st], (gst / kTcStages) & 1, abort_flag, kWaitCycles, 32)) { ok = false; break; }
          if (!mbar_wait(&S.s_empty[b2], ((gst >> 1) & 1) ^ 1, abort_flag, kWaitCycles, 32)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ka = smem_u32(S.k[st]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + b2 * 16, desc_kmajor_sw128(ka + kk * 32), desc_kmajor_sw128(qa + kk * 32), idesc_s,
                      kk > 0 ? 1u : 0u);
          umma_commit(&S.k_empty[st]);
          umma_commit(&S.s_full[b2]);
          if (s == U.n_stages - 1) umma_commit(&S.q_empty[qb]);
          // The previous stage's PV goes after this stage's scores, so that the
          // epilogue can work on one stage while the next one's scores run.
          if (pend && !issue_pv(pend_g, pend_kk)) { ok = false; break; }
          pend = true;
          pend_g = gst;
          pend_kk = tc_loaded_slots(U, s, sps, spk) * r / 8;
        }
      }
      if (ok && pend) issue_pv(pend_g, pend_kk);
      umma_commit(&S.mma_done);  // every MMA completes before TMEM is released
      volatile int never = 0;
      mbar_wait(&S.mma_done, 0, &never, 100000000LL);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int ew = warp - kTcMmaWarp - 1;  // 0..3
    const int q4 = warp & 3;           // TMEM lane quarter
    const int m = 32 * q4 + lane;      // stage row = PV K index
    const int h = lane & 1;            // half of the token this lane's row holds
    const int slot_in = m / (2 * r);   // slot of the row within a stage
    const int tok_in = (m % (2 * r)) >> 1;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    // P' byte offsets of this lane's stores: head 4h + k goes to row 4h + k
    // (value in the even column of pair m & ~1) and to row 8 + 4h + k (odd
    // column), which is the same position one 1024-byte atom further.
    uint32_t poff[4];
    {
      const int j0 = m & ~1, slab = j0 >> 6, ch = (j0 & 63) >> 3;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = 4 * h + k;
        poff[k] = (uint32_t)(slab * 2048 + n * 128 + ((ch ^ n) << 4) + (j0 & 7) * 2);
      }
    }
    uint32_t gst = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
      const TcUnit U = tc_unit(u, rows, n_q, Hkv, q_pos, count, L_cap, r, k_b, sps, ew == 0 && lane == 0);
      if (U.skip) continue;
      const int qh0 = U.g * kTcGroup;
      __nv_bfloat16* const orow = out + (U.row * Hq + qh0) * (int64_t)kHeadDim;
      if (U.n_stages == 0) {  // no token at all (a count of 0 where blocks exist): zeros, lse -inf
        for (int e = 32 * ew + lane; e < kTcGroup * kHeadDim; e += 32 * kTcEpiWarps) orow[e] = __float2bfloat16_rn(0.f);
        if (lse != nullptr && ew == 0 && lane < kTcGroup) lse[U.row * Hq + qh0 + lane] = -INFINITY;
        continue;
      }
      float m_ref[8], l[4], O[16], alpha_prev[8];
#pragma unroll
      for (int n = 0; n < 8; ++n) { m_ref[n] = -INFINITY; alpha_prev[n] = 1.f; }
#pragma unroll
      for (int k = 0; k < 4; ++k) l[k] = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) O[c] = 0.f;

      for (int s = 0; s < U.n_stages; ++s, ++gst) {
        const uint32_t b2 = gst & 1, ph = (gst >> 1) & 1;
        warp_wait_all(&S.s_full[b2], ph, abort_flag);
        tc_fence_after();
        uint32_t v[16];
        tmem_ld16(tmem + lane_off + b2 * 16, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_empty[b2]);
        // Scores of this row's token for heads 4h .. 4h + 3: own half plus the
        // partner lane's half.
        float x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float send = __uint_as_float(h ? v[8 + k] : v[4 + k]);
          const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
          const float own = __uint_as_float(h ? v[12 + k] : v[k]);
          x[k] = own + recv;
        }
        const int slot = s * sps + slot_in;
        const bool valid = slot < U.cnt || (slot == U.cnt && U.tail > 0 && tok_in >= r - U.tail);
        bool need = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[k] = valid ? x[k] * scale_log2 : -INFINITY;
          need |= x[k] > (h ? m_ref[4 + k] : m_ref[k]) + kTcRescale;
        }
        float alpha[8];
#pragma unroll
        for (int n = 0; n < 8; ++n) alpha[n] = 1.f;
        if (named_bar_or(need, kTcBar, 32 * kTcEpiWarps)) {
          // Raise the running maxima to this stage's maxima (over all warps).
          float mx[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mx[k] = x[k];
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], o));
          }
          float* const rw = S.red[gst & 1][ew];
          if (lane < 2) {
#pragma unroll
            for (int k = 0; k < 4; ++k) rw[4 * lane + k] = mx[k];
          }
          named_bar_sync(kTcBar, 32 * kTcEpiWarps);
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            float sm = S.red[gst & 1][0][n];
#pragma unroll
            for (int w = 1; w < kTcEpiWarps; ++w) sm = fmaxf(sm, S.red[gst & 1][w][n]);
            const float mn = fmaxf(m_ref[n], sm);
            alpha[n] = exp2f(m_ref[n] - mn);
            m_ref[n] = mn;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) l[k] *= (h ? alpha[4 + k] : alpha[k]);
        }
        float p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          p[k] = exp2f(x[k] - (h ? m_ref[4 + k] : m_ref[k]));
          l[k] += p[k];
        }
        warp_wait_all(&S.p_empty[b2], ph ^ 1, abort_flag);
        uint8_t* const pb = S.p[b2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          *reinterpret_cast<uint32_t*>(pb + poff[k]) = pack_bf16x2(p[k], 0.f);
          *reinterpret_cast<uint32_t*>(pb + poff[k] + 1024) = pack_bf16x2(0.f, p[k]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_full[b2]);
        if (s > 0) tc_fold(S, tmem + lane_off, gst - 1, alpha_prev, O, abort_flag);
#pragma unroll
        for (int n = 0; n < 8; ++n) alpha_prev[n] = alpha[n];
      }
      tc_fold(S, tmem + lane_off, gst - 1, alpha_prev, O, abort_flag);

      // Softmax denominators: lanes of equal parity hold the same 4 heads.
      float L4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        L4[k] = l[k];
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) L4[k] += __shfl_xor_sync(0xffffffffu, L4[k], o);
      }
      if (lane < 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) S.lred[ew][4 * lane + k] = L4[k];
      }
      named_bar_sync(kTcBar, 32 * kTcEpiWarps);
      float Ltot[8];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        Ltot[n] = 0.f;
#pragma unroll
        for (int w = 0; w < kTcEpiWarps; ++w) Ltot[n] += S.lred[w][n];
      }
      // Lane e < 16 of quarter q4 holds dims 16 q4 + e (columns 0-7) and
      // 64 + 16 q4 + e (columns 8-15) of the 8 heads.
      if (lane < 16) {
        const int d0 = 16 * q4 + lane;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_global_cs_b16(orow + (c & 7) * kHeadDim + d0 + 64 * (c >> 3), O[c] / Ltot[c & 7]);
      }
      if (lse != nullptr && ew == 0 && lane == 0) {
#pragma unroll
        for (int n = 0; n < 8; ++n) lse[U.row * Hq + qh0 + n] = (m_ref[n] + log2f(Ltot[n])) * 0.69314718055994531f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// The tensor-core path serves 8 query heads per kv head and micro-blocks of
// 4, 8 or 16 tokens (a block's K or V rows then fill whole 1024-byte atoms).
inline bool tc_attention_supported(int Hq, int Hkv, int r) {
  return Hkv > 0 && Hq == kTcGroup * Hkv && (r == 4 || r == 8 || r == 16);
}

cudaError_t launch_sparse_attn_tc(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                                  int64_t L_cap, const int64_t* q_pos, const int32_t* idx, const int32_t* count,
                                  int64_t B, int64_t n_q, int Hq, int Hkv, int r, int k_b, float scale,
                                  __nv_bfloat16* out, float* lse, cudaStream_t st) {
  const int64_t units = B * n_q * Hkv;
  if (units == 0) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tm_q, tm_k, tm_v;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(B * n_q * Hq)};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTcGroup};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // (dim within half, half, token, head) view of [B * Hkv][L_cap][128].
    const cuuint64_t dims[4] = {64, 2, (cuuint64_t)L_cap, (cuuint64_t)(B * Hkv)};
    const cuuint64_t strides[3] = {128, kHeadDim * 2, (cuuint64_t)L_cap * kHeadDim * 2};
    const cuuint32_t box[4] = {64, 2, (cuuint32_t)r, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<__nv_bfloat16*>(k), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<__nv_bfloat16*>(v), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(sparse_attn_tc_kernel), (int)kTcSmemBytes);
  if (e != cudaSuccess) return e;
  // Two CTAs per SM: registers (8 warps x 128) and shared memory (2 x 113 KB of
  // 228 KB) both allow it.  The kernel is persistent with no dependence between
  // CTAs, so the result does not depend on how many are resident at once.
  int sms = 0;
  e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sms * 2;
  if (grid > units) grid = units;
  sparse_attn_tc_kernel<<<(unsigned)grid, kTcThreads, kTcSmemBytes, st>>>(
      tm_q, tm_k, tm_v, L_cap, q_pos, idx, count, B, n_q, Hq, Hkv, r, k_b, scale * 1.4426950408889634f, out, lse);
  return count_launch(cudaGetLastError());
}

}  // namespace qsa
