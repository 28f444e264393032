// Sparse core attention over the selected micro-blocks plus the current-block
// tail.
//
// "On the Design of Qwen3.8-Next Architecture", paperglide reader, "Qwen Sparse
// Attention" steps 4-5 and Fig. 3: the selected block ids are expanded back to
// their tokens, joined with the tokens of the incomplete final block, and
// softmax attention runs over that set only ("sparse core attention").  The
// attention layout is grouped-query: Hq query heads share Hkv key/value heads.
//
// Work item = (query token, kv head, chunk of 8 query heads of that group), one
// warp each; warps are persistent and take items in an order that keeps one kv
// head's K/V hot in L2.  The per-token selection gives no reuse across tokens,
// so the kernel moves 512 B of K and V per selected token and kv head from
// L2/HBM.  Each warp streams its gathered rows through its own cp.async ring in
// shared memory (16 tokens = 8 KB of K and V per stage, 16-byte chunks
// XOR-swizzled by row so that ldmatrix reads are free of bank conflicts): the
// ring's other stages are in flight while one is consumed.  Prefill runs
// twelve warps per SM with two stages each, decode eight with three (see
// AttnShape).  The warps are bound by their instructions and dependent
// latencies per stage, so the stage is kept lean:
//   * the item's selected block ids are copied once into a 512-entry window in
//     the warp's shared memory (one coalesced load, repeated only past 512
//     blocks, ids checked there), so a stage's copies are issued after a
//     shared-memory read rather than after an L2 round trip;
//   * block and slot arithmetic uses shifts (r is a power of two);
//   * the streamed q rows, block ids and outputs are loaded and stored with
//     evict-first hints, so that L2 keeps the gathered K/V rows instead;
//   * S^T = K Q^T (m16n8k16 MMAs, 16 tokens x 8 heads, K fragments by
//     ldmatrix) runs its 8 k-steps as two accumulator chains of 4, summed;
//   * the fp32 online softmax keeps its running maximum until a score exceeds
//     it by more than 8 (log2 units); only then are the maximum reduced across
//     lanes and O and l rescaled (P stays at or below 2^8, so fp32 sums and the bf16
//     P are safe).  Its arithmetic uses packed fp32x2 adds, multiplies and
//     fmas on the lane's two heads.
// Then O^T += V^T P^T (V fragments by ldmatrix.trans, P transposed by
// movmatrix).
#include "common.cuh"

namespace qsa {

constexpr int kAGroup = 16;                                  // gathered tokens per stage
constexpr int kAStageBytes = kAGroup * 2 * kHeadDim * 2;     // K and V rows: 8 KB
constexpr int kAIds = 512;                                   // block ids per window

// Per-kernel shape: warps per CTA (one CTA per SM) and cp.async stages per
// warp; each warp's shared memory is its ring, then its id window.  Prefill
// gathers from L2 and is bound by each warp's per-stage dependencies, which
// twelve warps of two stages hide better than eight of three (measured 15.5
// against 18.9 ms at 128K); decode streams from HBM, where three stages per
// warp keep more bytes in flight (the twelve-warp shape was 14% slower there).
template <int kWarps_, int kRing_>
struct AttnShape {
  static constexpr int kWarps = kWarps_, kRing = kRing_;
  static constexpr int kRingBytes = kRing * kAStageBytes;
  static constexpr int kWarpBytes = kRingBytes + kAIds * 4;
  static constexpr int kSmemBytes = kWarps * kWarpBytes;
};
using PrefillShape = AttnShape<12, 2>;  // 216 KB
using DecodeShape = AttnShape<8, 3>;    // 208 KB
static_assert(PrefillShape::kSmemBytes <= 227 * 1024 && DecodeShape::kSmemBytes <= 227 * 1024, "shared memory");
constexpr float kLog2e = 1.4426950408889634f;

struct AttnRow {
  int64_t i;       // token position
  int64_t c;       // completed blocks visible
  int cnt;         // selected blocks
  int n_tok;       // |T_i| = cnt * r + tail
  int rs;          // log2 r (r is a power of two): slot / r and slot % r by shift and mask
  const int32_t* sel;
};

// Block ids [w0, w0 + kAIds) of the row's selection into the warp's window
// `ids` (shared memory); entries past cnt are 0.  An id outside [0, c) is
// reported and replaced by block 0 here, once per item, not per stage.
__device__ __forceinline__ void load_id_window(int32_t* ids, const AttnRow& a, int w0) {
  const int lane = threadIdx.x & 31;
  __syncwarp();  // every lane is done with the previous window
  int32_t v[kAIds / 32];
#pragma unroll
  for (int j = 0; j < kAIds / 32; ++j) {
    const int b = w0 + lane + 32 * j;
    v[j] = b < a.cnt ? __ldcs(a.sel + b) : 0;
  }
#pragma unroll
  for (int j = 0; j < kAIds / 32; ++j) {
    if (w0 + lane + 32 * j < a.cnt && (uint32_t)v[j] >= (uint64_t)a.c) {  // malformed: read block 0, report
      flag_device_error(kDevErrBlockId);
      v[j] = 0;
    }
  }
#pragma unroll
  for (int j = 0; j < kAIds / 32; ++j) ids[lane + 32 * j] = v[j];
  __syncwarp();
}

// slot_token with the selected block ids read from the window that starts at
// block w0 (every selected slot asked for has slot / r - w0 in [0, kAIds)).
__device__ __forceinline__ int64_t slot_token_window(const AttnRow& a, int r, int slot, const int32_t* ids,
                                                     int w0) {
  const int sel_tok = a.cnt << a.rs;
  if (slot < sel_tok) {
    const int64_t b = ids[(slot >> a.rs) - w0];  // checked against c when loaded
    return (b << a.rs) + (slot & (r - 1));
  }
  return (a.c << a.rs) + (slot - sel_tok);
}

__device__ __forceinline__ AttnRow make_row(int64_t i, int r, const int32_t* sel, int cnt, int k_b) {
  AttnRow a;
  a.i = i;
  a.rs = __ffs(r) - 1;
  a.c = (i + 1) >> a.rs;
  const int64_t cmax = a.c < k_b ? a.c : k_b;
  if (cnt < 0 || cnt > cmax) {  // count inconsistent with the position: clamp, report
    flag_device_error(kDevErrBlockId);
    cnt = cnt < 0 ? 0 : (int)cmax;
  }
  a.cnt = cnt;
  a.sel = sel;
  a.n_tok = (cnt << a.rs) + (int)(i + 1 - (a.c << a.rs));
  return a;
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t saddr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// Offset of 16-byte chunk `chunk` (0..15) of row `row` in a stage's K or V
// tile (rows of 256 B; chunk index XORed with row % 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

// Issue the copies of one stage: gathered slots [s0, s0 + 16) (slots past
// slot_end re-read the last valid slot; their logits are masked).  Each copy
// instruction moves two whole rows (lanes 0-15: row 2j, lanes 16-31: row 2j+1,
// 16 bytes per lane), so every request is a full, contiguous 256-byte row.
__device__ __forceinline__ void issue_stage(uint32_t kst, const AttnRow& a, int r, int s0, int slot_end,
                                            const __nv_bfloat16* __restrict__ kh,
                                            const __nv_bfloat16* __restrict__ vh, const int32_t* ids, int w0) {
  const int lane = threadIdx.x & 31;
  int slot = s0 + (lane & 15);
  if (slot >= slot_end) slot = slot_end - 1;
  const int my_tok = (int)slot_token_window(a, r, slot, ids, w0);  // token of row lane % 16 (L_cap < 2^31)
  const int chunk = lane & 15, sub = lane >> 4;
  const uint32_t vst = kst + kAGroup * 256;
#pragma unroll
  for (int j = 0; j < kAGroup / 2; ++j) {
    const int row = 2 * j + sub;
    const int tok = __shfl_sync(0xffffffffu, my_tok, row);
    cp_async16(kst + swz(row, chunk), reinterpret_cast<const char*>(kh + (int64_t)tok * kHeadDim) + chunk * 16);
    cp_async16(vst + swz(row, chunk), reinterpret_cast<const char*>(vh + (int64_t)tok * kHeadDim) + chunk * 16);
  }
}

// Attention of one token (row `a`) for 8 query heads (qh0 .. qh0+7, only the
// first n_heads valid) over gathered slots [slot_beg, slot_end), slot_beg <
// slot_end.  `ring` is the warp's kRing-stage buffer (shared-window address),
// `ids` its block-id window.
// Results per lane: o[mt][e] = unnormalised O^T (dims 16 mt + gid (+8), heads
// 2t, 2t+1), running max m2[2] (log2 units, scale folded in) and sum l[2] of
// the lane's heads 2t, 2t+1 (reduced across the warp).
template <int kRing>
__device__ __forceinline__ void attend_slots(const __nv_bfloat16* __restrict__ q_heads, int n_heads,
                                             const __nv_bfloat16* __restrict__ kh,
                                             const __nv_bfloat16* __restrict__ vh, const AttnRow& a,
                                             int r, int slot_beg, int slot_end, float scale_log2,
                                             uint32_t ring, int32_t* ids, float o[8][4], float m2[2], float l[2]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  const int ngroups = (slot_end - slot_beg + kAGroup - 1) / kAGroup;
  // The window holds blocks [w0, w0 + kAIds); a stage whose selected slots
  // reach past it moves it to the stage's first block (stages only advance,
  // so no later stage asks for a block below w0).
  const int sel_tok = a.cnt << a.rs;
  int w0 = slot_beg >> a.rs;
  load_id_window(ids, a, w0);
  auto issue = [&](int gi) {
    const int s0 = slot_beg + gi * kAGroup;
    const int last = min(s0 + kAGroup, min(slot_end, sel_tok)) - 1;
    if (last >= s0 && (last >> a.rs) >= w0 + kAIds) {
      w0 = s0 >> a.rs;
      load_id_window(ids, a, w0);
    }
    issue_stage(ring + (gi % kRing) * kAStageBytes, a, r, s0, slot_end, kh, vh, ids, w0);
  };
#pragma unroll
  for (int p = 0; p < kRing - 1; ++p) {
    if (p < ngroups) issue(p);
    cp_async_commit();
  }
  // B fragments of Q^T: lane holds head gid, dims 16 ks + 2t (+1) and + 8.
  uint32_t qf[8][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q_heads + gid * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = gid < n_heads ? __ldcs(qrow + 8 * ks + t) : 0u;
      qf[ks][1] = gid < n_heads ? __ldcs(qrow + 8 * ks + 4 + t) : 0u;
    }
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float mrun0 = -INFINITY, mrun1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  // ldmatrix lane roles: matrix mi = lane / 8, row ri = lane % 8.
  const int mi = lane >> 3, ri = lane & 7;
  const int krow = ri + 8 * (mi & 1), kchk = mi >> 1;   // K: rows 0-15, chunk 2 ks + kchk
  const int vrow = ri + 8 * (mi >> 1), vchk = mi & 1;   // V: tokens 0-15, chunk 2 mt + vchk

  for (int g = 0; g < ngroups; ++g) {
    const int gi = g + kRing - 1;
    if (gi < ngroups) issue(gi);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint32_t kst = ring + (g % kRing) * kAStageBytes;
    const uint32_t vst = kst + kAGroup * 256;
    const int s0 = slot_beg + g * kAGroup;
    const bool va_ok = s0 + gid < slot_end, vb_ok = s0 + gid + 8 < slot_end;

    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};  // k-steps 0, 2, 4, 6 | 1, 3, 5, 7
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
      uint32_t af[4], ag[4];
      ldsm_x4(kst + swz(krow, 2 * ks + kchk), af);
      ldsm_x4(kst + swz(krow, 2 * ks + 2 + kchk), ag);
      mma_bf16_16816(sc, af, qf[ks]);
      mma_bf16_16816(sd, ag, qf[ks + 1]);
    }
    {
      const float2 s01 = __fadd2_rn(make_float2(sc[0], sc[1]), make_float2(sd[0], sd[1]));
      const float2 s23 = __fadd2_rn(make_float2(sc[2], sc[3]), make_float2(sd[2], sd[3]));
      sc[0] = s01.x; sc[1] = s01.y; sc[2] = s23.x; sc[3] = s23.y;
    }
    // sc: (slot s0+gid, head 2t), (s0+gid, 2t+1), (s0+gid+8, 2t), (s0+gid+8, 2t+1)
    const float2 sl = make_float2(scale_log2, scale_log2);
    const float2 y01 = __fmul2_rn(make_float2(sc[0], sc[1]), sl);
    const float2 y23 = __fmul2_rn(make_float2(sc[2], sc[3]), sl);
    float x0 = y01.x, x1 = y01.y, x2 = y23.x, x3 = y23.y;
    if (s0 + kAGroup > slot_end) {  // the item's last stage: slots past slot_end are masked
      x0 = va_ok ? x0 : -INFINITY;
      x1 = va_ok ? x1 : -INFINITY;
      x2 = vb_ok ? x2 : -INFINITY;
      x3 = vb_ok ? x3 : -INFINITY;
    }
    // Lazy running maximum: the stage keeps mrun unless one of its scores
    // exceeds it by more than 8 (log2 units); then the maximum is reduced
    // across the head's lanes and O, l are rescaled.  Otherwise P = 2^(x - mrun)
    // <= 2^8, and O / l and mrun + log2 l are unchanged in exact arithmetic.
    float2 al = make_float2(1.f, 1.f);
    {
      const float t0 = mrun0 + 8.f, t1 = mrun1 + 8.f;
      const bool big = x0 > t0 || x2 > t0 || x1 > t1 || x3 > t1;
      if (__any_sync(0xffffffffu, big)) {
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // Slot s0 is always valid, so the new maxima are finite.
        const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
        const float2 da = __fadd2_rn(make_float2(mrun0, mrun1), make_float2(-mn0, -mn1));
        al = make_float2(exp2f(da.x), exp2f(da.y));
        mrun0 = mn0;
        mrun1 = mn1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const float2 u = __fmul2_rn(make_float2(o[mt][0], o[mt][1]), al);
          const float2 w = __fmul2_rn(make_float2(o[mt][2], o[mt][3]), al);
          o[mt][0] = u.x; o[mt][1] = u.y; o[mt][2] = w.x; o[mt][3] = w.y;
        }
      }
    }
    const float2 nmn = make_float2(-mrun0, -mrun1);
    const float2 d01 = __fadd2_rn(make_float2(x0, x1), nmn);
    const float2 d23 = __fadd2_rn(make_float2(x2, x3), nmn);
    const float p0 = exp2f(d01.x), p1 = exp2f(d01.y);
    const float p2 = exp2f(d23.x), p3 = exp2f(d23.y);
    {
      const float2 lf = __fadd2_rn(__ffma2_rn(make_float2(l0, l1), al, make_float2(p0, p1)), make_float2(p2, p3));
      l0 = lf.x;
      l1 = lf.y;
    }
    // P^T as the B operand: transpose the (slot x head) tiles.
    const uint32_t pb[2] = {movmatrix_trans(pack_bf16x2(p0, p1)), movmatrix_trans(pack_bf16x2(p2, p3))};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t av[4];
      ldsm_x4_t(vst + swz(vrow, 2 * mt + vchk), av);
      mma_bf16_16816(o[mt], av, pb);
    }
    __syncwarp();  // the stage is refilled by the next iteration's issue
  }
  cp_async_wait<0>();
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  m2[0] = mrun0; m2[1] = mrun1;
  l[0] = l0; l[1] = l1;
}

// Writes the warp's O^T fragments (scaled per head) as fp32 [8 heads][128] into
// the warp's ring (generic pointer), then __syncwarp.
__device__ __forceinline__ void stage_o(float* st, const float o[8][4], float s0, float s1) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  __syncwarp();
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    st[(2 * t) * kHeadDim + 16 * mt + gid] = o[mt][0] * s0;
    st[(2 * t + 1) * kHeadDim + 16 * mt + gid] = o[mt][1] * s1;
    st[(2 * t) * kHeadDim + 16 * mt + 8 + gid] = o[mt][2] * s0;
    st[(2 * t + 1) * kHeadDim + 16 * mt + 8 + gid] = o[mt][3] * s1;
  }
  __syncwarp();
}

// Prefill: persistent warps over (kv head, token, 8-head chunk) items, kv head
// outermost so that concurrently running warps gather from one head's K/V.
__global__ void __launch_bounds__(PrefillShape::kWarps * 32, 1)
sparse_attn_prefill_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                           const __nv_bfloat16* __restrict__ v, int64_t L_cap,
                           const int64_t* __restrict__ q_pos, const int32_t* __restrict__ idx,
                           const int32_t* __restrict__ count, int64_t B, int64_t n_q, int Hq, int Hkv,
                           int r, int k_b, float scale, __nv_bfloat16* __restrict__ out,
                           float* __restrict__ lse) {
  extern __shared__ __align__(128) uint8_t attn_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  uint8_t* const wbuf = attn_smem + warp * PrefillShape::kWarpBytes;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(wbuf));
  int32_t* const ids = reinterpret_cast<int32_t*>(wbuf + PrefillShape::kRingBytes);
  const int group = Hq / Hkv;
  const int n_hc = (group + 7) / 8;
  const int64_t per_head = B * n_q * n_hc;
  const int64_t items = per_head * Hkv;
  const int64_t nwarps = (int64_t)gridDim.x * PrefillShape::kWarps;
  for (int64_t item = (int64_t)blockIdx.x * PrefillShape::kWarps + warp; item < items; item += nwarps) {
    const int g = (int)(item / per_head);
    const int64_t rem = item % per_head;
    const int64_t row = rem / n_hc;
    const int hc = (int)(rem % n_hc);
    const int64_t bb = row / n_q;
    const int64_t i = q_pos[bb] + row % n_q;
    if (i < 0 || i >= L_cap) {  // token outside the K/V buffers: skip, report
      if (lane == 0) flag_device_error(kDevErrPosition);
      continue;
    }
    const AttnRow a = make_row(i, r, idx + row * (int64_t)k_b, count[row], k_b);
    const int qh0 = g * group + 8 * hc;
    const int n_heads = min(8, group - 8 * hc);
    const __nv_bfloat16* kh = k + (bb * Hkv + g) * L_cap * kHeadDim;
    const __nv_bfloat16* vh = v + (bb * Hkv + g) * L_cap * kHeadDim;
    float o[8][4], m2[2], l[2];
    attend_slots<PrefillShape::kRing>(q + (row * Hq + qh0) * kHeadDim, n_heads, kh, vh, a, r, 0, a.n_tok, scale * kLog2e, ring, ids, o,
                 m2, l);
    float* st = reinterpret_cast<float*>(wbuf);
    stage_o(st, o, 1.f / l[0], 1.f / l[1]);
    // Coalesced bf16 stores: lane writes 4 consecutive dims of each head.
    for (int h = 0; h < n_heads; ++h) {
      const float* srow = st + h * kHeadDim;
      const int d = 4 * lane;
      const uint2 pk = make_uint2(pack_bf16x2(srow[d], srow[d + 1]), pack_bf16x2(srow[d + 2], srow[d + 3]));
      __stcs(reinterpret_cast<uint2*>(out + ((row * Hq) + qh0 + h) * kHeadDim + d), pk);
    }
    if (lse != nullptr && gid == 0) {
      // natural-log LSE = (m2 + log2 l) * ln 2
      if (2 * t < n_heads) lse[row * Hq + qh0 + 2 * t] = (m2[0] + log2f(l[0])) * 0.69314718055994531f;
      if (2 * t + 1 < n_heads) lse[row * Hq + qh0 + 2 * t + 1] = (m2[1] + log2f(l[1])) * 0.69314718055994531f;
    }
    __syncwarp();  // the ring is reused by the next item
  }
}

// Decode: persistent warps over (query row, kv head, 8-head chunk, split)
// items; a split is `split_len` consecutive slots.  Sequence bb holds n_q new
// query rows (one for plain decode), row j at position cache_len[bb] - n_q + j,
// all reading the sequence's K/V cache.  A warp writes unnormalised O
// (fp32) with its running max and sum per head, then counts itself in the
// unit's counter; the warp that completes the count combines the unit's
// splits (log-sum-exp weights) into the bf16 output and resets the counter.
constexpr int kDecodeMinSplit = 192;  // fewest slots per split (4 x 1M, next_n = 4: 192 or 256 took
                                      // 28.7 us, 128 30.8 us, 64 41 us: every split adds a partial to combine)

// Combine of one (sequence, kv head, head chunk) by one warp.  Lane L owns
// dims 4L .. 4L + 3 of all 8 heads; every lane reads the splits' maxima and
// sums (the same 64-byte rows, broadcast) and its 8 float4 of each split, all
// loads independent, so the combine costs about one round trip to L2.
__device__ void combine_unit(const float* __restrict__ po_unit, const float* __restrict__ pml_unit, int n_split,
                             int n_heads, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  float mmax[8], L[8];
  float4 acc[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    mmax[h] = -INFINITY;
    L[h] = 0.f;
    acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll 4
  for (int sp = 0; sp < n_split; ++sp) {
    const float4* ml4 = reinterpret_cast<const float4*>(pml_unit + sp * 16);
    const float4 m0 = __ldcg(ml4), m1 = __ldcg(ml4 + 1);
    const float ms[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
    for (int h = 0; h < 8; ++h) mmax[h] = fmaxf(mmax[h], ms[h]);
  }
#pragma unroll 2
  for (int sp = 0; sp < n_split; ++sp) {
    const float4* ml4 = reinterpret_cast<const float4*>(pml_unit + sp * 16);
    const float4 m0 = __ldcg(ml4), m1 = __ldcg(ml4 + 1), l0 = __ldcg(ml4 + 2), l1 = __ldcg(ml4 + 3);
    const float ms[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    const float ls[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    float4 x[8];
#pragma unroll
    for (int h = 0; h < 8; ++h)
      x[h] = __ldcg(reinterpret_cast<const float4*>(po_unit + (sp * 8 + h) * kHeadDim) + lane);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      // An empty split stores max = -inf and never writes its partial output,
      // so whatever an earlier call left there (possibly Inf or NaN) must not
      // enter the sum, not even multiplied by a zero weight.
      if (ms[h] > -INFINITY) {
        const float w = exp2f(ms[h] - mmax[h]);
        L[h] += w * ls[h];
        acc[h].x += w * x[h].x; acc[h].y += w * x[h].y; acc[h].z += w * x[h].z; acc[h].w += w * x[h].w;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < n_heads) {
      const float inv = L[h] > 0.f ? 1.f / L[h] : 0.f;  // L = 0 only for a rejected cache length
      const uint2 pk = make_uint2(pack_bf16x2(acc[h].x * inv, acc[h].y * inv), pack_bf16x2(acc[h].z * inv, acc[h].w * inv));
      *reinterpret_cast<uint2*>(out + h * kHeadDim + 4 * lane) = pk;
      if (lse != nullptr && lane == 0) lse[h] = (mmax[h] + log2f(L[h])) * 0.69314718055994531f;
    }
  }
}

__global__ void __launch_bounds__(DecodeShape::kWarps * 32, 1)
sparse_attn_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                          const __nv_bfloat16* __restrict__ v, int64_t L_cap,
                          const int64_t* __restrict__ cache_len, const int32_t* __restrict__ idx,
                          const int32_t* __restrict__ count, int64_t B, int n_q, int Hq, int Hkv, int r,
                          int k_b, int n_split, int split_len, float scale, float* __restrict__ part_o,
                          float* __restrict__ part_ml, int* __restrict__ unit_done,
                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  extern __shared__ __align__(128) uint8_t attn_smem[];
  griddep_wait();  // the selection and the zeroed counters come from the previous kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  uint8_t* const wbuf = attn_smem + warp * DecodeShape::kWarpBytes;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(wbuf));
  int32_t* const ids = reinterpret_cast<int32_t*>(wbuf + DecodeShape::kRingBytes);
  const int group = Hq / Hkv;
  const int n_hc = (group + 7) / 8;
  const int64_t items = B * n_q * Hkv * n_hc * n_split;
  const int64_t nwarps = (int64_t)gridDim.x * DecodeShape::kWarps;
  for (int64_t item = (int64_t)blockIdx.x * DecodeShape::kWarps + warp; item < items; item += nwarps) {
    const int split = (int)(item % n_split);
    const int64_t wi = item / n_split;          // (row, g, hc)
    const int hc = (int)(wi % n_hc);
    const int g = (int)((wi / n_hc) % Hkv);
    const int64_t row = wi / (n_hc * Hkv);      // bb * n_q + j
    const int64_t bb = row / n_q;
    const int64_t i = cache_len[bb] - n_q + row % n_q;
    const int qh0 = g * group + 8 * hc;
    const int n_heads = min(8, group - 8 * hc);
    float* po = part_o + (wi * n_split + split) * (8 * kHeadDim);
    float* pml = part_ml + (wi * n_split + split) * 16;
    bool empty = false;
    AttnRow a{};
    int s_beg = 0, s_end = 0;
    if (i < 0 || i >= L_cap) {  // cache length outside [1, L_cap]: empty split, report
      if (lane == 0 && split == 0) flag_device_error(kDevErrPosition);
      empty = true;
    } else {
      a = make_row(i, r, idx + row * (int64_t)k_b, count[row], k_b);
      s_beg = split * split_len;
      s_end = min(a.n_tok, s_beg + split_len);
      empty = s_beg >= s_end;  // an empty split contributes nothing
    }
    if (empty) {
      if (lane < 8) { pml[lane] = -INFINITY; pml[8 + lane] = 0.f; }
    } else {
      const __nv_bfloat16* kh = k + (bb * Hkv + g) * L_cap * kHeadDim;
      const __nv_bfloat16* vh = v + (bb * Hkv + g) * L_cap * kHeadDim;
      float o[8][4], m2[2], l[2];
      attend_slots<DecodeShape::kRing>(q + (row * Hq + qh0) * kHeadDim, n_heads, kh, vh, a, r, s_beg, s_end, scale * kLog2e, ring, ids, o,
                   m2, l);
      float* st = reinterpret_cast<float*>(wbuf);
      stage_o(st, o, 1.f, 1.f);
      for (int h = 0; h < 8; ++h) {
        const float4 x = *reinterpret_cast<const float4*>(st + h * kHeadDim + 4 * lane);
        *reinterpret_cast<float4*>(po + h * kHeadDim + 4 * lane) = x;
      }
      if (gid == 0) {
        pml[2 * t] = m2[0]; pml[2 * t + 1] = m2[1];
        pml[8 + 2 * t] = l[0]; pml[8 + 2 * t + 1] = l[1];
      }
    }
    // Publish the partial, then count it; the last of the unit's splits combines.
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&unit_done[wi], 1) == n_split - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      combine_unit(part_o + wi * n_split * (8 * kHeadDim), part_ml + wi * n_split * 16, n_split, n_heads,
                   out + (row * Hq + qh0) * kHeadDim, lse != nullptr ? lse + row * Hq + qh0 : nullptr);
      if (lane == 0) unit_done[wi] = 0;
    }
    __syncwarp();
  }
}

// Zeroes the completion counters of a decode call (launched dependent, so it
// waits for the previous kernel, which may be the last call's attention still
// using them).
__global__ void zero_counters_kernel(int* __restrict__ p, int64_t n) {
  griddep_wait();
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) p[j] = 0;
}

// Most splits a (sequence, kv head, head chunk) can use: splits of at least
// kDecodeMinSplit slots over the longest token set, k_b r + r - 1.
int decode_max_splits(int k_b, int r) {
  const int max_tok = k_b * r + r - 1;
  return (max_tok + kDecodeMinSplit - 1) / kDecodeMinSplit;
}

// Partials (fp32 O of 8 heads, then max and sum per head) of every split, and
// one completion counter per unit.
size_t decode_workspace_bytes(int64_t B, int Hq, int Hkv, int k_b, int r) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int64_t units = B * Hkv * n_hc;
  const size_t parts = (size_t)units * decode_max_splits(k_b, r) * (8 * kHeadDim + 16) * sizeof(float);
  return (parts + 255) / 256 * 256 + (size_t)units * sizeof(int);
}

// Grid of a persistent attention kernel (<= one CTA per SM); raises the
// kernel's dynamic shared memory limit on the current device first.
static cudaError_t attn_grid(const void* kernel, int smem_bytes, int warps, int64_t items, int* grid) {
  cudaError_t e = ensure_dyn_smem(kernel, smem_bytes);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int64_t need = (items + warps - 1) / warps;
  *grid = (int)(need < sms ? need : sms);
  return cudaSuccess;
}

cudaError_t launch_sparse_attn_prefill(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                       const __nv_bfloat16* v, int64_t L_cap, const int64_t* q_pos,
                                       const int32_t* idx, const int32_t* count, int64_t B,
                                       int64_t n_q, int Hq, int Hkv, int r, int k_b, float scale,
                                       __nv_bfloat16* out, float* lse, cudaStream_t st) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int64_t items = B * n_q * Hkv * n_hc;
  if (items == 0) return cudaSuccess;
  int grid = 0;
  cudaError_t e = attn_grid(reinterpret_cast<const void*>(sparse_attn_prefill_kernel), PrefillShape::kSmemBytes,
                            PrefillShape::kWarps, items, &grid);
  if (e != cudaSuccess) return e;
  sparse_attn_prefill_kernel<<<grid, PrefillShape::kWarps * 32, PrefillShape::kSmemBytes, st>>>(q, k, v, L_cap, q_pos, idx, count, B, n_q,
                                                                    Hq, Hkv, r, k_b, scale, out, lse);
  return count_launch(cudaGetLastError());
}

cudaError_t launch_sparse_attn_decode(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                      const __nv_bfloat16* v, int64_t L_cap,
                                      const int64_t* cache_len, const int32_t* idx,
                                      const int32_t* count, int64_t B, int n_q, int Hq, int Hkv, int r,
                                      int k_b, float scale, __nv_bfloat16* out, float* lse,
                                      void* ws, cudaStream_t st) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int64_t units = B * n_q * Hkv * n_hc;
  if (units == 0) return cudaSuccess;
  const int max_split = decode_max_splits(k_b, r);
  float* part_o = reinterpret_cast<float*>(ws);
  float* part_ml = part_o + units * max_split * 8 * kHeadDim;
  const size_t parts = (size_t)units * max_split * (8 * kHeadDim + 16) * sizeof(float);
  int* unit_done = reinterpret_cast<int*>(static_cast<char*>(ws) + (parts + 255) / 256 * 256);
  const int64_t zblocks = (units + 255) / 256;
  cudaError_t e = count_launch(launch_dependent(zero_counters_kernel, dim3((unsigned)(zblocks < 1024 ? zblocks : 1024)),
                                                dim3(256), 0, st, unit_done, units));
  if (e != cudaSuccess) return e;
  // As many splits per unit as fill the resident warps once (at least one,
  // at most max_split), each a whole number of 16-slot groups.
  int grid = 0;
  e = attn_grid(reinterpret_cast<const void*>(sparse_attn_decode_kernel), DecodeShape::kSmemBytes,
                DecodeShape::kWarps, units * max_split, &grid);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  int64_t n_split = (int64_t)sms * DecodeShape::kWarps / units;
  n_split = n_split < 1 ? 1 : (n_split > max_split ? max_split : n_split);
  const int max_tok = k_b * r + r - 1;
  int split_len = (int)((max_tok + n_split - 1) / n_split);
  split_len = (split_len + kAGroup - 1) / kAGroup * kAGroup;
  n_split = (max_tok + split_len - 1) / split_len;
  e = attn_grid(reinterpret_cast<const void*>(sparse_attn_decode_kernel), DecodeShape::kSmemBytes,
                DecodeShape::kWarps, units * n_split, &grid);
  if (e != cudaSuccess) return e;
  return count_launch(launch_dependent(sparse_attn_decode_kernel, dim3((unsigned)grid),
                                      dim3(DecodeShape::kWarps * 32), (size_t)DecodeShape::kSmemBytes, st, q, k, v, L_cap, cache_len, idx, count, B, n_q, Hq, Hkv,
                                      r, k_b, (int)n_split, split_len, scale, part_o, part_ml, unit_done, out, lse));
}

}  // namespace qsa
