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
// warp each.  Per token the 8 heads of a kv group read the same gathered keys,
// so the warp computes S^T = K_T Q^T with m16n8k16 MMAs (16 gathered tokens x 8
// heads per tile) and O^T += V_T^T P^T (16 dims x 8 heads per tile), with an
// fp32 online softmax in between.  The per-token selection gives no reuse across
// tokens, so gathered rows go straight from L2/HBM into MMA fragments: every lane
// reads 64 contiguous bytes of each K or V row it needs (head dims visited in a
// permuted order that is applied to Q and undone for O), and movmatrix
// transposes the P and V fragments into operand layout.  There is no shared
// memory staging on the gather path.
#include "common.cuh"

namespace qsa {

constexpr int kAttnWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnRow {
  int64_t i;       // token position
  int64_t c;       // completed blocks visible
  int cnt;         // selected blocks
  int n_tok;       // |T_i| = cnt * r + tail
  const int32_t* sel;
};

__device__ __forceinline__ int64_t slot_token(const AttnRow& a, int r, int slot) {
  const int sel_tok = a.cnt * r;
  if (slot < sel_tok) {
    int64_t b = __ldg(a.sel + slot / r);
    if ((uint64_t)b >= (uint64_t)a.c) {  // malformed selection: read block 0, report
      flag_device_error(kDevErrBlockId);
      b = 0;
    }
    return b * r + (slot % r);
  }
  return a.c * r + (slot - sel_tok);
}

__device__ __forceinline__ void load_row64(uint32_t dst[16], const __nv_bfloat16* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 v = ldg16(q + u);
    dst[4 * u] = v.x; dst[4 * u + 1] = v.y; dst[4 * u + 2] = v.z; dst[4 * u + 3] = v.w;
  }
}

// Attention of one token (row `a`) for 8 query heads (qh0 .. qh0+7, only the
// first n_heads valid) over gathered slots [slot_beg, slot_end).
// Results per lane: o[mt][e] = unnormalised O^T (dims of m-tile mt, heads 2t,
// 2t+1), running max m2[2] (log2 units, scale folded in) and sum l[2] of the
// lane's heads 2t, 2t+1 (already reduced across the warp).
__device__ __forceinline__ void attend_slots(const __nv_bfloat16* __restrict__ q_heads, int n_heads,
                                             const __nv_bfloat16* __restrict__ kh,
                                             const __nv_bfloat16* __restrict__ vh, const AttnRow& a,
                                             int r, int slot_beg, int slot_end, float scale_log2,
                                             float o[8][4], float m2[2], float l[2]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  uint32_t qf[16];
  if (gid < n_heads) {
    load_row64(qf, q_heads + gid * kHeadDim + 32 * t);
  } else {
#pragma unroll
    for (int u = 0; u < 16; ++u) qf[u] = 0u;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float mrun0 = -INFINITY, mrun1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int s0 = slot_beg; s0 < slot_end; s0 += 16) {
    const int sa = s0 + gid, sb = s0 + gid + 8;
    const bool va_ok = sa < slot_end, vb_ok = sb < slot_end;
    const int64_t ta = slot_token(a, r, va_ok ? sa : s0);
    const int64_t tb = slot_token(a, r, vb_ok ? sb : s0);
    uint32_t ka[16], kb[16], xa[16], xb[16];
    load_row64(ka, kh + ta * kHeadDim + 32 * t);
    load_row64(kb, kh + tb * kHeadDim + 32 * t);
    load_row64(xa, vh + ta * kHeadDim + 32 * t);
    load_row64(xb, vh + tb * kHeadDim + 32 * t);

    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t af[4] = {ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1]};
      const uint32_t bf[2] = {qf[2 * ks], qf[2 * ks + 1]};
      mma_bf16_16816(sc, af, bf);
    }
    // sc: (slot sa, head 2t), (sa, 2t+1), (sb, 2t), (sb, 2t+1)
    float x0 = va_ok ? sc[0] * scale_log2 : -INFINITY;
    float x1 = va_ok ? sc[1] * scale_log2 : -INFINITY;
    float x2 = vb_ok ? sc[2] * scale_log2 : -INFINITY;
    float x3 = vb_ok ? sc[3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // Slot s0 is always valid, so the new maxima are finite.
    const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
    const float al0 = exp2f(mrun0 - mn0), al1 = exp2f(mrun1 - mn1);
    mrun0 = mn0;
    mrun1 = mn1;
    const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
    const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
    l0 = l0 * al0 + p0 + p2;
    l1 = l1 * al1 + p1 + p3;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= al0; o[mt][2] *= al0;
      o[mt][1] *= al1; o[mt][3] *= al1;
    }
    // P^T as the B operand: transpose the (slot x head) tiles.
    const uint32_t pb[2] = {movmatrix_trans(pack_bf16x2(p0, p1)), movmatrix_trans(pack_bf16x2(p2, p3))};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t af[4] = {movmatrix_trans(xa[2 * mt]), movmatrix_trans(xa[2 * mt + 1]),
                              movmatrix_trans(xb[2 * mt]), movmatrix_trans(xb[2 * mt + 1])};
      mma_bf16_16816(o[mt], af, pb);
    }
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  m2[0] = mrun0; m2[1] = mrun1;
  l[0] = l0; l[1] = l1;
}

// Physical dim of logical dim 16*mt + 8*half + gid in the O^T fragment.
__device__ __forceinline__ int o_phys_dim(int mt, int half, int gid) {
  return 32 * (gid >> 1) + 4 * mt + 2 * half + (gid & 1);
}

__device__ __forceinline__ AttnRow make_row(int64_t i, int r, const int32_t* sel, int cnt, int k_b) {
  AttnRow a;
  a.i = i;
  a.c = (i + 1) / r;
  const int64_t cmax = a.c < k_b ? a.c : k_b;
  if (cnt < 0 || cnt > cmax) {  // count inconsistent with the position: clamp, report
    flag_device_error(kDevErrBlockId);
    cnt = cnt < 0 ? 0 : (int)cmax;
  }
  a.cnt = cnt;
  a.sel = sel;
  a.n_tok = cnt * r + (int)(i + 1 - a.c * r);
  return a;
}

// Prefill: one warp per (token, kv head, 8-head chunk).  Item order puts the kv
// head outermost so that concurrently running warps gather from one head's K/V.
__global__ void __launch_bounds__(kAttnWarps * 32)
sparse_attn_prefill_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                           const __nv_bfloat16* __restrict__ v, int64_t L_cap,
                           const int64_t* __restrict__ q_pos, const int32_t* __restrict__ idx,
                           const int32_t* __restrict__ count, int64_t B, int64_t n_q, int Hq, int Hkv,
                           int r, int k_b, float scale, __nv_bfloat16* __restrict__ out,
                           float* __restrict__ lse) {
  __shared__ float stage[kAttnWarps][8][kHeadDim + 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  const int group = Hq / Hkv;
  const int n_hc = (group + 7) / 8;
  const int64_t item = (int64_t)blockIdx.x * kAttnWarps + warp;
  const int64_t per_head = B * n_q * n_hc;
  if (item >= per_head * Hkv) return;
  const int g = (int)(item / per_head);
  const int64_t rem = item % per_head;
  const int64_t row = rem / n_hc;
  const int hc = (int)(rem % n_hc);
  const int64_t bb = row / n_q;
  const int64_t i = q_pos[bb] + row % n_q;
  if (i < 0 || i >= L_cap) {  // token outside the K/V buffers: skip, report
    if (lane == 0) flag_device_error(kDevErrPosition);
    return;
  }
  const AttnRow a = make_row(i, r, idx + row * (int64_t)k_b, count[row], k_b);
  const int qh0 = g * group + 8 * hc;
  const int n_heads = min(8, group - 8 * hc);
  const __nv_bfloat16* kh = k + (bb * Hkv + g) * L_cap * kHeadDim;
  const __nv_bfloat16* vh = v + (bb * Hkv + g) * L_cap * kHeadDim;

  float o[8][4], m2[2], l[2];
  attend_slots(q + (row * Hq + qh0) * kHeadDim, n_heads, kh, vh, a, r, 0, a.n_tok,
               scale * kLog2e, o, m2, l);
  const float inv0 = 1.f / l[0], inv1 = 1.f / l[1];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d = o_phys_dim(mt, half, gid);
      stage[warp][2 * t][d] = o[mt][2 * half] * inv0;
      stage[warp][2 * t + 1][d] = o[mt][2 * half + 1] * inv1;
    }
  }
  __syncwarp();
  // Coalesced bf16 stores: lane writes 4 consecutive dims of each head.
  for (int h = 0; h < n_heads; ++h) {
    const float* srow = stage[warp][h];
    const int d = 4 * lane;
    const uint2 pk = make_uint2(pack_bf16x2(srow[d], srow[d + 1]), pack_bf16x2(srow[d + 2], srow[d + 3]));
    *reinterpret_cast<uint2*>(out + ((row * Hq) + qh0 + h) * kHeadDim + d) = pk;
  }
  if (lse != nullptr && gid == 0) {
    // natural-log LSE = (m2 + log2 l) * ln 2
    if (2 * t < n_heads) lse[row * Hq + qh0 + 2 * t] = (m2[0] + log2f(l[0])) * 0.69314718055994531f;
    if (2 * t + 1 < n_heads) lse[row * Hq + qh0 + 2 * t + 1] = (m2[1] + log2f(l[1])) * 0.69314718055994531f;
  }
}

// Decode partials: one warp per (sequence, kv head, 8-head chunk, split of
// kDecodeSplit slots).  Writes unnormalised O (fp32) with its max and sum.
constexpr int kDecodeSplit = 64;

__global__ void __launch_bounds__(kAttnWarps * 32)
sparse_attn_decode_partial_kernel(const __nv_bfloat16* __restrict__ q,
                                  const __nv_bfloat16* __restrict__ k,
                                  const __nv_bfloat16* __restrict__ v, int64_t L_cap,
                                  const int64_t* __restrict__ cache_len,
                                  const int32_t* __restrict__ idx, const int32_t* __restrict__ count,
                                  int64_t B, int Hq, int Hkv, int r, int k_b, int n_split,
                                  float scale, float* __restrict__ part_o, float* __restrict__ part_ml) {
  __shared__ float stage[kAttnWarps][8][kHeadDim + 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  const int group = Hq / Hkv;
  const int n_hc = (group + 7) / 8;
  const int64_t item = (int64_t)blockIdx.x * kAttnWarps + warp;
  if (item >= B * Hkv * n_hc * n_split) return;
  const int split = (int)(item % n_split);
  const int64_t wi = item / n_split;          // (bb, g, hc)
  const int hc = (int)(wi % n_hc);
  const int g = (int)((wi / n_hc) % Hkv);
  const int64_t bb = wi / (n_hc * Hkv);
  const int64_t i = cache_len[bb] - 1;
  float* po = part_o + (wi * n_split + split) * (8 * kHeadDim);
  float* pml = part_ml + (wi * n_split + split) * 16;
  if (i < 0 || i >= L_cap) {  // cache length outside [1, L_cap]: empty split, report
    if (lane == 0 && split == 0) flag_device_error(kDevErrPosition);
    if (lane < 8) { pml[lane] = -INFINITY; pml[8 + lane] = 0.f; }
    return;
  }
  const AttnRow a = make_row(i, r, idx + bb * (int64_t)k_b, count[bb], k_b);
  const int qh0 = g * group + 8 * hc;
  const int n_heads = min(8, group - 8 * hc);
  const int s_beg = split * kDecodeSplit;
  const int s_end = min(a.n_tok, s_beg + kDecodeSplit);
  if (s_beg >= s_end) {
    // Empty split: contributes nothing.
    if (lane < 8) { pml[lane] = -INFINITY; pml[8 + lane] = 0.f; }
    return;
  }
  const __nv_bfloat16* kh = k + (bb * Hkv + g) * L_cap * kHeadDim;
  const __nv_bfloat16* vh = v + (bb * Hkv + g) * L_cap * kHeadDim;
  float o[8][4], m2[2], l[2];
  attend_slots(q + (bb * Hq + qh0) * kHeadDim, n_heads, kh, vh, a, r, s_beg, s_end,
               scale * kLog2e, o, m2, l);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d = o_phys_dim(mt, half, gid);
      stage[warp][2 * t][d] = o[mt][2 * half];
      stage[warp][2 * t + 1][d] = o[mt][2 * half + 1];
    }
  }
  __syncwarp();
  for (int h = 0; h < 8; ++h) {
    const float4 x = *reinterpret_cast<const float4*>(&stage[warp][h][4 * lane]);
    *reinterpret_cast<float4*>(po + h * kHeadDim + 4 * lane) = x;
  }
  if (gid == 0) {
    pml[2 * t] = m2[0]; pml[2 * t + 1] = m2[1];
    pml[8 + 2 * t] = l[0]; pml[8 + 2 * t + 1] = l[1];
  }
}

// Combine the splits of one (sequence, kv head, head chunk): 8 heads x 128 dims.
__global__ void __launch_bounds__(256)
sparse_attn_decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                  int64_t B, int Hq, int Hkv, int n_split,
                                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int group = Hq / Hkv;
  const int n_hc = (group + 7) / 8;
  const int64_t wi = blockIdx.x;
  const int hc = (int)(wi % n_hc);
  const int g = (int)((wi / n_hc) % Hkv);
  const int64_t bb = wi / (n_hc * Hkv);
  const int qh0 = g * group + 8 * hc;
  const int n_heads = min(8, group - 8 * hc);
  const int h = threadIdx.x >> 5;  // 8 warps: one head each
  const int lane = threadIdx.x & 31;
  if (h >= n_heads) return;
  const float* ml = part_ml + wi * n_split * 16;
  float mmax = -INFINITY;
  for (int s = 0; s < n_split; ++s) mmax = fmaxf(mmax, ml[s * 16 + h]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < n_split; ++s) {
    const float ms = ml[s * 16 + h];
    if (!(ms > -INFINITY)) continue;
    const float w = exp2f(ms - mmax);
    L += w * ml[s * 16 + 8 + h];
    const float4 x = *reinterpret_cast<const float4*>(part_o + ((wi * n_split + s) * 8 + h) * kHeadDim + 4 * lane);
    acc.x += w * x.x; acc.y += w * x.y; acc.z += w * x.z; acc.w += w * x.w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;  // L = 0 only for a rejected cache length
  const uint2 pk = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  *reinterpret_cast<uint2*>(out + (bb * Hq + qh0 + h) * kHeadDim + 4 * lane) = pk;
  if (lse != nullptr && lane == 0) lse[bb * Hq + qh0 + h] = (mmax + log2f(L)) * 0.69314718055994531f;
}

int decode_num_splits(int k_b, int r) {
  const int max_tok = k_b * r + r - 1;
  return (max_tok + kDecodeSplit - 1) / kDecodeSplit;
}

size_t decode_workspace_bytes(int64_t B, int Hq, int Hkv, int k_b, int r) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int64_t units = B * Hkv * n_hc * (int64_t)decode_num_splits(k_b, r);
  return (size_t)units * (8 * kHeadDim + 16) * sizeof(float);
}

cudaError_t launch_sparse_attn_prefill(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                       const __nv_bfloat16* v, int64_t L_cap, const int64_t* q_pos,
                                       const int32_t* idx, const int32_t* count, int64_t B,
                                       int64_t n_q, int Hq, int Hkv, int r, int k_b, float scale,
                                       __nv_bfloat16* out, float* lse, cudaStream_t st) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int64_t items = B * n_q * Hkv * n_hc;
  if (items == 0) return cudaSuccess;
  const int64_t grid = (items + kAttnWarps - 1) / kAttnWarps;
  sparse_attn_prefill_kernel<<<(unsigned)grid, kAttnWarps * 32, 0, st>>>(
      q, k, v, L_cap, q_pos, idx, count, B, n_q, Hq, Hkv, r, k_b, scale, out, lse);
  return count_launch(cudaGetLastError());
}

cudaError_t launch_sparse_attn_decode(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                      const __nv_bfloat16* v, int64_t L_cap,
                                      const int64_t* cache_len, const int32_t* idx,
                                      const int32_t* count, int64_t B, int Hq, int Hkv, int r,
                                      int k_b, float scale, __nv_bfloat16* out, float* lse,
                                      void* ws, cudaStream_t st) {
  const int n_hc = (Hq / Hkv + 7) / 8;
  const int n_split = decode_num_splits(k_b, r);
  const int64_t units = B * Hkv * n_hc;
  if (units == 0) return cudaSuccess;
  float* part_o = reinterpret_cast<float*>(ws);
  float* part_ml = part_o + units * n_split * 8 * kHeadDim;
  const int64_t items = units * n_split;
  const int64_t grid = (items + kAttnWarps - 1) / kAttnWarps;
  sparse_attn_decode_partial_kernel<<<(unsigned)grid, kAttnWarps * 32, 0, st>>>(
      q, k, v, L_cap, cache_len, idx, count, B, Hq, Hkv, r, k_b, n_split, scale, part_o, part_ml);
  cudaError_t e = count_launch(cudaGetLastError());
  if (e != cudaSuccess) return e;
  sparse_attn_decode_combine_kernel<<<(unsigned)units, 256, 0, st>>>(part_o, part_ml, B, Hq, Hkv,
                                                                     n_split, out, lse);
  return count_launch(cudaGetLastError());
}

}  // namespace qsa
