// Key compression and query rotation for the QSA indexer.
//
// "On the Design of Qwen3.8-Next Architecture", research-hub notes, Key ideas,
// QSA compressed-indexer bullet: keys are average-pooled into blocks of r and get
// partial RoPE (64 of 128 dims) after compression.  paperglide reader, "Qwen
// Sparse Attention" step 2: the pooled key may pass through RMSNorm (optional
// here, unit weight).  Both operations are memory-bound: one warp per output row,
// 16-byte-friendly coalesced reads, fp32 arithmetic with fp64 RoPE angles, and a
// single round to bf16.
#include "common.cuh"

namespace qsa {

constexpr int kCompressWarps = 8;

// One warp per compressed block.  Pooling reads the block's r rows with
// 16-byte loads: lane l takes dims 8 (l % 16) .. + 7 of the rows t = l / 16,
// l / 16 + 2, ..., and the two half-warps add their sums.  The pooled fp32 row
// is staged in shared memory so that any even rope_dims can pair dim j with
// dim j + rope_dims/2; lane l then rotates and stores dims 4 l .. 4 l + 3
// (one 256-byte store per warp).  The angle of pair j (reduced in fp64,
// whose rate on this GPU is low) is computed once, by lane j % 32, into
// shared memory.
__global__ void __launch_bounds__(kCompressWarps * 32)
compress_keys_kernel(const __nv_bfloat16* __restrict__ k_idx, int64_t k_stride_b, int64_t B,
                     int64_t first_block, int64_t n_blocks, int r, int rmsnorm, float rms_eps,
                     RopeParams rope, __nv_bfloat16* __restrict__ kbar, int64_t kbar_stride_b) {
  __shared__ __align__(16) float pooled[kCompressWarps][kHeadDim];
  __shared__ float cs[kCompressWarps][2][kMaxRopePairs];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kCompressWarps + warp;
  if (item >= B * n_blocks) return;
  const int64_t bb = item / n_blocks;
  const int64_t blk = first_block + item % n_blocks;
  const __nv_bfloat16* src = k_idx + bb * k_stride_b + blk * r * kHeadDim;
  const int chunk = lane & 15;
  const int half = rope.half;
  for (int j = lane; j < half; j += 32) {
    float c, sn;
    rope_cos_sin(blk, rope.theta[j], &c, &sn);
    cs[warp][0][j] = c;
    cs[warp][1][j] = sn;
  }

  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int t = lane >> 4; t < r; t += 2) {
    const uint4 v = ldg_stream(src + t * kHeadDim + 8 * chunk);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc[2 * u] += bf16_lo(w[u]);
      acc[2 * u + 1] += bf16_hi(w[u]);
    }
  }
  const float inv_r = 1.0f / (float)r;  // r is a power of two: exact
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = (acc[u] + __shfl_xor_sync(0xffffffffu, acc[u], 16)) * inv_r;
  if (rmsnorm) {  // both half-warps hold the whole row: reduce over 16 lanes
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) ss += acc[u] * acc[u];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss * (1.0f / kHeadDim) + rms_eps);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] *= inv;
  }
  if (lane < 16) {
    float4* dstp = reinterpret_cast<float4*>(&pooled[warp][8 * chunk]);
    dstp[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dstp[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncwarp();

  float y[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int dim = 4 * lane + u;
    y[u] = pooled[warp][dim];
    if (dim < 2 * half) {
      const int j = dim < half ? dim : dim - half;
      const float c = cs[warp][0][j], s = cs[warp][1][j];
      const float x1 = pooled[warp][j], x2 = pooled[warp][j + half];
      y[u] = dim < half ? fmaf(x1, c, -x2 * s) : fmaf(x1, s, x2 * c);
    }
  }
  __nv_bfloat16* dst = kbar + bb * kbar_stride_b + blk * kHeadDim;
  *reinterpret_cast<uint2*>(dst + 4 * lane) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
}

// One warp per query token: the RoPE angles of position floor(i / r) are
// computed once per token and applied to all n_heads indexer heads.  The
// token's rows (n_heads x 256 bytes) are loaded up front, 16 bytes per lane
// and load, together with its position, so that the warp waits for one
// round trip to memory rather than one per head; they are staged as fp32 in
// shared memory, and lane l rotates and stores dims l + 32 u of each head.
__global__ void __launch_bounds__(kCompressWarps * 32)
rotate_queries_kernel(const __nv_bfloat16* __restrict__ q_idx, const int64_t* __restrict__ q_pos,
                      int64_t B, int64_t n_q, int r, int n_heads, RopeParams rope,
                      __nv_bfloat16* __restrict__ qt) {
  constexpr int kVecPerHead = kHeadDim / 8;                      // 16-byte vectors per head row
  constexpr int kMaxVec = kMaxIdxHeads * kVecPerHead / 32;       // per lane
  __shared__ float cs[kCompressWarps][2][kMaxRopePairs];
  __shared__ __align__(16) float rows[kCompressWarps][kMaxIdxHeads * kHeadDim];
  griddep_wait();  // launched dependent: the previous kernel may still write its inputs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kCompressWarps + warp;
  if (item >= B * n_q) return;
  const int nvec = n_heads * kVecPerHead;
  const uint4* src = reinterpret_cast<const uint4*>(q_idx + item * (n_heads * kHeadDim));
  uint4 v[kMaxVec];
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u)
    if (lane + 32 * u < nvec) v[u] = ldg_stream(src + lane + 32 * u);
  const int64_t bb = item / n_q;
  const int64_t pos = (q_pos[bb] + item % n_q) / r;
  const int half = rope.half;
  for (int j = lane; j < half; j += 32) {
    float c, s;
    rope_cos_sin(pos, rope.theta[j], &c, &s);
    cs[warp][0][j] = c;
    cs[warp][1][j] = s;
  }
  float* const row = rows[warp];
#pragma unroll
  for (int u = 0; u < kMaxVec; ++u) {
    const int e = lane + 32 * u;  // dims 8 e .. 8 e + 7 of the token's concatenated head rows
    if (e < nvec) {
      float4* d = reinterpret_cast<float4*>(row + 8 * e);
      d[0] = make_float4(bf16_lo(v[u].x), bf16_hi(v[u].x), bf16_lo(v[u].y), bf16_hi(v[u].y));
      d[1] = make_float4(bf16_lo(v[u].z), bf16_hi(v[u].z), bf16_lo(v[u].w), bf16_hi(v[u].w));
    }
  }
  __syncwarp();
  __nv_bfloat16* dst = qt + item * (n_heads * kHeadDim);
  for (int h = 0; h < n_heads; ++h) {
    const float* hrow = row + h * kHeadDim;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int dim = lane + 32 * u;
      float y = hrow[dim];
      if (dim < 2 * half) {
        const int j = dim < half ? dim : dim - half;
        const float c = cs[warp][0][j], s = cs[warp][1][j];
        const float x1 = hrow[j], x2 = hrow[j + half];
        y = dim < half ? fmaf(x1, c, -x2 * s) : fmaf(x1, s, x2 * c);
      }
      dst[h * kHeadDim + dim] = __float2bfloat16_rn(y);
    }
  }
}

cudaError_t launch_compress_keys(const __nv_bfloat16* k_idx, int64_t k_stride_b, int64_t B,
                                 int64_t first_block, int64_t n_blocks, int r, int rmsnorm,
                                 float rms_eps, const RopeParams& rope, __nv_bfloat16* kbar,
                                 int64_t kbar_stride_b, cudaStream_t st) {
  const int64_t items = B * n_blocks;
  if (items == 0) return cudaSuccess;
  const int64_t grid = (items + kCompressWarps - 1) / kCompressWarps;
  compress_keys_kernel<<<(unsigned)grid, kCompressWarps * 32, 0, st>>>(
      k_idx, k_stride_b, B, first_block, n_blocks, r, rmsnorm, rms_eps, rope, kbar, kbar_stride_b);
  return count_launch(cudaGetLastError());
}

cudaError_t launch_rotate_queries(const __nv_bfloat16* q_idx, const int64_t* q_pos, int64_t B,
                                  int64_t n_q, int r, int n_heads, const RopeParams& rope, __nv_bfloat16* qt,
                                  cudaStream_t st) {
  const int64_t items = B * n_q;
  if (items == 0) return cudaSuccess;
  const int64_t grid = (items + kCompressWarps - 1) / kCompressWarps;
  return count_launch(launch_dependent(rotate_queries_kernel, dim3((unsigned)grid), dim3(kCompressWarps * 32), 0, st,
                                      q_idx, q_pos, B, n_q, r, n_heads, rope, qt));
}

}  // namespace qsa
