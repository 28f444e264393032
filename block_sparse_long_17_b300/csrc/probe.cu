// Measurement helper: the L2 gather bandwidth that bounds sparse attention.
//
// Sparse core attention reads, per selected token, one 256-byte K row and one
// V row at data-dependent positions; with one kv head's K/V resident in L2 its
// speed is set by how fast the SMs can gather random 256-byte rows from L2.
// This kernel measures exactly that on a caller buffer: every half-warp reads
// pseudo-randomly chosen 256-byte rows (16 lanes x 16 bytes), four independent
// rows per step so that the rate is not limited by one load's latency (more in
// flight, or 1 KiB segments instead of rows, measured no faster).
#include "common.cuh"

namespace qsa {

__global__ void __launch_bounds__(512)
probe_gather_rows_kernel(const uint4* __restrict__ p, uint64_t nrows, int iters, uint32_t* __restrict__ sink) {
  uint32_t acc = 0;
  const int lane = threadIdx.x & 31;
  uint32_t seed = (uint32_t)((blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) / 16) * 2654435761u + 12345u;
  for (int it = 0; it < iters; it += 4) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      seed = seed * 1664525u + 1013904223u;
      const uint64_t row = (seed >> 4) % nrows;
      asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                   : "l"(p + row * 16 + (lane & 15)));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  if (acc == 0x9e3779b9u) sink[0] = acc;  // keeps the loads alive
}

}  // namespace qsa

extern "C" qsa_status qsa_probe_l2_gather(void* buf, size_t bytes, float* gbs, qsa_stream_t stream) {
  using namespace qsa;
  if (buf == nullptr || gbs == nullptr || bytes < (1u << 20) || (reinterpret_cast<uintptr_t>(buf) & 255) != 0)
    return QSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return from_cuda(e);
  // The last 256 bytes hold the sink word; rows cover the rest.
  const uint64_t nrows = (bytes - 256) / 256;
  uint32_t* sink = reinterpret_cast<uint32_t*>(static_cast<char*>(buf) + nrows * 256);
  const int grid = sms * 4, block = 512, iters = 256;
  cudaEvent_t a, b;
  if ((e = cudaEventCreate(&a)) != cudaSuccess) return from_cuda(e);
  if ((e = cudaEventCreate(&b)) != cudaSuccess) { cudaEventDestroy(a); return from_cuda(e); }
  probe_gather_rows_kernel<<<grid, block, 0, st>>>(static_cast<const uint4*>(buf), nrows, iters, sink);  // warm L2
  cudaEventRecord(a, st);
  probe_gather_rows_kernel<<<grid, block, 0, st>>>(static_cast<const uint4*>(buf), nrows, iters, sink);
  cudaEventRecord(b, st);
  e = cudaEventSynchronize(b);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (e != cudaSuccess) return from_cuda(e);
  const double moved = (double)grid * block / 16 * iters * 256;
  *gbs = (float)(moved / (ms * 1e-3) / 1e9);
  return QSA_OK;
}
