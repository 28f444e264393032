// Decode attention for callers that cannot allocate device memory.
//
// qsa_sparse_attn_decode needs a caller-provided workspace for its per-split
// partial results.  Some callers have no way to provide one: code running
// inside a framework or plugin that owns every device allocation, code paths
// that must not touch the allocator (no cudaMalloc or pool call allowed), or
// small C hosts without an allocator of their own.  For them this file holds a
// second entry point that keeps the partials in a fixed array of static device
// memory instead.  The paper has no counterpart of this; it is a packaging
// choice of this library.
//
// The array is a file-scope __device__ variable, so every device that loads
// the library holds kNoAllocScratchBytes of it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it only
// names a stand-in object), so the entry point looks up the real address once
// per device with cudaGetSymbolAddress, with that device current, and hands it
// to the kernels.
#include <mutex>

#include "common.cuh"

namespace qsa {

// QSA_NOALLOC_SCRATCH_BYTES (32 MiB): enough for the partials of 64 sequences x
// 2 kv heads at K = 2048, r = 4 (room for 11 splits of at least 192 tokens,
// 4160 B per split and head chunk, plus a completion counter per head chunk:
// 6 MB).
constexpr size_t kNoAllocScratchBytes = QSA_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on device `dev`, which must be the
// current device.  Only a successful lookup is kept: after a failed one (say,
// inside a stream capture, or with an error pending) the next call tries again.
cudaError_t noalloc_scratch_ptr(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

// The scratch address is per device, so the stream and the query tensor must
// both belong to the current device.
bool on_current_device(int dev, const void* q, cudaStream_t st) {
  int sdev = -1;
  if (cudaStreamGetDevice(st, &sdev) != cudaSuccess || sdev != dev) {
    cudaGetLastError();  // a failed query leaves no sticky error behind
    return false;
  }
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_sparse_attn_decode_noalloc(const qsa_config* cfg, const void* q,
                                                     const void* k_cache, const void* v_cache,
                                                     int64_t L_cap, const int64_t* cache_len,
                                                     const int32_t* idx, const int32_t* count,
                                                     int64_t B, int32_t Hq, int32_t Hkv, float scale,
                                                     void* out, float* lse, qsa_stream_t stream) {
  using namespace qsa;
  const size_t need = qsa_sparse_attn_decode_workspace(cfg, B, Hq, Hkv);
  if (B <= 0 || need == 0) {
    // No work, or invalid arguments: the regular entry point reports the status
    // that applies (it returns before touching the missing workspace).
    return qsa_sparse_attn_decode(cfg, q, k_cache, v_cache, L_cap, cache_len, idx, count, B, Hq,
                                  Hkv, scale, out, lse, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) return QSA_ERR_WORKSPACE;  // beyond the fixed scratch
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (q == nullptr || !on_current_device(dev, q, reinterpret_cast<cudaStream_t>(stream))) return QSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  e = noalloc_scratch_ptr(dev, &scratch);
  if (e != cudaSuccess) return from_cuda(e);
  return qsa_sparse_attn_decode(cfg, q, k_cache, v_cache, L_cap, cache_len, idx, count, B, Hq, Hkv,
                                scale, out, lse, scratch, kNoAllocScratchBytes, stream);
}
