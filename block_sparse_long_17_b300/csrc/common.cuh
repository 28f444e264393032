// Shared device helpers of the QSA library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <map>
#include <utility>

#include "../../include/qsa.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (B300) only"
#endif

namespace qsa {

constexpr int kHeadDim = 128;
constexpr int kMaxIdxHeads = 8;  // indexer query heads: 1, 2, 4 or 8
constexpr int kMaxRopePairs = 64;  // rope_dims <= head_dim = 128

// RoPE frequencies computed on the host in fp64: theta_j = base^(-2j/rope_dims).
struct RopeParams {
  double theta[kMaxRopePairs];
  int half;  // rope_dims / 2
};

// Library-wide device error word (the library is one translation unit).
// 0 = no error; otherwise one of the codes below, first one wins.
__device__ unsigned int g_device_error = 0;

// Device error codes.
constexpr unsigned int kDevErrPosition = 1;  // a row position beyond the stated bound
constexpr unsigned int kDevErrBlockId = 2;   // a selected block id outside [0, c_i)
constexpr unsigned int kDevErrTimeout = 3;   // a bounded wait gave up

// Host-side count of kernels launched by the library (see qsa_launch_count).
inline unsigned long long& launch_counter() {
  static unsigned long long n = 0;
  return n;
}
inline cudaError_t count_launch(cudaError_t e) {
  if (e == cudaSuccess) __atomic_add_fetch(&launch_counter(), 1ull, __ATOMIC_RELAXED);
  return e;
}

// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device.  The limit set is remembered per (kernel, device), and a
// call that needs more raises it again (a kernel whose shared memory depends
// on its arguments); the attribute belongs to each device's copy of the
// kernel, so a process that drives several GPUs sets it on each.
inline cudaError_t ensure_dyn_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> set_to;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto it = set_to.find({kernel, dev});
  if (it != set_to.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // All of the unified L1/shared storage as shared memory, so that the
  // occupancy the kernel was sized for (for some kernels two CTAs per SM) is
  // available.
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess) set_to[{kernel, dev}] = bytes;
  return e;
}

// SM count of the current device.
inline cudaError_t current_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

// Programmatic dependent launch: a kernel launched with launch_dependent() may
// start while the previous kernel on the stream finishes; it calls
// griddep_wait() before it reads anything that kernel wrote (a no-op when the
// previous work on the stream was not a kernel launched this way).  This hides
// the launch gap between the short kernels of a decode step.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream, if it was launched with
// launch_dependent(), start now and run beside this one (once every CTA of this
// grid has called it or exited).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void flag_device_error(unsigned int code) {
  atomicCAS(&g_device_error, 0u, code);
}

// fp32 pair -> packed bf16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// cos/sin of pos * theta with the product and the reduction to [-pi, pi] in
// fp64, so large positions (up to 2^20 blocks) keep full fp32 accuracy.
__device__ __forceinline__ void rope_cos_sin(long long pos, double theta, float* c, float* s) {
  const double two_pi = 6.283185307179586476925286766559;
  double a = (double)pos * theta;
  double k = rint(a * (1.0 / two_pi));
  double red = fma(-k, two_pi, a);
  sincosf((float)red, s, c);
}

// 16-byte global load that bypasses L1 allocation (streamed data).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte global load through L1/L2 (gathered K/V rows).
__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// D = A * B + D, bf16 inputs, fp32 accumulate, m16n8k16 (warp-wide).
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], const uint32_t b[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Transpose of an 8x8 b16 matrix held one 32-bit pair per lane
// (lane l holds row l/4, cols 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

}  // namespace qsa
