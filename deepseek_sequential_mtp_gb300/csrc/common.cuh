// Shared helpers of the libmtp kernels: status plumbing, the per-file device
// error word, bounded waits, bf16 conversion and small warp reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mtp.h"

#define MTP_CUDA_TRY(expr)                                \
  do {                                                    \
    cudaError_t mtp_e_ = (expr);                          \
    if (mtp_e_ != cudaSuccess) return MTP_ERR_CUDA;       \
  } while (0)

#define MTP_LAUNCH_CHECK()                                \
  do {                                                    \
    if (cudaPeekAtLastError() != cudaSuccess) {           \
      (void)cudaGetLastError();                           \
      return MTP_ERR_CUDA;                                \
    }                                                     \
  } while (0)

// Each kernel file owns one device error word; mtp_check_errors ORs them.
// `take` reads and clears it (the stream has been synchronised by then).
#define MTP_DEFINE_ERROR_WORD(take_fn)                                        \
  static __device__ unsigned int g_mtp_error_word = 0;                        \
  unsigned int take_fn() {                                                    \
    unsigned int v = 0, zero = 0;                                             \
    if (cudaMemcpyFromSymbol(&v, g_mtp_error_word, sizeof(v)) != cudaSuccess) \
      return 0xFFFFFFFFu;                                                     \
    cudaMemcpyToSymbol(g_mtp_error_word, &zero, sizeof(zero));                \
    return v;                                                                 \
  }

namespace mtp {

// Host-side launch accounting and the optional event hook (api.cu).
void note_launch();
void prof_begin(int kernel_class, cudaStream_t stream);
void prof_end(int kernel_class, cudaStream_t stream);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch attributes (the dynamic shared-memory limit of a kernel) and device
// properties belong to one device, so a process that drives several GPUs
// keeps one entry per device ordinal.  Objects of static storage duration
// start zeroed; concurrent first calls may both set an attribute, which is
// harmless.
constexpr int kMaxDevices = 64;
struct PerDevice {
  std::atomic<int> v[kMaxDevices];
};
inline int current_device() {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}
// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device.
template <typename Kernel>
inline bool smem_limit(PerDevice& done, Kernel* kernel, int bytes) {
  const int dev = current_device();
  if (dev < 0) return false;
  if (dev < kMaxDevices && done.v[dev].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  if (dev < kMaxDevices) done.v[dev].store(1, std::memory_order_release);
  return true;
}
// Streaming multiprocessors of the current device (cached per device).
inline int sm_count_current() {
  static PerDevice cache;
  const int dev = current_device();
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache.v[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < kMaxDevices) cache.v[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Bounded waits count SM clock cycles (clock64 is monotonic per SM; the
// global nanosecond timer can step when it is resynchronised with the host).
// A legitimate wait lasts microseconds; the limit is ~1.5 s at 2 GHz.
constexpr long long kWaitLimitCycles = 3000000000ll;

__device__ __forceinline__ long long cycles_now() { return clock64(); }

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream is still
// running; it must call pdl_wait() before its first access to memory that
// earlier kernels write (the wait returns once they have completed and their
// writes are visible).  pdl_trigger() lets such a dependent start early; a
// kernel that never calls it releases its dependent at completion.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` as a programmatic dependent of the stream's previous kernel (the
// kernel calls pdl_wait() before reading what earlier kernels wrote).  Only for a launch
// whose stream predecessor is a kernel.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
// two bf16 in one 32-bit word, the first (lower address) in the low half
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack2_bf16(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}
__device__ __forceinline__ __nv_bfloat16 f32_to_bf16(float v) { return __float2bfloat16_rn(v); }

template <typename T> __device__ __forceinline__ float load_f32(const T* p);
template <> __device__ __forceinline__ float load_f32<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Inclusive prefix sum across the warp (lane order).
__device__ __forceinline__ double warp_inclusive_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace mtp
