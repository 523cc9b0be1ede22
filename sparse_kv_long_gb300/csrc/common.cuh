// common.cuh -- shared device helpers of libsparsekv (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/sparsekv.h"

#define SKV_EXPORT extern "C" __attribute__((visibility("default")))

namespace skv {

constexpr float kLog2e = 1.4426950408889634f;

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Host-side launch check: maps a failed launch to SKV_ECUDA.
inline int launch_status() {
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free launch error for the caller
    return SKV_ECUDA;
  }
  return SKV_OK;
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Host-side set-up that belongs to a device (a kernel's shared-memory limit,
// an occupancy figure) is done once per device and cached here: `slot` is a
// call site's own zero-initialised table holding value + 1 (0: not yet
// computed).  `compute` returns the value (>= 0), or -1 on failure, which is
// not cached.  Safe to call from several host threads: two of them may both
// compute the value the first time, which the set-up calls used here allow.
constexpr int kMaxDevices = 64;
template <typename F>
inline int once_per_device(std::atomic<int> (&slot)[kMaxDevices], F&& compute) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return compute();
  }
  const int v = slot[dev].load(std::memory_order_acquire);
  if (v > 0) return v - 1;
  const int r = compute();
  if (r >= 0) slot[dev].store(r + 1, std::memory_order_release);
  return r;
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device and call site; SKV_OK or SKV_ECUDA.
template <typename K>
inline int smem_limit_once(std::atomic<int> (&slot)[kMaxDevices], K kernel, size_t bytes) {
  const int r = once_per_device(slot, [&]() -> int {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
        cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    return 0;
  });
  return r < 0 ? SKV_ECUDA : SKV_OK;
}

// Raises `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes` (the limit only grows; per device and call site, under a
// lock so that a concurrent call never lowers it).  SKV_OK or SKV_ECUDA.
template <typename K>
inline int smem_limit_at_least(std::atomic<int> (&slot)[kMaxDevices], std::mutex& mu, K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return SKV_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  if (static_cast<size_t>(slot[dev].load(std::memory_order_acquire)) >= bytes) return SKV_OK;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<size_t>(slot[dev].load(std::memory_order_relaxed)) >= bytes) return SKV_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
      cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  slot[dev].store(static_cast<int>(bytes), std::memory_order_release);
  return SKV_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Programmatic dependent launch: a kernel launched with the programmatic
// stream serialization attribute may start while the previous kernel in the
// stream runs; it must call grid_dependency_wait() before touching anything
// that kernel writes.  The previous kernel lets it start early with
// allow_dependent_launch().
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t* st, unsigned bits) {
  if (st) atomicOr(reinterpret_cast<unsigned*>(st), bits);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Round-half-even then clamp; NaN and -inf go to lo, +inf to hi.
__device__ __forceinline__ int rint_clamp(float x, int lo, int hi) {
  if (!(x > static_cast<float>(lo))) return lo;
  if (!(x < static_cast<float>(hi))) return hi;
  return __float2int_rn(x);
}

// Order key of an int32 score: unsigned order == signed order.
__device__ __forceinline__ uint32_t order_key_i32(int32_t s) {
  return static_cast<uint32_t>(s) ^ 0x80000000u;
}

// Order key of an fp32 score; -0 taken as +0.
__device__ __forceinline__ uint32_t order_key_f32(float s) {
  uint32_t u = __float_as_uint(s);
  if ((u & 0x7fffffffu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Block-wide exclusive prefix sum of one int per thread (blockDim.x <= 1024,
// multiple of 32).  `scratch` holds >= 33 ints.  Returns the exclusive sum and
// writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) scratch[lane] = w;  // inclusive warp totals
    if (lane == nw - 1) scratch[32] = w;
  }
  __syncthreads();
  int base = warp ? scratch[warp - 1] : 0;
  int res = base + x - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

}  // namespace skv
