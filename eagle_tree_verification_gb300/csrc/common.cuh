// Shared device/host helpers of the tree-verify kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "../../include/eagle.h"

#define EAGLE_HOST_CHECK(cond, code) \
  do {                               \
    if (!(cond)) return (code);      \
  } while (0)

namespace eagle {

// Record the first device-side error of a call.
__device__ __forceinline__ void fail(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Total order on fp32 values as unsigned ints: larger float -> larger key.
// -0 is folded onto +0 so that equal values compare equal.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  uint32_t b = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(b);
}

// Key for "value descending, then index ascending" selection as a max.
__device__ __forceinline__ unsigned long long desc_key(float v, uint32_t idx) {
  return ((unsigned long long)ordered_bits(v) << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return 0xffffffffu - (uint32_t)(k & 0xffffffffull);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  return from_ordered_bits((uint32_t)(k >> 32));
}

// Target probability of a logit: q = 2^(z * log2(e)/T - lse * log2(e)),
// the exponent formed by one fused multiply-add and evaluated by the SFU's
// ex2 (relative error about 2^-22; results below 2^-126 flush to zero).  The
// LM head's probability mode and the walk that reads logits both call this
// with scales from prob_scales, so their q agree bit for bit.
struct ProbScales {
  float k2;     // log2(e) / T
  float lse2;   // lse * log2(e)
};
__device__ __forceinline__ ProbScales prob_scales(float temperature, float lse) {
  ProbScales s;
  s.k2 = __fdiv_rn(1.4426950408889634f, temperature);
  s.lse2 = __fmul_rn(lse, 1.4426950408889634f);
  return s;
}
__device__ __forceinline__ float prob_from_logit(float z, ProbScales s) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(fmaf(z, s.k2, -s.lse2)));
  return y;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
// Sum over the warp of a 64-bit value (every lane gets it), exact whenever
// the sum fits 64 bits: the 22-bit pieces of the 32 values are added by the
// warp's integer reduction unit (no piece sum reaches 2^27), then recombined.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
  const uint32_t a = (uint32_t)(v & 0x3FFFFFull);
  const uint32_t b = (uint32_t)((v >> 22) & 0x3FFFFFull);
  const uint32_t c = (uint32_t)(v >> 44);
  const uint32_t sa = __reduce_add_sync(0xffffffffu, a);
  const uint32_t sb = __reduce_add_sync(0xffffffffu, b);
  const uint32_t sc = __reduce_add_sync(0xffffffffu, c);
  return (unsigned long long)sa + ((unsigned long long)sb << 22) + ((unsigned long long)sc << 44);
}

// Programmatic dependent launch.  Every kernel of the library starts with
// pdl_begin(): it waits until the previous kernel of the stream has finished
// and its writes are visible (a no-op when launched without the attribute),
// then lets the next kernel be scheduled.  Stream order is unchanged; only
// the next kernel's launch latency overlaps this kernel's run.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline eagle_status launch_status(cudaError_t e) {
  return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Device ordinals for which host code keeps per-device state (kernel
// attributes, occupancy answers, resolved symbol addresses).
constexpr int kMaxDevices = 64;

// Host-side set-up that must run once on every device a process uses
// (function attributes such as the dynamic shared-memory limit apply to the
// device that is current when they are set).  run(f) calls f() the first
// time it is reached with a given device current, and again later only if
// that call failed.  Thread-safe.
struct PerDeviceOnce {
  std::mutex mu;
  bool done[kMaxDevices] = {};
  template <typename F>
  cudaError_t run(F&& f) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
      return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    const cudaError_t e = f();
    if (e == cudaSuccess) done[dev] = true;
    return e;
  }
};

// The current device's ordinal (0 if it cannot be read or is out of range
// of kMaxDevices, in which case callers' per-device caches use slot 0).
inline int current_device_slot() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

}  // namespace eagle
