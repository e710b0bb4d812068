// Device-side helpers shared by the kernels: error reporting, fast exp2 and
// 16-bit element conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace mla {

// Error codes stored in the device error word (the first writer wins).
__device__ __forceinline__ void report_error(int *err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// 2^x with the SFU instruction (flushes denormals; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2 with the SFU instruction.
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T> struct Elem;
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ float bits_to_f(uint16_t x) {
    return __half2float(__ushort_as_half(x));
  }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float bits_to_f(uint16_t x) {
    return __bfloat162float(__ushort_as_bfloat16(x));
  }
};

// Round a float to the element type and back (softmax weights are rounded to
// the input dtype before the value product, as the TileLang split kernel's
// fp32 -> fp16 cast of acc_s does).
template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return Elem<T>::to_f(Elem<T>::from_f(x));
}

constexpr float kLn2 = 0.69314718055994530942f;

}  // namespace mla
