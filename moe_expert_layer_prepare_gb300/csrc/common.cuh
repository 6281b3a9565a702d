// Shared device helpers of the CUDA path (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_prep.h"

#ifndef __CUDACC__
#error "compile with nvcc"
#endif

namespace moe {

constexpr int kGroup = 128;  // 1x128 activation groups, 128x128 weight blocks

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Round-to-nearest-even fp32 -> bf16 bit pattern (NaN kept quiet).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two fp32 -> two e4m3 codes, round to nearest even, saturating to +-448.
// Returns lo | hi << 8.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b16 h; cvt.rn.satfinite.e4m3x2.f32 h, %2, %1; cvt.u32.u16 %0, h; }"
      : "=r"(r)
      : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// UE8M0 group scale of one 1x128 group from its amax: exponent byte and the
// reciprocal of the power-of-two scale (exact).
__device__ __forceinline__ uint32_t ue8m0_exponent(float amax) {
  float s = __fdiv_rn(fmaxf(amax, 1.0e-4f), 448.0f);
  uint32_t b = __float_as_uint(s);
  uint32_t e = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
  return min(max(e, 1u), 254u);
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe

// Host-side launchers shared between translation units.
namespace moe_host {
moe_status_t set_error(moe_status_t st, const char* fmt, ...);
int num_sms();
}  // namespace moe_host
