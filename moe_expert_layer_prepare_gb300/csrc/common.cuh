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

// UE8M0 exponent of a 1x128 group from its amax.  The pages' recipe is
// s = max(amax, 1e-4) / 448 in fp32, then the exponent field of s plus one if
// its mantissa is not zero (the power of two rounded up), clamped to [1, 254].
// With a = max(amax, 1e-4) = (1 + m) * 2^(E - 127) and 448 = 1.75 * 2^8 that
// power of two is 2^ceil(log2 a/448) = 2^(E - 135 + [m > 0.75]); the fp32
// quotient is an exact power of two only when a / 448 is one (448 * 2^k * (1 +
// d) with 0 < d < 2^-24 is not an fp32 number), so the integer form below gives
// the same byte for every finite fp32 a without the division.  An infinite
// amax gives an infinite quotient, whose exponent field 255 clamps to 254.
__device__ __forceinline__ uint32_t ue8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(fmaxf(amax, 1.0e-4f));
  const uint32_t e = ((b >> 23) & 0xFFu) - 8u + ((b & 0x7FFFFFu) > 0x600000u ? 1u : 0u);
  return b >= 0x7F800000u ? 254u : min(max(e, 1u), 254u);
}

// 1 / 2^(e - 127) for an exponent byte in [1, 254] (exact; 2^-127 is subnormal).
__device__ __forceinline__ float ue8m0_inverse(uint32_t e) {
  return e <= 253u ? __uint_as_float((254u - e) << 23) : __uint_as_float(0x00400000u);
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

// 32-byte global store (p 32-byte aligned): one full sector per lane, half
// the store instructions of st_v4.
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
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

// Programmatic dependent launch: every kernel of the path is launched so that
// it may start while its predecessor in the stream finishes; it waits here
// (until the predecessor grid has completed and its writes are visible)
// before touching global memory, and lets its own successor start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe

// Host-side launchers shared between translation units.
namespace moe_host {

// Launch with programmatic stream serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

moe_status_t set_error(moe_status_t st, const char* fmt, ...);
int num_sms();
int resident_blocks(const void* kernel, int block);
}  // namespace moe_host
