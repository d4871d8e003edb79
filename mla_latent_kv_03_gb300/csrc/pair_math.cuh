// Arithmetic helpers of the tensor-core softmax loops: packed fp32 pairs
// and a three-input maximum, as single sm_100-family instructions.
#pragma once

#include <stdint.h>

namespace mla {

// Packed fp32 arithmetic (fma.rn.f32x2 / add.rn.f32x2): two lanes of
// round-to-nearest fp32 work per issued instruction, the same results as two
// fmaf / __fadd_rn.
__device__ __forceinline__ uint64_t f32x2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f32x2_unpack(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(f32x2_pack(a.x, a.y)), "l"(f32x2_pack(b.x, b.y)), "l"(f32x2_pack(c.x, c.y)));
  return f32x2_unpack(d);
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f32x2_pack(a.x, a.y)), "l"(f32x2_pack(b.x, b.y)));
  return f32x2_unpack(d);
}

// max(a, b, c) in one instruction (the three-input form of max.f32; like
// fmaxf, a NaN operand is ignored)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace mla
