// Shared device helpers of the nf4q kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "tables.h"

namespace nf4q {

constexpr int kBlock = 64;      // elements per absmax block
constexpr int kDqBlock = 256;   // absmax values per double-quant block

// Sticky device error word (bit 0: a pipeline wait gave up).
__device__ uint32_t g_device_error;

// The 16 code values (float32, indexed by code); 8-byte aligned so that
// consecutive pairs can be read as one 64-bit operand.
struct __align__(8) CodeValues {
  float v[16];
};

// Everything a dequantizer needs to rebuild one block's scale.
struct ScaleView {
  const int8_t* absmax_q;
  const float* absmax;
  const float* scale2;
  const float* offset;
  int double_quant;
};

// s_b = fmaf(q_b, scale2[b / 256], offset), or the fp32 absmax without
// double quantization ("bitsandbytes tutorial", sec. 3.3).
__device__ __forceinline__ float block_scale(const ScaleView& sv, int64_t b) {
  if (sv.double_quant) {
    float q = static_cast<float>(__ldg(sv.absmax_q + b));
    return __fmaf_rn(q, __ldg(sv.scale2 + (b >> 8)), __ldg(sv.offset));
  }
  return __ldg(sv.absmax + b);
}

// Relaxed atomic add on a shared-memory word (a 32-bit shared address);
// returns the value before the add.
__device__ __forceinline__ uint32_t atom_add_shared(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two float32 -> packed bf16x2 (lo in the low half), each rounded to nearest
// even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two float32 -> packed fp16x2 (lo in the low half), each rounded to nearest
// even (overflow to infinity).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Compute dtypes: 0 = bf16, 1 = fp16 (nf4q_compute_dtype).
template <int DT>
__device__ __forceinline__ uint32_t pack_x2(float lo, float hi) {
  return DT == 0 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
template <int DT>
__device__ __forceinline__ uint16_t round_to_dt(float v) {
  return static_cast<uint16_t>(pack_x2<DT>(v, 0.f) & 0xFFFFu);
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t v) {
  float r;
  asm("{\n .reg .b16 h;\n mov.b32 {h, _}, %1;\n cvt.f32.f16 %0, h;\n}" : "=f"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t v) {
  float r;
  asm("{\n .reg .b16 h;\n mov.b32 {_, h}, %1;\n cvt.f32.f16 %0, h;\n}" : "=f"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) {
  return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

}  // namespace nf4q
