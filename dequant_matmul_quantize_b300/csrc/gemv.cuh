// nf4_gemv: y[m, n] = sum_k x[m, k] * w_hat[n, k] for 1 <= M <= 16
// ("bitsandbytes tutorial", sec. 3.4 and sec. 七 myth 5: the packed weights
// are what is moved, the dequantization is extra arithmetic).
//
// Warp-per-row reference kernel: each lane takes 8 consecutive weights
// (one 32-bit word of packed codes) per 256-column step, rebuilds
// w_hat = bf16(code * s_b) exactly as the dequantizer does, and accumulates
// x * w_hat in fp32; a butterfly sums the lanes and lane 0 writes bf16.
#pragma once

#include "common.cuh"

namespace nf4q {

constexpr int kGemvSimpleThreads = 256;

template <int MT>
__global__ void __launch_bounds__(kGemvSimpleThreads)
gemv_simple_kernel(const uint32_t* __restrict__ packed, ScaleView sv,
                   const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                   int64_t N, int64_t K, int M,
                   const __grid_constant__ CodeValues C) {
  __shared__ float s_code[16 * 32];
  for (int i = threadIdx.x; i < 16 * 32; i += blockDim.x) s_code[i] = C.v[i >> 5];
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31u;
  const float* code = s_code + lane;
  const int64_t gwarp =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t units_per_row = K / 8;
  for (int64_t n = gwarp; n < N; n += nwarps) {
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    for (int64_t ku = lane; ku < units_per_row; ku += 32) {
      const int64_t unit = n * units_per_row + ku;
      const uint32_t p = ld_stream_u32(packed + unit);
      const float s = block_scale(sv, unit >> 3);
      float wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t nib = (p >> (8 * (i >> 1) + ((i & 1) ? 0 : 4))) & 0xFu;
        const float prod = __fmul_rn(code[nib * 32], s);
        wv[i] = __bfloat162float(__float2bfloat16_rn(prod));
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + m * K) + ku);
          float a = acc[m];
          a = __fmaf_rn(bf16lo_to_f32(xv.x), wv[0], a);
          a = __fmaf_rn(bf16hi_to_f32(xv.x), wv[1], a);
          a = __fmaf_rn(bf16lo_to_f32(xv.y), wv[2], a);
          a = __fmaf_rn(bf16hi_to_f32(xv.y), wv[3], a);
          a = __fmaf_rn(bf16lo_to_f32(xv.z), wv[4], a);
          a = __fmaf_rn(bf16hi_to_f32(xv.z), wv[5], a);
          a = __fmaf_rn(bf16lo_to_f32(xv.w), wv[6], a);
          a = __fmaf_rn(bf16hi_to_f32(xv.w), wv[7], a);
          acc[m] = a;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = acc[m];
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
      if (lane == 0 && m < M) {
        const __nv_bfloat16 b = __float2bfloat16_rn(a);
        y[m * N + n] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
}

}  // namespace nf4q
