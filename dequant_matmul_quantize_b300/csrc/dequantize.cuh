// nf4_dequantize: packed 4-bit codes + (double-quantized) block scales ->
// bf16 ("bitsandbytes tutorial", sec. 3.4: weights kept in 4 bits are
// turned back into the 16-bit compute dtype before the matmul).
//
// w_hat = bf16_rn(fp32(code_value[code] * s_b)).  One thread handles units
// of 4 packed bytes = 8 elements and writes 16 bytes of bf16; 8 consecutive
// lanes share a 64-block.  The 16 code values sit in shared memory, one copy
// per lane (value j of lane l at word j*32 + l), so the data-dependent
// lookups never collide on a bank.
#pragma once

#include "common.cuh"

namespace nf4q {

constexpr int kDequantThreads = 256;

template <int U>
__global__ void __launch_bounds__(kDequantThreads)
dequantize_kernel(const uint32_t* __restrict__ packed, ScaleView sv,
                  uint4* __restrict__ out, int64_t n_units,
                  const __grid_constant__ CodeValues C) {
  __shared__ float s_code[16 * 32];
  for (int i = threadIdx.x; i < 16 * 32; i += blockDim.x) s_code[i] = C.v[i >> 5];
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31u;
  const float* code = s_code + lane;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // thread t handles units t, t + nthreads, ... in groups of U
  for (int64_t u0 = tid; u0 < n_units; u0 += nthreads * U) {
    uint32_t word[U];
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t unit = u0 + static_cast<int64_t>(u) * nthreads;
      word[u] = unit < n_units ? ld_stream_u32(packed + unit) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t unit = u0 + static_cast<int64_t>(u) * nthreads;
      s[u] = unit < n_units ? block_scale(sv, unit >> 3) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t unit = u0 + static_cast<int64_t>(u) * nthreads;
      if (unit >= n_units) continue;
      const uint32_t p = word[u];
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // element i: byte i/2, high nibble for even i
        const uint32_t nib = (p >> (8 * (i >> 1) + ((i & 1) ? 0 : 4))) & 0xFu;
        f[i] = __fmul_rn(code[nib * 32], s[u]);
      }
      uint4 o;
      o.x = pack_bf16x2(f[0], f[1]);
      o.y = pack_bf16x2(f[2], f[3]);
      o.z = pack_bf16x2(f[4], f[5]);
      o.w = pack_bf16x2(f[6], f[7]);
      st_u4(out + unit, o);
    }
  }
}

}  // namespace nf4q
