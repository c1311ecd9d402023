// double_quant: the fp32 absmax scales are quantized a second time
// ("bitsandbytes tutorial", sec. 3.3): offset = mean(absmax); c = absmax -
// offset; per block of 256, scale2 = max|c| / 127 and q = rint(c / scale2)
// as int8.
//
// The mean is the float32 nearest to the EXACT mean, whatever the order in
// which the GPU adds things up:
//   pass 1 (dq_sum_kernel): every CTA adds its values in fp64 and atomically
//     accumulates the fp64 sum, the largest value and the smallest non-zero
//     value (as bit patterns; non-negative floats order like integers).  The
//     last CTA to finish checks whether fp64 addition was exact for this
//     tensor (all values are multiples of the smallest one's ulp and the
//     total stays below 2^53 such ulps), which makes the sum independent of
//     the order of the additions; it then rounds the fp64 quotient to float32,
//     with the exact remainder deciding the one case where that could round
//     twice (a quotient exactly on a float32 midpoint).  Otherwise (absmax
//     values spread over more than ~29 binades) that CTA re-adds all values
//     exactly as per-exponent integer mantissa sums into a 320-bit integer
//     (sum * 2^149), divides by n_b and rounds with integer arithmetic.
//   pass 2 (dq_quant_kernel): one warp per 256-block.
#pragma once

#include "common.cuh"

namespace nf4q {


// Layout of the double-quant workspace (cleared before pass 1).
struct DqWorkspace {
  double sum;             // fp64 sum of all absmax values
  uint32_t max_bits;      // largest value, as bits
  uint32_t inv_min_bits;  // ~(smallest non-zero value, as bits)
  uint32_t ticket;        // CTAs finished
  uint32_t pad[11];
};
static_assert(sizeof(DqWorkspace) == 64, "workspace layout");

// ---------------------------------------------------------------- big ints
constexpr int kLimbs = 10;  // 320 bits: sum * 2^149 < 2^32 * 2^128 * 2^149

__device__ __forceinline__ void big_add_shifted(uint32_t (&A)[kLimbs],
                                                uint64_t v, int shift) {
  // A += v << shift  (v < 2^64, shift >= 0, no overflow past 320 bits)
  int limb = shift >> 5, bit = shift & 31;
  uint32_t parts[3];
  parts[0] = static_cast<uint32_t>(v << bit);
  parts[1] = static_cast<uint32_t>((v >> (32 - bit)) >> 0);
  if (bit == 0) parts[1] = static_cast<uint32_t>(v >> 32);
  parts[2] = bit == 0 ? 0u : static_cast<uint32_t>(v >> (64 - bit));
  uint64_t carry = 0;
  for (int i = 0; i < kLimbs - limb; ++i) {
    uint64_t add = i < 3 ? parts[i] : 0u;
    if (i >= 3 && carry == 0) break;
    uint64_t s = static_cast<uint64_t>(A[limb + i]) + add + carry;
    A[limb + i] = static_cast<uint32_t>(s);
    carry = s >> 32;
  }
}

// Float32 nearest (ties to even) to A * 2^-149 / n.
__device__ float big_round_mean(const uint32_t (&A)[kLimbs], uint32_t n) {
  uint32_t Q[kLimbs];
  uint64_t r = 0;
  for (int i = kLimbs - 1; i >= 0; --i) {
    const uint64_t cur = (r << 32) | A[i];
    Q[i] = static_cast<uint32_t>(cur / n);
    r = cur % n;
  }
  int top = -1;
  for (int i = kLimbs - 1; i >= 0; --i)
    if (Q[i]) { top = i * 32 + 31 - __clz(Q[i]); break; }
  const int p = top + 1;  // bit length of the quotient
  if (p <= 24) {          // subnormal or first binade: quantum 2^-149
    uint32_t q = Q[0];
    const uint64_t twice = 2 * r;
    if (twice > n || (twice == n && (q & 1u))) q += 1;
    return __uint_as_float(q);  // bits == q for q <= 2^24
  }
  const int sh = p - 24;  // drop `sh` low bits of Q
  auto bit_at = [&](int b) -> uint32_t { return (Q[b >> 5] >> (b & 31)) & 1u; };
  uint32_t mant = 0;
  for (int b = p - 1; b >= sh; --b) mant = (mant << 1) | bit_at(b);
  const uint32_t rb = bit_at(sh - 1);
  bool sticky = r != 0;
  for (int b = sh - 2; b >= 0 && !sticky; --b) sticky = bit_at(b) != 0;
  if (rb && (sticky || (mant & 1u))) ++mant;
  int be = p - 23;
  if (mant == (1u << 24)) { mant >>= 1; ++be; }
  return __uint_as_float((static_cast<uint32_t>(be) << 23) | (mant & 0x7FFFFFu));
}

// Float32 nearest (ties to even) to S / n for an exact fp64 sum S.
__device__ __forceinline__ float dq_mean_from_exact_sum(double gsum, uint32_t n) {
  const double dn = static_cast<double>(n);
  const double q = gsum / dn;
  float f = static_cast<float>(q);
  if (static_cast<double>(f) != q) {
    const float up = __uint_as_float(__float_as_uint(f) + 1u);
    const float dn_f = f > 0.f ? __uint_as_float(__float_as_uint(f) - 1u) : 0.f;
    const float other = static_cast<double>(f) < q ? up : dn_f;
    const double mid = (static_cast<double>(f) + static_cast<double>(other)) * 0.5;
    if (mid == q) {  // quotient exactly on a midpoint: the remainder decides
      const double rem = fma(-q, dn, gsum);
      const float lo = fminf(f, other), hi = fmaxf(f, other);
      if (rem > 0.0) f = hi;
      else if (rem < 0.0) f = lo;
      else f = (__float_as_uint(lo) & 1u) ? hi : lo;
    }
  }
  return f;
}

constexpr int kDqSumThreads = 512;
constexpr int kDqQuantThreads = 256;

// ---------------------------------------------------------------- pass 1
__global__ void __launch_bounds__(kDqSumThreads)
dq_sum_kernel(const float* __restrict__ absmax, int64_t nb,
              DqWorkspace* __restrict__ ws, float* __restrict__ offset) {
  __shared__ double s_sum[kDqSumThreads / 32];
  __shared__ uint32_t s_max[kDqSumThreads / 32], s_imin[kDqSumThreads / 32];
  __shared__ bool s_last;
  __shared__ unsigned long long s_hist[256];

  double sum = 0.0;
  uint32_t mx = 0, imn = 0;  // imn = ~min over non-zero values
  auto add = [&](float a) {
    const uint32_t bits = __float_as_uint(a) & 0x7FFFFFFFu;
    sum += static_cast<double>(__uint_as_float(bits));
    mx = max(mx, bits);
    if (bits) imn = max(imn, ~bits);
  };
  const int64_t nvec = nb / 4;  // absmax is 16-byte aligned
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += stride) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(absmax) + i);
    add(v.x); add(v.y); add(v.z); add(v.w);
  }
  if (blockIdx.x == 0 && threadIdx.x < (nb & 3)) add(__ldg(absmax + nvec * 4 + threadIdx.x));
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    imn = max(imn, __shfl_xor_sync(0xFFFFFFFFu, imn, o));
  }
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { s_sum[wid] = sum; s_max[wid] = mx; s_imin[wid] = imn; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kDqSumThreads / 32; ++k) {
      sum += s_sum[k]; mx = max(mx, s_max[k]); imn = max(imn, s_imin[k]);
    }
    atomicAdd(&ws->sum, sum);
    atomicMax(&ws->max_bits, mx);
    atomicMax(&ws->inv_min_bits, imn);
    __threadfence();
    const uint32_t t = atomicAdd(&ws->ticket, 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA: exactness check, optional exact re-sum, rounding
  const uint32_t gmax = atomicAdd(&ws->max_bits, 0u);
  const uint32_t gmin = ~atomicAdd(&ws->inv_min_bits, 0u);
  const double gsum = atomicAdd(&ws->sum, 0.0);
  const int e_hi = max(static_cast<int>(gmax >> 23), 1);
  const int e_lo = max(static_cast<int>(gmin >> 23), 1);
  const uint32_t n = static_cast<uint32_t>(nb);
  const int log2n = n <= 1 ? 0 : 32 - __clz(n - 1);
  const bool exact = gmax == 0u || (e_hi < 255 && log2n + (e_hi - e_lo) + 24 <= 53);

  if (!exact) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0ull;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < nb; i += blockDim.x) {
      const uint32_t bits = __float_as_uint(__ldg(absmax + i)) & 0x7FFFFFFFu;
      const uint32_t e = min(bits >> 23, 254u);
      const uint32_t m = e ? ((bits & 0x7FFFFFu) | 0x800000u) : bits;
      atomicAdd(&s_hist[max(e, 1u)], static_cast<unsigned long long>(m));
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (exact) {
      *offset = nb == 0 ? 0.f : dq_mean_from_exact_sum(gsum, n);
    } else {
      uint32_t A[kLimbs];
      for (int i = 0; i < kLimbs; ++i) A[i] = 0u;
      for (int e = 1; e < 255; ++e)
        if (s_hist[e]) big_add_shifted(A, s_hist[e], e - 1);
      *offset = big_round_mean(A, n);
    }
  }
}

// ---------------------------------------------------------------- pass 2
__global__ void __launch_bounds__(kDqQuantThreads)
dq_quant_kernel(const float* __restrict__ absmax, int64_t nb,
                const float* __restrict__ offset, int8_t* __restrict__ absmax_q,
                float* __restrict__ scale2) {
  const int lane = threadIdx.x & 31;
  const int64_t nd = (nb + kDqBlock - 1) / kDqBlock;
  const int64_t warp0 =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float off = __ldg(offset);
  for (int64_t d = warp0; d < nd; d += nwarps) {
    const int64_t i0 = d * kDqBlock + lane * 8;
    float a[8];
    if (i0 + 8 <= nb) {  // absmax is 16-byte aligned and i0 % 8 == 0
      const float4 v0 = __ldg(reinterpret_cast<const float4*>(absmax + i0));
      const float4 v1 = __ldg(reinterpret_cast<const float4*>(absmax + i0) + 1);
      a[0] = v0.x; a[1] = v0.y; a[2] = v0.z; a[3] = v0.w;
      a[4] = v1.x; a[5] = v1.y; a[6] = v1.z; a[7] = v1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = i0 + i < nb ? __ldg(absmax + i0 + i) : off;
    }
    float c[8];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = __fsub_rn(a[i], off);  // 0 for the padding of a partial block
      m = fmaxf(m, fabsf(c[i]));
    }
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float s2 = __fdiv_rn(m, 127.0f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int q = 0;
      if (s2 != 0.f) {
        q = __float2int_rn(__fdiv_rn(c[i], s2));
        q = max(-127, min(127, q));
      }
      const uint32_t byte = static_cast<uint32_t>(q) & 0xFFu;
      if (i < 4) lo |= byte << (8 * i); else hi |= byte << (8 * (i - 4));
    }
    if (i0 + 8 <= nb) {
      *reinterpret_cast<uint2*>(absmax_q + i0) = make_uint2(lo, hi);
    } else {
      for (int i = 0; i < 8; ++i)
        if (i0 + i < nb)
          absmax_q[i0 + i] = static_cast<int8_t>(((i < 4 ? lo : hi) >> (8 * (i & 3))) & 0xFFu);
    }
    if (lane == 0) scale2[d] = s2;
  }
}

}  // namespace nf4q
