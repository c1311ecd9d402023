// nf4_quantize: per-64-element fp32 absmax, nearest-code search and
// two-codes-per-byte packing ("bitsandbytes tutorial", sec. 2.3 absmax
// blocks, sec. 3.2 NF4 levels; FP4 per "bitsandbytes introduction",
// sec. 一 item 7).
//
// Work unit: 8 consecutive elements -> one 32-bit word of packed codes.  A
// 64-block is 8 consecutive units, held by 8 consecutive lanes, so its
// absmax is a 3-step butterfly.  Each warp pass covers U*256 elements.
//
// Code search.  The exact rule is on wn = fp32(w / absmax) (IEEE division):
// code = #{ j : wn > T_j } over the round-down midpoints T_j (FP4: on |wn|,
// plus the sign).  The kernel does not divide per element.  It forms
// q = fp32(w * r) with r an approximate reciprocal of absmax (relative error
// at most 2^-22), which is within 2^-21 of wn, and looks q up
// in 259-bin tables (bin = nearest integer of q*128 + 129): every bin is
// narrower than the gap between decision points (FP4's are mirrored onto the
// signed value), so at most one point T is in reach and
// code = lo(bin) + (q > T) * dl(bin).  When q lies within 2^-19 of that T the
// two could disagree, so the unit is recomputed with the exact division and
// a plain count over all T_j; so are blocks whose absmax is zero, below
// 2^-126 or above 2^126 (1/absmax not a normal number) or not finite.  The result is therefore
// exactly the rule; the fast path only saves work.  The tables are
// replicated once per lane in shared memory (entry e of lane l at word
// e*32 + l), so the data-dependent lookups of a warp never collide on a
// bank, and the per-element work is spread over the FMA pipe (bin, address,
// packing), the load pipe (table reads) and the integer pipe (compare bit,
// near test).
#pragma once

#include "common.cuh"

namespace nf4q {

constexpr int kQuantThreads = 512;
constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kNearEps = 1.9073486328125e-06f;  // 2^-19
constexpr float kTinyScale = 1.17549435e-38f;     // 2^-126
constexpr float kHugeScale = 8.50705917e37f;      // 2^126
constexpr int kLutWords = kLutEntries * 32;       // one table, replicated per lane

struct QuantParams {
  float lut_t[kLutEntries];     // decision point within reach of each bin
  int32_t lut_lo[kLutEntries];  // code below it
  int32_t lut_dl[kLutEntries];  // change of code across it (FP4 only)
  float thr[15];                // exact-path decision points
};

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Fast code of one element: bin lookup (2 or 3 shared loads) and a compare.
// `lane_tab` is this lane's column of the tables minus the magic offset of
// the bin computation, so that the address is one multiply-add.  The code is
// added into `word` at nibble shift `sh` with multiply-adds.
template <int CODE>
__device__ __forceinline__ void code_fast(float q, uint32_t lane_tab, bool& near, uint32_t& word,
                                          int sh) {
  const float y = __fmaf_rn(q, 128.0f, 129.0f + kMagic);
  const uint32_t a = __float_as_uint(y) * 128u + lane_tab;
  const float t = lds_f32(a);
  const int lo = lds_s32(a + kLutWords * 4);
  const float d = __fsub_rn(t, q);
  near |= fabsf(d) <= kNearEps;
  const int bit = static_cast<int>(__float_as_uint(d) >> 31);  // q > t
  const int dl = CODE == 0 ? 1 : lds_s32(a + 2 * kLutWords * 4);
  const int c = bit * dl + lo;
  word += static_cast<uint32_t>(c) * (1u << sh);
}

template <int CODE>
__device__ __forceinline__ uint32_t code_exact(float w, float a, const QuantParams& P) {
  const float q = a == 0.f ? 0.f : __fdiv_rn(w, a);
  const float v = CODE == 0 ? q : fabsf(q);
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < (CODE == 0 ? 15 : 7); ++j) c += v > P.thr[j] ? 1u : 0u;
  if (CODE == 1) c |= (q < 0.f && c != 0u) ? 8u : 0u;
  return c;
}

// Nibble position of element i (0..7) of a unit inside its 32-bit word:
// element 2j -> bits 7..4 of byte j, element 2j+1 -> bits 3..0.
__device__ __forceinline__ constexpr int nib_shift(int i) {
  return 8 * (i >> 1) + ((i & 1) ? 0 : 4);
}

template <int CODE>
__device__ __noinline__ uint32_t encode_unit_exact(float w0, float w1, float w2,
                                                   float w3, float w4, float w5,
                                                   float w6, float w7, float a,
                                                   const QuantParams& P) {
  const float w[8] = {w0, w1, w2, w3, w4, w5, w6, w7};
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) word |= code_exact<CODE>(w[i], a, P) << nib_shift(i);
  return word;
}

template <bool BF16IN>
__device__ __forceinline__ void load_unit(const void* base, int64_t unit,
                                          float (&v)[8]) {
  if (BF16IN) {
    const uint4 r = ld_stream_u4(static_cast<const uint16_t*>(base) + unit * 8);
    v[0] = bf16lo_to_f32(r.x); v[1] = bf16hi_to_f32(r.x);
    v[2] = bf16lo_to_f32(r.y); v[3] = bf16hi_to_f32(r.y);
    v[4] = bf16lo_to_f32(r.z); v[5] = bf16hi_to_f32(r.z);
    v[6] = bf16lo_to_f32(r.w); v[7] = bf16hi_to_f32(r.w);
  } else {
    const float* p = static_cast<const float*>(base) + unit * 8;
    const uint4 r0 = ld_stream_u4(p);
    const uint4 r1 = ld_stream_u4(p + 4);
    v[0] = __uint_as_float(r0.x); v[1] = __uint_as_float(r0.y);
    v[2] = __uint_as_float(r0.z); v[3] = __uint_as_float(r0.w);
    v[4] = __uint_as_float(r1.x); v[5] = __uint_as_float(r1.y);
    v[6] = __uint_as_float(r1.z); v[7] = __uint_as_float(r1.w);
  }
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;  // NaN if either is NaN, so a non-finite block is always seen
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int CODE, bool BF16IN, int U>
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const void* __restrict__ w, uint32_t* __restrict__ packed,
                float* __restrict__ absmax, int64_t n_units,
                const __grid_constant__ QuantParams P) {
  extern __shared__ uint32_t s_lut[];  // [tables][kLutEntries][32]
  for (int i = threadIdx.x; i < kLutWords; i += blockDim.x) {
    const int e = i >> 5;
    s_lut[i] = __float_as_uint(P.lut_t[e]);
    s_lut[kLutWords + i] = static_cast<uint32_t>(P.lut_lo[e]);
    if (CODE == 1) s_lut[2 * kLutWords + i] = static_cast<uint32_t>(P.lut_dl[e]);
  }
  __syncthreads();

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t lane_tab = static_cast<uint32_t>(__cvta_generic_to_shared(s_lut)) + lane * 4u -
                            kMagicBits * 128u;
  const int64_t gwarp =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t base = gwarp * (32 * U); base < n_units;
       base += nwarps * (32 * U)) {
    float v[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t unit = base + u * 32 + lane;
      if (unit < n_units) {
        load_unit<BF16IN>(w, unit, v[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
      }
    }
    float amax[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float m = fabsf(v[u][0]);
#pragma unroll
      for (int i = 1; i < 8; ++i) m = max_nan(m, fabsf(v[u][i]));
      m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
      amax[u] = m;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t unit = base + u * 32 + lane;
      const float a = amax[u];
      // 2^-126 <= a <= 2^126: the reciprocal is a normal number (the
      // approximate one flushes subnormal results), |w * rcp(a)| <= 1 + 2^-21
      // and every bin index is inside the table; anything else (zero, tiny,
      // huge or non-finite absmax) takes the exact path
      const bool ok = a >= kTinyScale && a <= kHugeScale;
      bool near = false;
      uint32_t word = 0;
      if (ok) {
        // Approximate reciprocal (relative error <= 2^-22): q stays within
        // 2^-21 of the exact quotient, inside the 2^-19 exact-fallback window.
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          code_fast<CODE>(__fmul_rn(v[u][i], r), lane_tab, near, word, nib_shift(i));
      }
      if (near || !ok)
        word = encode_unit_exact<CODE>(v[u][0], v[u][1], v[u][2], v[u][3],
                                       v[u][4], v[u][5], v[u][6], v[u][7], a, P);
      if (unit < n_units) {
        packed[unit] = word;
        if ((lane & 7u) == 0u) absmax[unit >> 3] = a;
      }
    }
  }
}

inline size_t quantize_smem_bytes(int code) {
  return static_cast<size_t>(code == 0 ? 2 : 3) * kLutWords * 4;
}

}  // namespace nf4q
