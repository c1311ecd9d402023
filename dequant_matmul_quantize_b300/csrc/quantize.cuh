// nf4_quantize: per-64-element fp32 absmax, nearest-code search and
// two-codes-per-byte packing ("bitsandbytes tutorial", sec. 2.3 absmax
// blocks, sec. 3.2 NF4 levels; FP4 per "bitsandbytes introduction",
// sec. 一 item 7).
//
// Work unit: 16 consecutive elements -> two 32-bit words of packed codes.  A
// 64-block is 4 consecutive units, held by 4 consecutive lanes, so its
// absmax is a 2-step butterfly.
//
// Code search.  The exact rule is on wn = fp32(w / absmax) (IEEE division):
// code = #{ j : wn > T_j } over the round-down midpoints T_j (FP4: on |wn|,
// plus the sign).  The kernel does not divide per element.  With r an
// approximate reciprocal of absmax (relative error at most 2^-22), the exact
// product v r is within 2^-21 of wn.  One FMA on v r gives the bin of a
// 259-entry table (bin = nearest integer of 128 v r + 129): every bin is
// narrower than the gap between decision points (FP4's are mirrored onto
// the signed value), so at most one point T is in reach, and
// code = lo(bin) + [wn > T] * dl(bin) (dl = 1 for NF4).  A second FMA forms
// e = (v r - T) 2^19 from the table's -T 2^19; if |e| <= 1 (v r within about
// 2^-19 of T) the two sides of T could disagree and that element's compare
// is redone on the exact quotient (IEEE division) at the same T - frequent
// for bf16 FP4 input, whose quotients often land exactly on 1/8; blocks
// whose absmax is zero, below 2^-100 (2^19 / absmax would overflow) or above
// 2^126 (1/absmax not a normal number) or not finite take the exact rule
// (division and a plain count over all T_j) for every element.  Otherwise
// sat(e) is the compare bit exactly, and lo + bit (one add on the table's
// float 2^23 + lo) is the code in the low mantissa bits.  The result is therefore exactly the rule; the fast path
// only saves work.  The eight codes of a word are packed by a multiply-add
// chain (Horner) on those float bit patterns, and one addition removes the
// 2^23 terms.  The tables are replicated once per lane in shared memory, so
// the data-dependent lookups of a warp never collide on a bank.
#pragma once

#include "common.cuh"
#include "double_quant.cuh"

namespace nf4q {

constexpr int kQuantThreads = 512;
constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kTinyScale = 7.88860905e-31f;     // 2^-100
constexpr float kHugeScale = 8.50705917e37f;      // 2^126
constexpr int kLutWords = kLutEntries * 32;       // one table, replicated per lane

struct QuantParams {
  float lut_t[kLutEntries];     // decision point within reach of each bin
  int32_t lut_lo[kLutEntries];  // code below it
  int32_t lut_dl[kLutEntries];  // change of code across it (FP4 only)
  float thr[15];                // exact-path decision points
};

// Shared-memory tables, one copy per lane: entry e of lane l is the pair
// {-T * 2^19, 2^23 + lo} at byte (e * 32 + l) * 8 (T the decision point in
// reach of bin e, lo the code below it), and for FP4 the float code step dl
// at byte kPairBytes + (e * 32 + l) * 4.
constexpr uint32_t kPairBytes = kLutEntries * 32 * 8;
constexpr float kTwo19 = 524288.0f;
constexpr uint32_t kCodeMagicFix = 0x05000000u;  // -(2^23 bits * (16 + 1)) mod 2^32

__device__ __forceinline__ float sat_add0(float e) {
  float r;  // clamp to [0, 1]
  asm("add.sat.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(e));
  return r;
}

// Fast code of one element v of a block with approximate reciprocal scale
// r (r128 = 128 r, r19 = 2^19 r, both exact): bin from v * r128, then
// e = (v r - T) 2^19 in one FMA on the exact product v r.  |e| <= 1 flags the
// unit for the exact path; otherwise sat(e) is the compare bit exactly.
// `lane_tab` / `lane_dl` are this lane's table columns minus the magic
// offset of the bin, so each address is one multiply-add.  Returns the code
// as the bits of the float 2^23 + code.
template <int CODE>
__device__ __forceinline__ uint32_t code_fast(float v, float r128, float r19, uint32_t lane_tab,
                                              uint32_t lane_dl, float& near) {
  const float y = __fmaf_rn(v, r128, 129.0f + kMagic);
  const uint32_t yb = __float_as_uint(y);
  float ntp, lof;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(ntp), "=f"(lof) : "r"(yb * 256u + lane_tab));
  const float e = __fmaf_rn(v, r19, ntp);
  near = fminf(near, fabsf(e));  // <= 1: v r within about 2^-19 of T
  const float bit = sat_add0(e);
  float c;
  if (CODE == 0) {
    c = __fadd_rn(lof, bit);
  } else {
    float dl;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(dl) : "r"(yb * 128u + lane_dl));
    c = __fmaf_rn(bit, dl, lof);
  }
  return __float_as_uint(c);
}

// The code of v (bits of 2^23 + code, as code_fast) with the comparison at
// the bin's decision point T made on the exact quotient q = fp32(v / a) when
// v r is within reach of T (|e| <= 1); otherwise the fast compare bit, which
// is exact there.  The bins carry a quarter-bin margin and v r is within
// 2^-21 of the quotient, so T is also the only decision point that can
// separate q from the bin's lower code: lo + [q beyond T] dl is the rule,
// with "beyond" q > T for NF4 and for FP4's positive points, and q >= T for
// FP4's negative points -T_j (the FP4 rule compares |q| > T_j, so a tie
// keeps the smaller magnitude).
template <int CODE>
__device__ __forceinline__ uint32_t code_fixed(float v, float a, float r128, float r19,
                                               uint32_t lane_tab, uint32_t lane_dl) {
  const float y = __fmaf_rn(v, r128, 129.0f + kMagic);
  const uint32_t yb = __float_as_uint(y);
  float ntp, lof;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(ntp), "=f"(lof) : "r"(yb * 256u + lane_tab));
  const float e = __fmaf_rn(v, r19, ntp);
  float bit = sat_add0(e);
  if (fabsf(e) <= 1.0f) {
    const float q = __fdiv_rn(v, a), t = -ntp * (1.0f / kTwo19);  // t exact: a power-of-two scaling
    bit = (CODE == 1 && t < 0.f) ? (q >= t ? 1.0f : 0.0f) : (q > t ? 1.0f : 0.0f);
  }
  if (CODE == 0) return __float_as_uint(__fadd_rn(lof, bit));
  float dl;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(dl) : "r"(yb * 128u + lane_dl));
  return __float_as_uint(__fmaf_rn(bit, dl, lof));
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

// Widening of the two 16-bit values of a word: IN = 1 bf16, 2 fp16 (exact).
template <int IN>
__device__ __forceinline__ float lo16_to_f32(uint32_t v) {
  return IN == 1 ? bf16lo_to_f32(v) : f16lo_to_f32(v);
}
template <int IN>
__device__ __forceinline__ float hi16_to_f32(uint32_t v) {
  return IN == 1 ? bf16hi_to_f32(v) : f16hi_to_f32(v);
}

// Input dtype IN: 0 fp32, 1 bf16, 2 fp16 (nf4q_in_dtype).
template <int IN>
__device__ __forceinline__ void load_unit(const void* base, int64_t unit,
                                          float (&v)[8]) {
  if (IN != 0) {
    const uint4 r = ld_stream_u4(static_cast<const uint16_t*>(base) + unit * 8);
    v[0] = lo16_to_f32<IN>(r.x); v[1] = hi16_to_f32<IN>(r.x);
    v[2] = lo16_to_f32<IN>(r.y); v[3] = hi16_to_f32<IN>(r.y);
    v[4] = lo16_to_f32<IN>(r.z); v[5] = hi16_to_f32<IN>(r.z);
    v[6] = lo16_to_f32<IN>(r.w); v[7] = hi16_to_f32<IN>(r.w);
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

// Raw 16-byte loads of the 16 elements of unit `unit` (zeros if !live).
template <int IN>
__device__ __forceinline__ void load_raw(const void* base, int64_t unit, bool live,
                                         uint4 (&raw)[IN != 0 ? 2 : 4]) {
#pragma unroll
  for (int i = 0; i < (IN != 0 ? 2 : 4); ++i)
    raw[i] = live ? ld_stream_u4(static_cast<const uint4*>(base) + unit * (IN != 0 ? 2 : 4) + i)
                  : make_uint4(0u, 0u, 0u, 0u);
}

template <int IN>
__device__ __forceinline__ void unpack_raw(const uint4 (&raw)[IN != 0 ? 2 : 4], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < (IN != 0 ? 2 : 4); ++i) {
    const uint32_t q[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (IN != 0) {
        v[8 * i + 2 * j] = lo16_to_f32<IN>(q[j]);
        v[8 * i + 2 * j + 1] = hi16_to_f32<IN>(q[j]);
      } else {
        v[4 * i + j] = __uint_as_float(q[j]);
      }
    }
  }
}

// The exact rule for the word (8 elements) `word` of the weight, reading
// its elements again (rare: only words with a value near a decision point
// or blocks with an extreme scale come here).
template <int CODE, int IN>
__device__ __noinline__ uint32_t encode_word_exact(const void* w, int64_t word, float a,
                                                   const QuantParams& P) {
  float v[8];
  load_unit<IN>(w, word, v);
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) out |= code_exact<CODE>(v[i], a, P) << nib_shift(i);
  return out;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;  // NaN if either is NaN, so a non-finite block is always seen
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// One lane handles units of 16 consecutive elements (two packed words); a
// 64-block is four consecutive lanes, so its absmax is a 2-step butterfly.
// DQ: also the first pass of double quantization - the absmax values are
// summed exactly into `ws` and the last CTA writes their mean to `offset`
// (double_quant.cuh).
template <int CODE, int IN, bool DQ>
__global__ void __launch_bounds__(kQuantThreads, 2)
quantize_kernel(const void* __restrict__ w, uint2* __restrict__ packed,
                float* __restrict__ absmax, int64_t n_units,
                const __grid_constant__ QuantParams P, DqWorkspace* __restrict__ ws,
                float* __restrict__ offset) {
  extern __shared__ __align__(16) uint32_t s_lut[];  // pairs, then (FP4) steps
  // DQ: exact running sum of each group leader's absmax values (a leader is
  // the lane that stores a block's absmax), kept in shared memory to spare
  // registers; and the out-of-range flag
  __shared__ unsigned long long s_dq[DQ ? kQuantThreads / 4 : 1][2];
  __shared__ int s_dq_oor;
  if (DQ && (threadIdx.x & 3) == 0) s_dq[threadIdx.x >> 2][0] = s_dq[threadIdx.x >> 2][1] = 0ull;
  if (DQ && threadIdx.x == 0) s_dq_oor = 0;
  // 16-byte stores: two pairs (same entry) per store, four steps per store.
  // Every parameter load of the build is issued before the first store, so
  // that their latency (the parameters are not yet cached at kernel start)
  // is paid once.
  static_assert(kLutWords % 4 == 0, "table stores");
  {
    constexpr int kPairIt = (kLutWords / 2 + kQuantThreads - 1) / kQuantThreads;
    constexpr int kStepIt = (kLutWords / 4 + kQuantThreads - 1) / kQuantThreads;
    float tv[kPairIt], lv[kPairIt], dv[kStepIt];
#pragma unroll
    for (int k = 0; k < kPairIt; ++k) {
      const int e = min((static_cast<int>(threadIdx.x) + k * kQuantThreads) >> 4, kLutEntries - 1);
      tv[k] = P.lut_t[e];
      lv[k] = static_cast<float>(P.lut_lo[e]);
    }
#pragma unroll
    for (int k = 0; k < kStepIt; ++k) {
      const int e = min((static_cast<int>(threadIdx.x) + k * kQuantThreads) >> 3, kLutEntries - 1);
      dv[k] = CODE == 1 ? static_cast<float>(P.lut_dl[e]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPairIt; ++k) {
      const int i = threadIdx.x + k * kQuantThreads;
      if (i < kLutWords / 2) {
        const uint32_t a = __float_as_uint(-(tv[k] * kTwo19));
        const uint32_t b = __float_as_uint(8388608.0f + lv[k]);
        reinterpret_cast<uint4*>(s_lut)[i] = make_uint4(a, b, a, b);
      }
    }
    if (CODE == 1) {
#pragma unroll
      for (int k = 0; k < kStepIt; ++k) {
        const int i = threadIdx.x + k * kQuantThreads;
        if (i < kLutWords / 4) {
          const uint32_t d = __float_as_uint(dv[k]);
          reinterpret_cast<uint4*>(s_lut + 2 * kLutWords)[i] = make_uint4(d, d, d, d);
        }
      }
    }
  }
  // Launched as a programmatic dependent of the kernel before it: the
  // tables above are built while that kernel finishes; nothing in global
  // memory is read or written before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t tab = static_cast<uint32_t>(__cvta_generic_to_shared(s_lut));
  const uint32_t lane_tab = tab + lane * 8u - kMagicBits * 256u;
  const uint32_t lane_dl = tab + kPairBytes + lane * 4u - kMagicBits * 128u;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;

  // The raw input of the next unit is loaded before the current one is
  // encoded, which doubles the bytes each lane keeps in flight.
  constexpr int kRaw = IN != 0 ? 2 : 4;  // 16-byte loads per unit
  uint4 nxt[kRaw];
  int64_t unit = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  load_raw<IN>(w, unit, unit < n_units, nxt);
  for (; unit - lane < n_units; unit += nthreads) {
    const bool live = unit < n_units;
    float v[16];
    unpack_raw<IN>(nxt, v);
    load_raw<IN>(w, unit + nthreads, unit + nthreads < n_units, nxt);
    float a = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 16; ++i) a = max_nan(a, fabsf(v[i]));
    a = max_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = max_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    // 2^-100 <= a <= 2^126: the reciprocal is a normal number (the
    // approximate one flushes subnormal results) and 2^19 r <= 2^119 is
    // finite, so |v r| <= 1 + 2^-21 and every bin index is inside the
    // table; anything else (zero, tiny, huge or non-finite absmax) takes
    // the exact path
    const bool ok = a >= kTinyScale && a <= kHugeScale;
    uint32_t word[2] = {0u, 0u};
    float near[2] = {2.0f, 2.0f};
    if (ok) {
      // Approximate reciprocal (relative error <= 2^-22): v r stays within
      // 2^-21 of the exact quotient, inside the 2^-19 exact-fallback window.
      float r;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
      const float r128 = r * 128.0f, r19 = r * kTwo19;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // Horner over the nibble order of the word: elements 6, 7, 4, 5,
        // 2, 3, 0, 1 (element 2j is the high nibble of byte j); the 2^23
        // of each code adds a constant that one addition removes
        const float* vh = v + 8 * h;
        uint32_t wd = code_fast<CODE>(vh[6], r128, r19, lane_tab, lane_dl, near[h]);
#pragma unroll
        for (int k = 1; k < 8; ++k) {
          const int i = (6 - 2 * (k >> 1)) + (k & 1);
          wd = wd * 16u + code_fast<CODE>(vh[i], r128, r19, lane_tab, lane_dl, near[h]);
        }
        if (IN != 0 && near[h] <= 1.0f) {
          // a value within reach of a decision point: the word again, with
          // the exact quotient at that point (16-bit inputs: the values are
          // still in registers; fp32 inputs are read again below, which
          // costs their register-heavier loop less)
          wd = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = (6 - 2 * (k >> 1)) + (k & 1);
            wd = wd * 16u + code_fixed<CODE>(vh[i], a, r128, r19, lane_tab, lane_dl);
          }
        }
        word[h] = wd + kCodeMagicFix;
      }
    }
    if (live) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!ok) {
          word[h] = encode_word_exact<CODE, IN>(w, 2 * unit + h, a, P);
        } else if (IN == 0 && near[h] <= 1.0f) {
          float r;
          asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
          const float r128 = r * 128.0f, r19 = r * kTwo19;
          float vh[8];
          load_unit<IN>(w, 2 * unit + h, vh);
          uint32_t wd = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = (6 - 2 * (k >> 1)) + (k & 1);
            wd = wd * 16u + code_fixed<CODE>(vh[i], a, r128, r19, lane_tab, lane_dl);
          }
          word[h] = wd + kCodeMagicFix;
        }
      }
      packed[unit] = make_uint2(word[0], word[1]);
      if ((lane & 3u) == 0u) {
        absmax[unit >> 2] = a;
        if constexpr (DQ) {
          unsigned long long A;
          if (dq_fixed(a, A)) {
            unsigned long long* acc = s_dq[threadIdx.x >> 2];
            const unsigned long long lo = acc[0] + A;
            acc[0] = lo;
            if (lo < A) acc[1] += 1ull;
          } else {
            s_dq_oor = 1;
          }
        }
      }
    }
  }
  if constexpr (DQ) {
    // the second double-quant pass may start launching (it waits for this
    // grid to complete before it reads anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    DqStats st;
    if ((threadIdx.x & 3) == 0) {
      st.lo = s_dq[threadIdx.x >> 2][0];
      st.hi = s_dq[threadIdx.x >> 2][1];
    }
    st.oor = threadIdx.x == 0 && s_dq_oor != 0;
    if (dq_commit<kQuantThreads / 32>(st, ws)) dq_finalize(absmax, n_units / 4, ws, offset);
  }
}

inline size_t quantize_smem_bytes(int code) {
  return kPairBytes + (code == 0 ? 0 : static_cast<size_t>(kLutWords) * 4);
}

}  // namespace nf4q
