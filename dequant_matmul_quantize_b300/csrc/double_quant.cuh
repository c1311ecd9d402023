// double_quant: the fp32 absmax scales are quantized a second time
// ("bitsandbytes tutorial", sec. 3.3): offset = mean(absmax); c = absmax -
// offset; per block of 256, scale2 = max|c| / 127 and q = rint(c / scale2)
// as int8.
//
// The mean is the float32 nearest to the EXACT mean, whatever the order in
// which the GPU adds things up:
//   pass 1 (dq_sum_kernel, or fused into the quantize kernel): every value
//     a in [2^-32, 2^8) is the integer a * 2^55 < 2^63 exactly; threads add
//     these integers in 128 bits, CTAs combine theirs with 64-bit atomics
//     (carry propagated by hand), so the total is exact and independent of
//     the order.  A non-zero value outside that range (or not finite) raises
//     a flag.  The last CTA to finish divides the exact total by n_b with
//     integer arithmetic and rounds to float32 (ties to even); if the flag
//     is up it first re-adds all values exactly as per-exponent integer
//     mantissa sums into a 320-bit integer instead.  Integer work only: the
//     fp64 units of this GPU are far too slow to sit in the quantize loop.
//   pass 2 (dq_quant_kernel): one warp per 256-block.
#pragma once

#include "common.cuh"

namespace nf4q {


// Layout of the double-quant workspace.  It is zero before pass 1, and the
// CTA that finalizes the mean reads it and clears it again, so a caller
// zero-fills it once and reuses it without clearing.  The exact
// total of a * 2^55 over the in-range values (below 2^128) is kept as three
// 43-bit chunks, each summed over the CTAs on its own: a CTA's chunk is
// below 2^43 and there are fewer than 2^20 CTAs, so no chunk sum carries
// out of 64 bits and the CTAs add without reading anything back.
constexpr int kDqChunkBits = 43;
struct DqWorkspace {
  unsigned long long chunk[3];  // bits [0, 43), [43, 86), [86, 128) of the total, summed
  uint32_t out_of_range;        // some non-zero value outside [2^-32, 2^8)
  uint32_t ticket;              // CTAs finished
  uint32_t pad[8];
};
static_assert(sizeof(DqWorkspace) == 64, "workspace layout");
constexpr int kDqFixShift = 55;  // fixed point: a * 2^55

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

constexpr int kDqSumThreads = 512;
constexpr int kDqQuantThreads = 256;

// Running exact sum of one thread over absmax values (fixed point 2^-55,
// 128 bits) and the out-of-range flag.
// a * 2^55 as an integer (0 for a == 0); false if a is non-zero and outside
// [2^-32, 2^8) (or not finite).
__device__ __forceinline__ bool dq_fixed(float a, unsigned long long& A) {
  const uint32_t bits = __float_as_uint(a) & 0x7FFFFFFFu;
  const uint32_t e = bits >> 23;  // a = 1.m * 2^(e - 127)
  A = 0ull;
  if (bits == 0u) return true;
  if (e < 95u || e > 134u) return false;
  A = static_cast<unsigned long long>((bits & 0x7FFFFFu) | 0x800000u) << (e - 95u);
  return true;
}

struct DqStats {
  unsigned long long lo = 0, hi = 0;
  bool oor = false;
  __device__ __forceinline__ void add(float a) {
    unsigned long long A;
    if (!dq_fixed(a, A)) { oor = true; return; }
    lo += A;
    hi += lo < A ? 1ull : 0ull;
  }
};

// Combines the sums of all threads of the CTA into the workspace and takes
// a ticket; true (in every thread) in the last CTA to finish.  Every
// thread's earlier global writes are visible grid-wide before the ticket.
template <int NWARPS>
__device__ __forceinline__ bool dq_commit(DqStats st, DqWorkspace* ws) {
  __shared__ unsigned long long s_lo[NWARPS], s_hi[NWARPS];
  __shared__ int s_oor[NWARPS];
  __shared__ bool s_last;
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long l2 = __shfl_xor_sync(0xFFFFFFFFu, st.lo, o);
    const unsigned long long h2 = __shfl_xor_sync(0xFFFFFFFFu, st.hi, o);
    st.lo += l2;
    st.hi += h2 + (st.lo < l2 ? 1ull : 0ull);
  }
  const int oor = __any_sync(0xFFFFFFFFu, st.oor);
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { s_lo[wid] = st.lo; s_hi[wid] = st.hi; s_oor[wid] = oor; }
  // Every thread's earlier global writes happen before the barrier, and
  // thread 0's fence after it is cumulative: they are visible grid-wide
  // before its ticket.
  __syncthreads();
  if (threadIdx.x == 0) {
    int any = s_oor[0];
    for (int k = 1; k < NWARPS; ++k) {
      st.lo += s_lo[k];
      st.hi += s_hi[k] + (st.lo < s_lo[k] ? 1ull : 0ull);
      any |= s_oor[k];
    }
    // the CTA's 128-bit total in three carry-free chunks (reductions whose
    // results are not read back, then one fence before the ticket)
    constexpr unsigned long long kMask = (1ull << kDqChunkBits) - 1ull;
    atomicAdd(&ws->chunk[0], st.lo & kMask);
    atomicAdd(&ws->chunk[1], ((st.lo >> kDqChunkBits) | (st.hi << (64 - kDqChunkBits))) & kMask);
    atomicAdd(&ws->chunk[2], st.hi >> (2 * kDqChunkBits - 64));
    if (any) atomicOr(&ws->out_of_range, 1u);
    __threadfence();
    const uint32_t t = atomicAdd(&ws->ticket, 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  return s_last;
}

// Float32 nearest (ties to even) to (hi * 2^64 + lo) * 2^-55 / n, when that
// quotient is at least 2^-31 (so floor(S / n) has 25 bits or more and the
// remainder only feeds the sticky bit); otherwise returns false.  S / n is
// below 2^63 because every summand is.
__device__ __forceinline__ bool dq_round_fixed(unsigned long long lo, unsigned long long hi,
                                               uint32_t n, float* out) {
  const uint32_t limb[4] = {static_cast<uint32_t>(hi >> 32), static_cast<uint32_t>(hi),
                            static_cast<uint32_t>(lo >> 32), static_cast<uint32_t>(lo)};
  unsigned long long q = 0, r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned long long cur = (r << 32) | limb[i];
    const unsigned long long d = cur / n;
    r = cur - d * n;
    q = (q << 32) | d;  // the top limbs of the quotient are zero
  }
  const int p = 64 - __clzll(static_cast<long long>(q));  // bit length of q
  if (p < 25) return false;
  const int sh = p - 24;
  unsigned long long mant = q >> sh;
  const unsigned long long rest = q & ((1ull << sh) - 1ull);
  const unsigned long long half = 1ull << (sh - 1);
  if (rest > half || (rest == half && (r != 0 || (mant & 1ull))) ) ++mant;
  int be = p + 71;  // biased exponent of q * 2^-55: (p - 1) - 55 + 127
  if (mant == (1ull << 24)) { mant >>= 1; ++be; }
  *out = __uint_as_float((static_cast<uint32_t>(be) << 23) | (static_cast<uint32_t>(mant) & 0x7FFFFFu));
  return true;
}

// Run by every thread of the last CTA: *offset = the float32 nearest to the
// exact mean of the nb values at absmax.
__device__ __noinline__ void dq_finalize(const float* __restrict__ absmax, int64_t nb,
                                        DqWorkspace* __restrict__ ws,
                                        float* __restrict__ offset) {
  __shared__ unsigned long long s_hist[256];
  __threadfence();
  const bool oor = __ldcg(&ws->out_of_range) != 0u;
  unsigned long long c0 = 0ull, c1 = 0ull, c2 = 0ull;
  if (threadIdx.x == 0) {
    c0 = __ldcg(&ws->chunk[0]);
    c1 = __ldcg(&ws->chunk[1]);
    c2 = __ldcg(&ws->chunk[2]);
  }
  // every CTA has committed (this one holds the last ticket) and every
  // thread here has read the record: leave it zero for the next call
  __syncthreads();
  if (threadIdx.x == 0) {
    ws->chunk[0] = 0ull;
    ws->chunk[1] = 0ull;
    ws->chunk[2] = 0ull;
    ws->out_of_range = 0u;
    ws->ticket = 0u;
  }
  if (oor) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0ull;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < nb; i += blockDim.x) {
      const uint32_t bits = __float_as_uint(__ldcg(absmax + i)) & 0x7FFFFFFFu;
      const uint32_t e = min(bits >> 23, 254u);
      const uint32_t m = e ? ((bits & 0x7FFFFFu) | 0x800000u) : bits;
      atomicAdd(&s_hist[max(e, 1u)], static_cast<unsigned long long>(m));
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    uint32_t A[kLimbs];  // sum * 2^149
    for (int i = 0; i < kLimbs; ++i) A[i] = 0u;
    if (oor) {
      for (int e = 1; e < 255; ++e)
        if (s_hist[e]) big_add_shifted(A, s_hist[e], e - 1);
    } else {
      // the total from its three chunk sums
      const unsigned long long lo = c0 + (c1 << kDqChunkBits);
      const unsigned long long hi = (c1 >> (64 - kDqChunkBits)) + (c2 << (2 * kDqChunkBits - 64)) +
                                    (lo < c0 ? 1ull : 0ull);
      float m;
      if (dq_round_fixed(lo, hi, static_cast<uint32_t>(nb), &m)) {
        *offset = m;
        return;
      }
      big_add_shifted(A, lo, 149 - kDqFixShift);
      big_add_shifted(A, hi, 149 - kDqFixShift + 64);
    }
    *offset = big_round_mean(A, static_cast<uint32_t>(nb));
  }
}

// ---------------------------------------------------------------- pass 1
__global__ void __launch_bounds__(kDqSumThreads)
dq_sum_kernel(const float* __restrict__ absmax, int64_t nb,
              DqWorkspace* __restrict__ ws, float* __restrict__ offset) {
  DqStats st;
  const int64_t nvec = nb / 4;  // absmax is 16-byte aligned
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += stride) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(absmax) + i);
    st.add(v.x); st.add(v.y); st.add(v.z); st.add(v.w);
  }
  if (blockIdx.x == 0 && threadIdx.x < (nb & 3)) st.add(__ldg(absmax + nvec * 4 + threadIdx.x));
  if (dq_commit<kDqSumThreads / 32>(st, ws)) dq_finalize(absmax, nb, ws, offset);
}

// ---------------------------------------------------------------- pass 2
__global__ void __launch_bounds__(kDqQuantThreads)
dq_quant_kernel(const float* __restrict__ absmax, int64_t nb,
                const float* __restrict__ offset, int8_t* __restrict__ absmax_q,
                float* __restrict__ scale2) {
  // Launched as a programmatic dependent of the fused quantize kernel, this
  // waits here until that grid has completed and its writes (absmax, the
  // mean) are visible; launched normally it returns at once.
  // The next kernel on the stream may launch at once (a quantize kernel
  // builds its tables meanwhile).  Every kernel here launched as a
  // programmatic dependent waits for this grid before it reads or writes
  // memory, save L2 prefetches and the first weight loads of a GEMV called
  // with NF4Q_GEMV_WEIGHTS_STATIC, whose caller guarantees that no running
  // kernel writes those weights.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
