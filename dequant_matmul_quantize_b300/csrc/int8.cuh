// LLM.int8(): vector-wise int8 quantization and the mixed-precision
// decomposition matmul ("bitsandbytes tutorial", sec. 3.1 and the
// llm_int8_threshold setting of sec. 四; "bitsandbytes introduction", core
// techniques item 2).
//
// Y [M x N] = fp16( C * sx_m * sw_n / 127^2 + sum over outlier k of
//                   X[m, k] * w_hat[n, k] )
// where the outlier columns k are those in which some |X[m, k]| exceeds the
// threshold, C is the integer sum of the int8 codes of X (per row, outlier
// columns excluded) and of W (per row) over the other columns, and w_hat is
// the fp16 weight the int8 code gives back, fp16(RN(RN(q * sw) / 127)).
//
// Kernels:
//   int8_quant_weight_kernel  W (fp16 / bf16) -> int8 codes + per-row absmax
//                             (one CTA per row: absmax, then the codes
//                             q = rint(RN(127 w / s)), IEEE division)
//   int8_outlier_flags_kernel one byte per column of X: max |X| > threshold
//   int8_outlier_list_kernel  the outlier columns in ascending order and
//                             their count (one CTA, a block-wide scan)
//   int8_quant_act_kernel     per-row absmax of X over the other columns and
//                             the codes, stored as fp16 integers (exact), the
//                             B operand of the matmul
//   int8_act_small_kernel     the three above in one CTA, for M <= 16
//   int8_mm_kernel            16 rows of W per CTA, K split over 8 warps;
//                             int8 codes -> fp16 integers with a byte permute
//                             and one subtraction (1024 + 128 + q - 1152),
//                             mma.sync m16n8k16 f16 with fp32 accumulation
//                             (products and sums of codes are integers, exact
//                             while a partial sum stays below 2^24); then the
//                             8 partial sums are added in shared memory; the
//                             CTA gathers w_hat and x of the outlier columns
//                             into shared memory and one thread per output
//                             adds their products in fp32 (ascending k) and
//                             applies the two scales.
// The matmul streams the int8 weight once per 8 or 16 rows of X: the decode
// case (M <= 16) is bound by HBM; larger M runs the same kernel once per 16
// rows (correct, not tuned for prefill).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv_mma.cuh"

namespace nf4q {

constexpr int kI8Threads = 256;
constexpr int kI8Rows = 16;     // weight rows per matmul CTA
constexpr int kI8Warps = 8;     // K split across the warps of a CTA
constexpr int kI8Chunk = 128;   // k per warp step
constexpr float kI8Levels = 127.f;
constexpr int kI8OutlierTile = 128;  // outlier columns gathered per pass

// Workspace of nf4q_int8_matmul: sections 256-byte aligned.
struct Int8Workspace {
  size_t flags, count, list, sx, xq, total;
};
inline size_t i8_align(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
inline Int8Workspace int8_workspace_layout(int64_t M, int64_t K) {
  Int8Workspace w;
  w.flags = 0;
  w.count = i8_align(static_cast<size_t>(K));
  w.list = w.count + 256;
  w.sx = w.list + i8_align(4 * static_cast<size_t>(K));
  w.xq = w.sx + i8_align(4 * static_cast<size_t>(M));
  w.total = w.xq + i8_align(2 * static_cast<size_t>(M) * static_cast<size_t>(K));
  return w;
}

template <int IN>  // 1 bf16, 2 fp16
__device__ __forceinline__ void widen8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (IN == 1) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    } else {
      f[2 * i] = f16lo_to_f32(w[i]);
      f[2 * i + 1] = f16hi_to_f32(w[i]);
    }
  }
}

// Block-wide max of non-negative values (all threads get the result).
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red may still be read from a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  return m;
}

// q = rint(RN(127 v / s)) (127 v is exact for 16-bit inputs); s > 0.
__device__ __forceinline__ int code_of(float v, float s) {
  return __float2int_rn(__fdiv_rn(kI8Levels * v, s));
}

// ---------------------------------------------------------------- weights
template <int IN>
__global__ void __launch_bounds__(kI8Threads)
int8_quant_weight_kernel(const uint16_t* __restrict__ w, int8_t* __restrict__ q,
                         float* __restrict__ scale, int K) {
  __shared__ float red[kI8Threads / 32];
  const int64_t row = blockIdx.x;
  const uint16_t* wr = w + row * K;
  float m = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += kI8Threads * 8) {
    float f[8];
    widen8<IN>(*reinterpret_cast<const uint4*>(wr + k), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
  const float s = block_max(m, red);
  if (threadIdx.x == 0) scale[row] = s;
  int8_t* qr = q + row * K;
  for (int k = threadIdx.x * 8; k < K; k += kI8Threads * 8) {
    float f[8];
    widen8<IN>(*reinterpret_cast<const uint4*>(wr + k), f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = static_cast<uint32_t>(s > 0.f ? code_of(f[j], s) : 0) & 0xFFu;
      if (j < 4) lo |= b << (8 * j); else hi |= b << (8 * (j - 4));
    }
    *reinterpret_cast<uint2*>(qr + k) = make_uint2(lo, hi);
  }
}

// ---------------------------------------------------------------- activations
// flags[k] = 1 when some |X[m, k]| > threshold (threshold > 0).  A CTA takes
// 256 columns: 32 groups of 8 columns x 8 row phases.
__global__ void __launch_bounds__(kI8Threads)
int8_outlier_flags_kernel(const uint16_t* __restrict__ X, int M, int K, float threshold,
                          uint8_t* __restrict__ flags) {
  __shared__ float colmax[8][256];
  const int cg = threadIdx.x & 31, rp = threadIdx.x >> 5;
  const int k0 = blockIdx.x * 256 + cg * 8;
  float mx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (k0 < K) {
    for (int m = rp; m < M; m += 8) {
      float f[8];
      widen8<2>(*reinterpret_cast<const uint4*>(X + static_cast<int64_t>(m) * K + k0), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) mx[j] = fmaxf(mx[j], fabsf(f[j]));
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) colmax[rp][cg * 8 + j] = mx[j];
  __syncthreads();
  const int k = blockIdx.x * 256 + threadIdx.x;
  if (k < K) {
    float v = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) v = fmaxf(v, colmax[p][threadIdx.x]);
    flags[k] = (threshold > 0.f && v > threshold) ? 1 : 0;
  }
}

// The outlier columns in ascending order and their count (one CTA of 1024).
__global__ void __launch_bounds__(1024)
int8_outlier_list_kernel(const uint8_t* __restrict__ flags, int K, int32_t* __restrict__ list,
                         int32_t* __restrict__ count) {
  __shared__ int warp_sum[32];
  const int per = (K + 1023) / 1024;
  const int b = threadIdx.x * per, e = min(K, b + per);
  int n = 0;
  for (int k = b; k < e; ++k) n += flags[k];
  // exclusive scan of n over the block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += t;
    }
    warp_sum[lane] = v;  // inclusive prefix over warps
  }
  __syncthreads();
  int pos = incl - n + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (int k = b; k < e; ++k)
    if (flags[k]) list[pos++] = k;
  if (threadIdx.x == 1023) *count = pos;
}

// Row m of X: scale sx[m] = max |X[m, k]| over the non-outlier columns, and
// the codes as fp16 integers (0 in outlier columns and when sx = 0).
__global__ void __launch_bounds__(kI8Threads)
int8_quant_act_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ flags, int K,
                      float* __restrict__ sx, uint16_t* __restrict__ xq) {
  __shared__ float red[kI8Threads / 32];
  const int64_t row = blockIdx.x;
  const uint16_t* xr = X + row * K;
  float m = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += kI8Threads * 8) {
    float f[8];
    widen8<2>(*reinterpret_cast<const uint4*>(xr + k), f);
    const uint2 fl = *reinterpret_cast<const uint2*>(flags + k);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t bit = ((j < 4 ? fl.x : fl.y) >> (8 * (j & 3))) & 0xFFu;
      if (!bit) m = fmaxf(m, fabsf(f[j]));
    }
  }
  const float s = block_max(m, red);
  if (threadIdx.x == 0) sx[row] = s;
  uint16_t* qr = xq + row * K;
  for (int k = threadIdx.x * 8; k < K; k += kI8Threads * 8) {
    float f[8];
    widen8<2>(*reinterpret_cast<const uint4*>(xr + k), f);
    const uint2 fl = *reinterpret_cast<const uint2*>(flags + k);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t bit = (((j + h) < 4 ? fl.x : fl.y) >> (8 * ((j + h) & 3))) & 0xFFu;
        c[h] = (bit || !(s > 0.f)) ? 0.f : static_cast<float>(code_of(f[j + h], s));
      }
      o[j / 2] = pack_f16x2(c[0], c[1]);
    }
    *reinterpret_cast<uint4*>(qr + k) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The whole activation side in one CTA of 1024 threads, for M <= 16 (one
// launch instead of three): thread t owns the column groups (8 columns)
// [t * per, (t + 1) * per), writes their flags and counts its outliers; a
// block-wide scan orders the list; then the rows' scales and codes.  Flags
// written here are read back by other threads after __syncthreads with
// ordinary loads (not the read-only path).
__global__ void __launch_bounds__(1024)
int8_act_small_kernel(const uint16_t* __restrict__ X, int M, int K, float threshold,
                      uint8_t* flags, int32_t* __restrict__ list, int32_t* __restrict__ count,
                      float* __restrict__ sx, uint16_t* __restrict__ xq) {
  __shared__ int warp_sum[32];
  __shared__ float red[32];
  const int groups = K / 8;
  const int per = (groups + 1023) / 1024;
  const int gb = threadIdx.x * per, ge = min(groups, gb + per);
  int n = 0;
  for (int gi = gb; gi < ge; ++gi) {
    float mx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int m = 0; m < M; ++m) {
      float f[8];
      widen8<2>(*reinterpret_cast<const uint4*>(X + static_cast<int64_t>(m) * K + gi * 8), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) mx[j] = fmaxf(mx[j], fabsf(f[j]));
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t o = (threshold > 0.f && mx[j] > threshold) ? 1u : 0u;
      n += static_cast<int>(o);
      if (j < 4) lo |= o << (8 * j); else hi |= o << (8 * (j - 4));
    }
    *reinterpret_cast<uint2*>(flags + gi * 8) = make_uint2(lo, hi);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += t;
    }
    warp_sum[lane] = v;
  }
  __syncthreads();
  int pos = incl - n + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (int k = gb * 8; k < ge * 8; ++k)
    if (flags[k]) list[pos++] = k;
  if (threadIdx.x == 1023) *count = warp_sum[31];
  __syncthreads();  // every flag is visible to the whole block
  // rows: a team of 1024 / M2 threads per row (M2 = M rounded up to a power
  // of two), all rows at once; team maxima through warp shuffles and one
  // shared-memory pass over the team's warps
  int M2 = 1;
  while (M2 < M) M2 *= 2;
  const int ts = 1024 / M2;            // >= 64: whole warps
  const int team = threadIdx.x / ts, tin = threadIdx.x - team * ts;
  const bool has_row = team < M;
  const uint16_t* xr = X + static_cast<int64_t>(has_row ? team : 0) * K;
  float mx = 0.f;
  if (has_row) {
#pragma unroll 4
    for (int gi = tin; gi < groups; gi += ts) {
      float f[8];
      widen8<2>(*reinterpret_cast<const uint4*>(xr + gi * 8), f);
      const uint2 fl = *reinterpret_cast<const uint2*>(flags + gi * 8);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!(((j < 4 ? fl.x : fl.y) >> (8 * (j & 3))) & 0xFFu)) mx = fmaxf(mx, fabsf(f[j]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  const int wpt = ts / 32;
  float sm = 0.f;
  for (int i = 0; i < wpt; ++i) sm = fmaxf(sm, red[team * wpt + i]);
  if (!has_row) return;
  if (tin == 0) sx[team] = sm;
#pragma unroll 4
  for (int gi = tin; gi < groups; gi += ts) {
    float f[8];
    widen8<2>(*reinterpret_cast<const uint4*>(xr + gi * 8), f);
    const uint2 fl = *reinterpret_cast<const uint2*>(flags + gi * 8);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float c2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t bit = (((j + h) < 4 ? fl.x : fl.y) >> (8 * ((j + h) & 3))) & 0xFFu;
        c2[h] = (bit || !(sm > 0.f)) ? 0.f : static_cast<float>(code_of(f[j + h], sm));
      }
      o[j / 2] = pack_f16x2(c2[0], c2[1]);
    }
    *reinterpret_cast<uint4*>(xq + static_cast<int64_t>(team) * K + gi * 8) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// 4-byte asynchronous copy global -> shared; `valid` false fills zeros and
// reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- matmul
// Four int8 codes (bytes 0..3 of w) -> fp16x2 of codes 0, 1 and of 2, 3:
// the byte q + 128 under the fp16 exponent of 1024 is 1152 + q exactly, and
// one subtraction of 1152 leaves q.
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = prmt(u, 0x64646464u, 0x4140u);
  const uint32_t b = prmt(u, 0x64646464u, 0x4342u);
  const uint32_t k1152 = 0x64806480u;  // fp16x2 (1152, 1152)
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(k1152));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(k1152));
}

// NT n-tiles of 8 activation rows.  Thread (g, c) = (lane / 4, lane % 4) of
// a warp holds, per k step of 128, the 32 consecutive k = k0 + 32c .. + 31
// of weight rows g and g + 8 (two 16-byte loads each) and of activation row
// m0 + 8t + g; MMA i (0..7) takes physical k = k0 + 32c + 4i .. + 3 as its
// logical k {2c, 2c+1, 2c+8, 2c+9} for both operands (any common
// permutation of k leaves the dot products unchanged).
template <int NT>
__global__ void __launch_bounds__(kI8Threads)
int8_mm_kernel(const int8_t* __restrict__ Wq, const float* __restrict__ sw,
               const uint16_t* __restrict__ X, const uint16_t* __restrict__ Xq,
               const float* __restrict__ sx, const int32_t* __restrict__ outl,
               const int32_t* __restrict__ n_outl, uint16_t* __restrict__ Y, int N, int K,
               int M) {
  __shared__ float red[kI8Warps][NT][kI8Rows][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int n0 = blockIdx.x * kI8Rows;
  const int m0 = blockIdx.y * 8 * NT;
  const int r0 = n0 + g, r1 = n0 + g + 8;
  const int nchunks = (K + kI8Chunk - 1) / kI8Chunk;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  auto load_w = [&](int kc, uint4 (&w)[4]) {
    const int p = kc * kI8Chunk + 32 * c;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool in = p + 16 * h < K;
      w[h] = (r0 < N && in) ? ld_stream_u4(Wq + static_cast<int64_t>(r0) * K + p + 16 * h)
                            : make_uint4(0, 0, 0, 0);
      w[2 + h] = (r1 < N && in) ? ld_stream_u4(Wq + static_cast<int64_t>(r1) * K + p + 16 * h)
                                : make_uint4(0, 0, 0, 0);
    }
  };
  // the next k step's weight loads are issued before the current one is used
  uint4 wcur[4], wnext[4];
  if (warp < nchunks) load_w(warp, wcur);
  // Outlier columns, kI8OutlierTile at a time.  The tile's column list is
  // copied to shared memory; then every 4-byte word holding W[n, k] (16
  // rows) and X[m, k] (8 NT rows) is gathered into shared memory with
  // cp.async, which needs no registers: for the first tile the copies are
  // issued before the main loop and land while it streams the weight.
  // After the loop the words become w_hat and x (fp32), and one thread per
  // output adds their products in ascending k.
  __shared__ int32_t lst[kI8OutlierTile];
  __shared__ uint32_t gw[kI8Rows][kI8OutlierTile + 1];
  __shared__ uint32_t gx[8 * NT][kI8OutlierTile + 1];
  const int row = threadIdx.x & (kI8Rows - 1);
  const int col = threadIdx.x >> 4;       // 0 .. 8 NT - 1 for the output threads
  const bool outputs = threadIdx.x < kI8Rows * 8 * NT;
  const int n = n0 + row, m = m0 + col;
  float out = 0.f;
  const int no = *n_outl;
  auto issue_tile = [&](int j0, int cnt) {
    for (int i = threadIdx.x; i < cnt; i += kI8Threads) lst[i] = outl[j0 + i];
    __syncthreads();
    for (int i = threadIdx.x; i < kI8Rows * cnt; i += kI8Threads) {
      const int r = i / cnt, j = i - r * cnt;
      const int nn = n0 + r;
      const int8_t* src = Wq + static_cast<int64_t>(nn < N ? nn : 0) * K + (lst[j] & ~3);
      cp_async_4(smem_u32(&gw[r][j]), src, nn < N);
    }
    for (int i = threadIdx.x; i < 8 * NT * cnt; i += kI8Threads) {
      const int r = i / cnt, j = i - r * cnt;
      const int mm = m0 + r;
      const uint16_t* src = X + static_cast<int64_t>(mm < M ? mm : 0) * K + (lst[j] & ~1);
      cp_async_4(smem_u32(&gx[r][j]), src, mm < M);
    }
    cp_async_commit();
  };
  auto finish_tile = [&](int cnt) {
    cp_async_wait_all();
    __syncthreads();
    for (int i = threadIdx.x; i < kI8Rows * cnt; i += kI8Threads) {
      const int r = i / cnt, j = i - r * cnt;
      const int nn = n0 + r;
      const int q = static_cast<int8_t>((gw[r][j] >> (8 * (lst[j] & 3))) & 0xFFu);
      const float v = nn < N
          ? __half2float(__float2half_rn(__fdiv_rn(__fmul_rn(static_cast<float>(q),
                                                             __ldg(sw + nn)), kI8Levels)))
          : 0.f;
      gw[r][j] = __float_as_uint(v);
    }
    for (int i = threadIdx.x; i < 8 * NT * cnt; i += kI8Threads) {
      const int r = i / cnt, j = i - r * cnt;
      const uint32_t h = (gx[r][j] >> (16 * (lst[j] & 1))) & 0xFFFFu;
      gx[r][j] = __float_as_uint(__half2float(__ushort_as_half(static_cast<uint16_t>(h))));
    }
    __syncthreads();
    if (outputs) {
      for (int j = 0; j < cnt; ++j)
        out = __fmaf_rn(__uint_as_float(gx[col][j]), __uint_as_float(gw[row][j]), out);
    }
    __syncthreads();  // the tile's shared memory may be reused
  };
  if (no > 0) issue_tile(0, min(kI8OutlierTile, no));
  for (int kc = warp; kc < nchunks; kc += kI8Warps) {
    if (kc + kI8Warps < nchunks) load_w(kc + kI8Warps, wnext);
    const int p = kc * kI8Chunk + 32 * c;
    const uint32_t w0[8] = {wcur[0].x, wcur[0].y, wcur[0].z, wcur[0].w,
                            wcur[1].x, wcur[1].y, wcur[1].z, wcur[1].w};
    const uint32_t w1[8] = {wcur[2].x, wcur[2].y, wcur[2].z, wcur[2].w,
                            wcur[3].x, wcur[3].y, wcur[3].z, wcur[3].w};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int xm = m0 + 8 * t + g;  // activation row of this thread's B fragment
      uint32_t xw[16];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 v = (xm < M && p + 8 * h < K)
            ? __ldg(reinterpret_cast<const uint4*>(Xq + static_cast<int64_t>(xm) * K + p + 8 * h))
            : make_uint4(0, 0, 0, 0);
        xw[4 * h] = v.x; xw[4 * h + 1] = v.y; xw[4 * h + 2] = v.z; xw[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a0, a2, a1, a3;
        codes_to_f16(w0[i], a0, a2);  // row g: k 4i, 4i+1 | 4i+2, 4i+3
        codes_to_f16(w1[i], a1, a3);  // row g + 8
        mma_16816<1>(acc[t], a0, a1, a2, a3, xw[2 * i], xw[2 * i + 1]);
      }
    }
    if (kc + kI8Warps < nchunks) {
#pragma unroll
      for (int j = 0; j < 4; ++j) wcur[j] = wnext[j];
    }
  }
  if (no > 0) {
    finish_tile(min(kI8OutlierTile, no));
    for (int j0 = kI8OutlierTile; j0 < no; j0 += kI8OutlierTile) {
      issue_tile(j0, min(kI8OutlierTile, no - j0));
      finish_tile(min(kI8OutlierTile, no - j0));
    }
  }
  // C fragment: acc[t][0..1] = rows g, columns 2c, 2c+1; [2..3] = rows g + 8
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    red[warp][t][g][2 * c] = acc[t][0];
    red[warp][t][g][2 * c + 1] = acc[t][1];
    red[warp][t][g + 8][2 * c] = acc[t][2];
    red[warp][t][g + 8][2 * c + 1] = acc[t][3];
  }
  __syncthreads();
  if (outputs && n < N && m < M) {
    const int t = col >> 3, cc = col & 7;
    float cint = 0.f;
#pragma unroll
    for (int w = 0; w < kI8Warps; ++w) cint += red[w][t][row][cc];
    const float scale = __fmul_rn(__fmul_rn(__ldg(sx + m), __ldg(sw + n)),
                                  1.f / (kI8Levels * kI8Levels));
    Y[static_cast<int64_t>(m) * N + n] =
        __half_as_ushort(__float2half_rn(__fmaf_rn(cint, scale, out)));
  }
}

}  // namespace nf4q
