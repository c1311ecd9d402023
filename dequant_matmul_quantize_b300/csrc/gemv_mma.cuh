// nf4_gemv, decode shapes (M <= 16): y[m, n] = sum_k x[m, k] * w_hat[n, k]
// ("bitsandbytes tutorial", sec. 3.4, sec. 七 myth 5: bandwidth-bound, the
// dequantization is extra arithmetic on top of moving the packed weights).
//
// At M = 1 a B300 must turn ~45 packed weights per SM clock into bf16 to keep
// up with HBM, i.e. under three instructions per weight, and at M = 16 the
// CUDA cores could not even do the FMAs.  So the contraction runs on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with the
// weights as the 16-row A operand and x as the 8-column B operand, and the
// per-weight work is a register table lookup:
//   * For each (row, 64-block) the lane that owns it builds the 16 products
//     w_hat_j = bf16(code_j * s_b) - exactly the dequantizer's values - and
//     splits them into a table of high bytes and one of low bytes (4+4
//     registers, 16 one-byte entries each).
//   * Four codes (16 bits of packed data) are looked up with byte permutes:
//     two PRMTs per byte table on the low 3 bits of each nibble, a select on
//     bit 3 (mask built by one sign-replicating PRMT), and two PRMTs that
//     interleave high and low bytes into two bf16x2 A-fragment registers.
// The order of k inside an MMA does not matter as long as x uses the same
// one: lane (g, t) feeds rows g and g+8, 64-block t of each 256-column chunk,
// four columns per MMA; its B fragment is then 64 consecutive x values.
// A CTA owns 16 rows; its warps split K and add their fragments in shared
// memory in a fixed order (deterministic), then one warp writes bf16 y.
#pragma once

#include "common.cuh"
#include "tma.cuh"
#include "lut.cuh"

namespace nf4q {

constexpr int kGemvRows = 16;
constexpr int kGemvChunk = 256;  // columns per warp step (4 blocks)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kGemvStages = 3;
constexpr int kGemvR = 2;  // 16-row tiles per warp (they share x fragments)
constexpr int kGemvTileBytes = kGemvR * kGemvRows * (kGemvChunk / 2);  // 32 rows x 128 B

__device__ __forceinline__ uint32_t lds_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Scale of row r, 64-block blk; 0 outside the weight (so the lookups of
// padded rows and blocks produce zeros and x there may be anything finite).
__device__ __forceinline__ float row_scale(const ScaleView& sv, float off, int r, int N,
                                           int kblocks, int blk) {
  if (r >= N || blk >= kblocks) return 0.f;
  const int64_t b = static_cast<int64_t>(r) * kblocks + blk;
  if (sv.double_quant)
    return __fmaf_rn(static_cast<float>(__ldg(sv.absmax_q + b)), __ldg(sv.scale2 + (b >> 8)), off);
  return __ldg(sv.absmax + b);
}

// Each warp streams its own K range of the CTA's 32 rows through a private
// ring of kGemvStages shared-memory tiles (32 rows x 128 packed bytes = 256
// columns), filled by TMA (128-byte swizzle, so the 8 rows a lane group
// reads land in distinct banks) and tracked by one mbarrier per stage.
// Columns of the MMA beyond M are computed and dropped: lanes of those
// columns load x row min(g, M-1), which keeps every lane's loads identical
// in shape (no predication, no zero fill).
template <int CODE, int NT>
__global__ void __launch_bounds__(512)
gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
                const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int N, int K, int M,
                int per_warp, const __grid_constant__ CodeValues C) {
  extern __shared__ __align__(1024) uint8_t gsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * (kGemvRows * kGemvR);
  const int nchunks = (K + kGemvChunk - 1) / kGemvChunk;
  const int c_begin = warp * per_warp;
  const int c_end = min(nchunks, c_begin + per_warp);
  const int kblocks = K / kBlock;
  const float off = sv.double_quant ? __ldg(sv.offset) : 0.f;
  const uint16_t* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    xrow[nt] = x + static_cast<int64_t>(min(g + 8 * nt, M - 1)) * K;

  const uint32_t smem0 = (lds_addr(gsm) + 1023u) & ~1023u;
  const uint32_t ring = smem0 + warp * (kGemvStages * kGemvTileBytes);
  const uint32_t bars = smem0 + nwarps * (kGemvStages * kGemvTileBytes) + warp * 64;
  float* s_red = reinterpret_cast<float*>(gsm + (smem0 - lds_addr(gsm)) +
                                          nwarps * (kGemvStages * kGemvTileBytes) + nwarps * 64);

  if (lane == 0) {
    for (int st = 0; st < kGemvStages; ++st) mbar_init(bars + 8 * st, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
    for (int i = 0; i < kGemvStages && c_begin + i < c_end; ++i) {
      mbar_arrive_expect_tx(bars + 8 * i, kGemvTileBytes);
      tma_load_2d(ring + i * kGemvTileBytes, &tmap_w, (c_begin + i) * (kGemvChunk / 2), row0,
                  bars + 8 * i);
    }
  }
  __syncwarp();

  float acc[kGemvR][NT][4];
#pragma unroll
  for (int r = 0; r < kGemvR; ++r)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][nt][i] = 0.f;

  // scales of the current chunk, fetched one chunk ahead: [tile][row g, g+8]
  float scur[kGemvR][2];
#pragma unroll
  for (int r = 0; r < kGemvR; ++r) {
    scur[r][0] = row_scale(sv, off, row0 + 16 * r + g, N, kblocks, c_begin * 4 + t);
    scur[r][1] = row_scale(sv, off, row0 + 16 * r + g + 8, N, kblocks, c_begin * 4 + t);
  }
  const int nmine = max(0, c_end - c_begin);
  int issued = min(nmine, kGemvStages);  // TMA loads issued by this warp
  for (int c = c_begin; c < c_end; ++c) {
    const int i = c - c_begin, st = i % kGemvStages;
    const uint32_t ph = (i / kGemvStages) & 1;
    const int blk = c * 4 + t;
    RowTable<CODE> T[kGemvR][2];
#pragma unroll
    for (int r = 0; r < kGemvR; ++r) {
      build_table<CODE>(T[r][0], scur[r][0], C);
      build_table<CODE>(T[r][1], scur[r][1], C);
    }
    if (c + 1 < c_end) {
#pragma unroll
      for (int r = 0; r < kGemvR; ++r) {
        scur[r][0] = row_scale(sv, off, row0 + 16 * r + g, N, kblocks, blk + 4);
        scur[r][1] = row_scale(sv, off, row0 + 16 * r + g + 8, N, kblocks, blk + 4);
      }
    }
    // x columns of this lane's block; blocks past K read block 0 (their
    // weights are zero)
    const int xblk = blk < kblocks ? blk : 0;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_timed(bars + 8 * st, ph))) break;
    const uint32_t tile = ring + st * kGemvTileBytes;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      // 16-byte chunk (2t + hb) of rows g and g + 8 of each tile (128-byte swizzle)
      const uint32_t chunk = ((2 * t + hb) ^ g) << 4;
      uint32_t wds[kGemvR][2][4];
#pragma unroll
      for (int r = 0; r < kGemvR; ++r) {
        const uint4 pa = lds128(tile + (16 * r + g) * 128 + chunk);
        const uint4 pb = lds128(tile + (16 * r + g + 8) * 128 + chunk);
        wds[r][0][0] = pa.x; wds[r][0][1] = pa.y; wds[r][0][2] = pa.z; wds[r][0][3] = pa.w;
        wds[r][1][0] = pb.x; wds[r][1][1] = pb.y; wds[r][1][2] = pb.z; wds[r][1][3] = pb.w;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int wi = 4 * hb + q;  // word of the block: elements 8wi .. 8wi+7
        uint32_t xb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(xrow[nt] + xblk * 64 + wi * 8));
          xb[nt][0] = v.x; xb[nt][1] = v.y; xb[nt][2] = v.z; xb[nt][3] = v.w;
        }
#pragma unroll
        for (int r = 0; r < kGemvR; ++r) {
          uint32_t ra[4], rb[4];
          dequant_word<CODE>(T[r][0], wds[r][0][q], ra);
          dequant_word<CODE>(T[r][1], wds[r][1][q], rb);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16_16816(acc[r][nt], ra[2 * h], rb[2 * h], ra[2 * h + 1], rb[2 * h + 1],
                             xb[nt][2 * h], xb[nt][2 * h + 1]);
        }
      }
    }
    __syncwarp();
    if (c + kGemvStages < c_end) {  // refill this stage
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bars + 8 * st, kGemvTileBytes);
        tma_load_2d(tile, &tmap_w, (c + kGemvStages) * (kGemvChunk / 2), row0, bars + 8 * st);
      }
      ++issued;
    }
  }
  // drain: no copy may still be landing when the CTA exits
  if (lane == 0) {
    for (int i = max(0, issued - kGemvStages); i < issued; ++i)
      mbar_wait_drain(bars + 8 * (i % kGemvStages), (i / kGemvStages) & 1);
  }

  // fixed-order reduction over the warps of the CTA
#pragma unroll
  for (int r = 0; r < kGemvR; ++r)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s_red[(((warp * kGemvR + r) * NT + nt) * 4 + i) * 32 + lane] = acc[r][nt][i];
  __syncthreads();
  for (int item = warp; item < kGemvR * NT * 4; item += nwarps) {
    const int i = item & 3, nt = (item >> 2) % NT, r = (item >> 2) / NT;
    float v = 0.f;
    for (int w = 0; w < nwarps; ++w) v += s_red[(((w * kGemvR + r) * NT + nt) * 4 + i) * 32 + lane];
    // d0,d1: row g, cols 2t, 2t+1; d2,d3: row g+8
    const int row = row0 + 16 * r + g + (i < 2 ? 0 : 8);
    const int col = 8 * nt + 2 * t + (i & 1);
    if (row < N && col < M) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      y[static_cast<int64_t>(col) * N + row] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

inline size_t gemv_smem_bytes(int warps, int NT) {
  return 1024 + static_cast<size_t>(warps) * (kGemvStages * kGemvTileBytes + 64) +
         static_cast<size_t>(warps) * kGemvR * NT * 4 * 32 * sizeof(float);
}

}  // namespace nf4q
