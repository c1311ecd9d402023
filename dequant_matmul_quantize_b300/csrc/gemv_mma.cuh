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

constexpr int kGemvStages = 4;
constexpr int kGemvTileBytes = kGemvRows * (kGemvChunk / 2);  // 16 rows x 128 B

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

// Raw scale inputs of rows g and g+8 for one chunk (prefetched a chunk ahead).
struct ScaleLoad {
  float qa, qb, s2a, s2b;
};

__device__ __forceinline__ void load_scales(ScaleLoad& L, const ScaleView& sv, int rA, int rB,
                                            int N, int kblocks, int blk) {
  L.qa = L.qb = L.s2a = L.s2b = 0.f;
  if (blk >= kblocks) return;
  if (rA < N) {
    const int64_t b = static_cast<int64_t>(rA) * kblocks + blk;
    if (sv.double_quant) {
      L.qa = static_cast<float>(__ldg(sv.absmax_q + b));
      L.s2a = __ldg(sv.scale2 + (b >> 8));
    } else {
      L.qa = __ldg(sv.absmax + b);
    }
  }
  if (rB < N) {
    const int64_t b = static_cast<int64_t>(rB) * kblocks + blk;
    if (sv.double_quant) {
      L.qb = static_cast<float>(__ldg(sv.absmax_q + b));
      L.s2b = __ldg(sv.scale2 + (b >> 8));
    } else {
      L.qb = __ldg(sv.absmax + b);
    }
  }
}

// Each warp streams its own K range of the CTA's 16 rows through a private
// ring of kGemvStages shared-memory tiles (16 rows x 128 packed bytes = 256
// columns), filled by TMA (128-byte swizzle, so the 8 rows a lane group
// reads land in distinct banks) and tracked by one mbarrier per stage.
template <int CODE, int NT>
__global__ void __launch_bounds__(512)
gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
                const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int N, int K, int M,
                int per_warp, const __grid_constant__ CodeValues C) {
  extern __shared__ __align__(1024) uint8_t gsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * kGemvRows;
  const int rA = row0 + g, rB = row0 + g + 8;
  const int nchunks = (K + kGemvChunk - 1) / kGemvChunk;
  const int c_begin = warp * per_warp;
  const int c_end = min(nchunks, c_begin + per_warp);
  const int kblocks = K / kBlock;
  const float off = sv.double_quant ? __ldg(sv.offset) : 0.f;

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

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

  ScaleLoad sc;
  load_scales(sc, sv, rA, rB, N, kblocks, c_begin * 4 + t);
  const int nmine = max(0, c_end - c_begin);
  int issued = min(nmine, kGemvStages);  // TMA loads issued by this warp
  for (int c = c_begin; c < c_end; ++c) {
    const int i = c - c_begin, st = i % kGemvStages;
    const uint32_t ph = (i / kGemvStages) & 1;
    const int blk = c * 4 + t;
    const bool bok = blk < kblocks;
    const float sA = sv.double_quant ? __fmaf_rn(sc.qa, sc.s2a, off) : sc.qa;
    const float sB = sv.double_quant ? __fmaf_rn(sc.qb, sc.s2b, off) : sc.qb;
    if (c + 1 < c_end) load_scales(sc, sv, rA, rB, N, kblocks, blk + 4);
    RowTable<CODE> TA, TB;
    build_table<CODE>(TA, sA, C);
    build_table<CODE>(TB, sB, C);
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_timed(bars + 8 * st, ph))) break;
    const uint32_t tile = ring + st * kGemvTileBytes;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      // 16-byte chunk (2t + hb) of rows g and g + 8, 128-byte swizzle
      const uint32_t chunk = ((2 * t + hb) ^ g) << 4;
      const uint4 pa = lds128(tile + g * 128 + chunk);
      const uint4 pb = lds128(tile + (g + 8) * 128 + chunk);
      const uint32_t wa[4] = {pa.x, pa.y, pa.z, pa.w};
      const uint32_t wb[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int wi = 4 * hb + q;  // word of the block: elements 8wi .. 8wi+7
        uint32_t xb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = g + 8 * nt;
          if (bok && col < M) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                x + static_cast<int64_t>(col) * K + blk * 64 + wi * 8));
            xb[nt][0] = v.x; xb[nt][1] = v.y; xb[nt][2] = v.z; xb[nt][3] = v.w;
          } else {
            xb[nt][0] = xb[nt][1] = xb[nt][2] = xb[nt][3] = 0u;
          }
        }
        uint32_t ra[4], rb[4];
        dequant_word<CODE>(TA, wa[q], ra);
        dequant_word<CODE>(TB, wb[q], rb);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16_16816(acc[nt], ra[2 * h], rb[2 * h], ra[2 * h + 1], rb[2 * h + 1],
                           xb[nt][2 * h], xb[nt][2 * h + 1]);
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
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s_red[((warp * NT + nt) * 4 + i) * 32 + lane] = acc[nt][i];
  __syncthreads();
  for (int item = warp; item < NT * 4; item += nwarps) {
    const int i = item & 3, nt = item >> 2;
    float v = 0.f;
    for (int w = 0; w < nwarps; ++w) v += s_red[((w * NT + nt) * 4 + i) * 32 + lane];
    // d0,d1: row g, cols 2t, 2t+1; d2,d3: row g+8
    const int row = i < 2 ? rA : rB;
    const int col = 8 * nt + 2 * t + (i & 1);
    if (row < N && col < M) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      y[static_cast<int64_t>(col) * N + row] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

inline size_t gemv_smem_bytes(int warps, int NT) {
  return 1024 + static_cast<size_t>(warps) * (kGemvStages * kGemvTileBytes + 64) +
         static_cast<size_t>(warps) * NT * 4 * 32 * sizeof(float);
}

}  // namespace nf4q
