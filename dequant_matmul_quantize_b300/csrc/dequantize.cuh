// nf4_dequantize: packed 4-bit codes + (double-quantized) block scales ->
// the compute dtype, bf16 or fp16 ("bitsandbytes tutorial", sec. 3.4: weights
// kept in 4 bits are turned back into the 16-bit compute dtype before the
// matmul; sec. 四: bnb_4bit_compute_dtype).
//
// w_hat = round(fp32(code_value[code] * s_b)) to the compute dtype.  One lane owns one 64-block:
// it reads the block's 32 packed bytes and its scale, builds the 16 values
// w_hat_j of the block once as register byte tables (the GEMV's lookup,
// lut.cuh), and turns each 32-bit word of codes into four bf16x2 registers
// with byte permutes - about three instructions per weight, against the
// HBM budget of roughly fourteen.  A warp's 32 blocks (4 KB of bf16) go to a
// shared-memory tile laid out with the 128-byte swizzle (so the 16-byte
// stores of eight consecutive lanes hit distinct banks), and one TMA store
// writes the tile out; two tiles per warp alternate so the store of one
// overlaps the work on the next.
#pragma once

#include "common.cuh"
#include "lut.cuh"
#include "tma.cuh"

namespace nf4q {

constexpr int kDequantWarps = 8;
constexpr int kDequantThreads = kDequantWarps * 32;
constexpr uint32_t kDequantTileBytes = 32 * kBlock * 2;  // 32 blocks of bf16
constexpr size_t kDequantSmemBytes = 1024 + 2 * kDequantWarps * kDequantTileBytes;
constexpr int kDequantCtasPerSm = 3;  // 65 KB of staging each

// Output tensor map: [n_blocks rows][64 bf16], box {64, 32}, 128-byte swizzle.
template <int CODE, int DT>
__global__ void __launch_bounds__(kDequantThreads)
dequantize_kernel(const uint4* __restrict__ packed, ScaleView sv,
                  const __grid_constant__ CUtensorMap tmap_out, int64_t n_blocks,
                  const __grid_constant__ CodeValues C) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
  const uint32_t bufs = base + warp * 2 * kDequantTileBytes;
  const int64_t n_tiles = (n_blocks + 31) / 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kDequantWarps;
  int parity = 0;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * kDequantWarps + warp; tile < n_tiles;
       tile += nwarps, parity ^= 1) {
    const int64_t b = tile * 32 + lane;
    uint4 p0 = make_uint4(0u, 0u, 0u, 0u), p1 = p0;
    float s = 0.f;
    if (b < n_blocks) {
      p0 = ld_stream_u4(packed + 2 * b);
      p1 = ld_stream_u4(packed + 2 * b + 1);
      s = block_scale(sv, b);
    }
    RowTable<CODE> T;
    build_table<CODE, DT>(T, s, C);
    const uint32_t buf = bufs + parity * kDequantTileBytes;
    // the store issued from this buffer two tiles ago must have read it
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    const uint32_t row = buf + lane * 128;
    const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t r[4];
      dequant_word<CODE>(T, words[k], r);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((k ^ (lane & 7)) << 4)),
                   "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&tmap_out, buf, 0, static_cast<int>(tile * 32));
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait_all();
}

}  // namespace nf4q
