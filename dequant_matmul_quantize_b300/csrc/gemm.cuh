// nf4_gemm: Y [M x N] = X [M x K] . w_hat^T on the 5th-generation tensor
// cores ("bitsandbytes tutorial", sec. 3.4: the 4-bit weight is dequantized
// to bf16 and an ordinary bf16 matmul with fp32 accumulation follows).
//
// One CTA computes a 256 x BN tile of Y as two 128 x BN halves that share
// every dequantized W tile (so each weight is rebuilt once per 256 rows of
// X), with tcgen05.mma (kind::f16, bf16 operands, two fp32 accumulators in
// tensor memory), K in steps of 64:
//   warp 0      TMA producer: the two X tiles (128 x 64 bf16 each, 128-byte
//               swizzle) and the packed W tile (BN rows x 32 bytes, 32-byte
//               swizzle) of a stage, one mbarrier with the byte count.
//   warp 1      allocates 512 TMEM columns; one lane issues the 2 x 4
//               128xBNx16 MMAs of a stage and commits them to the stage's
//               "empty" barrier, after the last stage to "acc_full".
//   warps 2..17 dequantize, as two groups of 8 warps taking alternate
//               k-steps (one group alone cannot keep the ALUs busy): thread
//               r of a group rebuilds row r of the W tile with the register
//               byte tables of lut.cuh (bit-exact w_hat) into the K-major
//               128-byte-swizzled layout the MMA reads, then
//               fence.proxy.async and arrive on the stage's "b_full".
//               Afterwards the 16 warps drain the two accumulators
//               (tcgen05.ld), round to bf16 and store Y.
// BN (128..256) is picked per shape so the tile count fills whole waves of
// the SMs.  For M <= 128 a CTA has one accumulator (128 x 128 tiles) and,
// with X stages half the size, an 8-stage TMA ring.  Every wait is bounded (1 s of %globaltimer); a wait that gives up
// sets bit 0 of the device error word and the CTA winds down: its other
// waits stop, its TMA copies and MMAs are drained (bounded), its TMEM freed.
// No multicast: every CTA loads its own tiles.
//
// Split K (M <= 128 with fewer 128 x 128 tiles than SMs): a thread-block
// cluster of S <= 4 CTAs shares one tile, CTA r taking k-steps
// [r KT / S, (r + 1) KT / S).  After a cluster barrier (every CTA's main
// loop has finished, so rank 0's rings are idle) ranks 1 .. S-1 write their
// fp32 accumulators into rank 0's shared memory (distributed shared memory,
// 128 x 128 floats each, 16-byte chunks swizzled by row); after a second
// barrier rank 0 adds them in rank order to its own and stores Y, so the
// result is deterministic.
#pragma once

#include <mutex>

#include "common.cuh"
#include "host.h"
#include "lut.cuh"
#include "tma.cuh"

namespace nf4q {

constexpr int kGemmBM = 128;   // rows per accumulator (two per CTA)
constexpr int kGemmBK = 64;
constexpr int kGemmATile = kGemmBM * kGemmBK * 2;    // 16 KB
constexpr int kGemmTmemCols = 512;

// MT = X tiles (128-row accumulators) per CTA: 2, or 1 for M <= 128, where
// the smaller TMA stages leave room for a deeper ring.
template <int BN, int MT = 2>
struct GemmCfg {
  static constexpr int kBTile = BN * kGemmBK * 2;     // bf16 W tile
  static constexpr int kPTile = BN * kGemmBK / 2;     // packed W tile (bytes the TMA moves)
  static constexpr int kPSlot = (kPTile + 1023) / 1024 * 1024;  // its room in a stage
  static constexpr int kAStages =                     // TMA stages: MT X tiles + packed W
      MT == 2 ? 4 : (BN <= 128 ? 8 : 6);
  static constexpr int kAStage = MT * kGemmATile + kPSlot;
  static constexpr int kBStages =                     // dequantized W stages
      (kAStages * kAStage + 3 * kBTile + 2048 <= 232448 - 1024) ? 3 : 2;
  static constexpr size_t kSmem = 1024 + kAStages * kAStage + kBStages * kBTile + 1024;
  // One group of 8 dequant warps per B stage: group g produces the k-steps
  // kt % kBStages == g, always into stage g, so no producer can run more than
  // one mbarrier phase ahead of the MMA on its stage.
  static constexpr int kGroups = kBStages;
  static constexpr int kThreads = 64 + kGroups * 256;   // + TMA warp and MMA warp
  static_assert(kPTile % 256 == 0 && kBTile % 1024 == 0, "tile alignment (swizzle atoms)");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(MT == 1 || MT == 2, "one or two accumulators");
};

// Scale inputs of one W row for 16 consecutive k-steps (64-blocks): the 16
// absmax_q bytes (or fp32 absmax) and their scale2, loaded a group ahead.
struct ScaleGroup {
  uint4 q;          // 16 int8 codes of the scales
  float s2a, s2b;   // scale2 of the first block and of the block after the
  int split;        // first k-step (0..16) whose block uses s2b
};

// K-major operand in the 128-byte swizzled layout: rows of 128 bytes, 8-row
// groups 1024 bytes apart.  Shared-memory matrix descriptor fields: start
// address >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused for
// swizzled K-major, set to 1), stride byte offset >> 4 (32-45), the fixed
// value 1 in bits 46-47, swizzle mode 2 = 128-byte in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, A and
// B both bf16 (DT 0) or both fp16 (DT 1), K-major, N >> 3 and M >> 4.
template <int DT>
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4) | ((DT == 0 ? 1u : 0u) << 7) | ((DT == 0 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Epilogue of a CTA's 256 x BN tile: warps 2..17 drain the two fp32
// accumulators (warp w reads TMEM lane quarter w % 4 - the only one it may
// access - of accumulator ((w - 2) / 4) % 2, every other 32-column chunk
// from ((w - 2) / 8) * 32), round to the compute dtype and store rows
// m0 .. m0 + 255 (< M) and columns c0 .. c0 + BN - 1 (< ncols) of the
// row-major Y [M x ncols].
template <int BN, int DT, int MT = 2>
__device__ __forceinline__ void store_accumulators(uint32_t tmem, int warp, int lane,
                                                   uint16_t* __restrict__ Y, int M, int ncols,
                                                   int m0, int c0) {
  const int q = warp & 3;
  const int h = ((warp - 2) >> 2) & 1;
  if (h >= MT) return;  // a CTA with one accumulator owns only its first 128 rows
  const int cc = ((warp - 2) >> 3) * 32;
  const int m = m0 + h * kGemmBM + q * 32 + lane;
  uint16_t* yrow = Y + static_cast<int64_t>(m) * ncols + c0;
  const bool vec = (ncols & 7) == 0;
#pragma unroll 1
  for (int col = cc; col < BN; col += 64) {
    uint32_t v[32];
    tmem_ld32(tmem + h * 256 + (static_cast<uint32_t>(q * 32) << 16) + col, v);
    if (m < M) {
      const int n = min(min(32, BN - col), ncols - (c0 + col));
      if (n == 32 && vec) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 o;
          o.x = pack_x2<DT>(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
          o.y = pack_x2<DT>(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
          o.z = pack_x2<DT>(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
          o.w = pack_x2<DT>(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
          *reinterpret_cast<uint4*>(yrow + col + 8 * j) = o;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < n) yrow[col + j] = round_to_dt<DT>(__uint_as_float(v[j]));
        }
      }
    }
  }
}

// Split-K partials: rank p (1 .. S-1) of a cluster writes its 128 x BN fp32
// accumulator to rank 0's shared memory at base + (p - 1) * 128 * BN * 4,
// row-major, the 16-byte chunk c of row r at chunk c ^ (r & 7).  Warp w
// (2 .. 17) takes TMEM lane quarter w % 4 (the one it may access) and the
// 32-column chunks from ((w - 2) / 8) * 32 in steps of 64; warps with
// ((w - 2) / 4) odd have no second accumulator to drain (one per CTA here).
__device__ __forceinline__ uint32_t split_partial_addr(uint32_t base, int bn, int p, int r,
                                                       int col) {
  return base + static_cast<uint32_t>((p - 1) * 128 * bn * 4 + r * bn * 4) +
         static_cast<uint32_t>((((col >> 2) ^ (r & 7)) << 4) + (col & 3) * 4);
}

// With mt accumulators per CTA (dX), rank r's accumulator a goes to partial
// region (r - 1) mt + a + 1.
template <int BN>
__device__ __forceinline__ void send_partials(uint32_t tmem, int warp, int lane, uint32_t base,
                                              uint32_t rank, int acc = 0, int mt = 1) {
  static_assert(BN % 32 == 0, "split K runs with whole 32-column chunks");
  const int q = warp & 3;
  if ((((warp - 2) >> 2) & 1) != 0) return;
  const int cc = ((warp - 2) >> 3) * 32;
  const int r = q * 32 + lane;
#pragma unroll 1
  for (int col = cc; col < BN; col += 64) {
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + col, v);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t local =
          split_partial_addr(base, BN, (static_cast<int>(rank) - 1) * mt + acc + 1, r, col + 4 * c);
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(local));
      asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(remote),
                   "r"(v[4 * c]), "r"(v[4 * c + 1]), "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                   : "memory");
    }
  }
}

// Rank 0: its accumulator plus ranks 1 .. S-1 in order, rounded and stored
// as store_accumulators does for rows m0 .. m0 + 127.
template <int BN, int DT>
__device__ __forceinline__ void store_split_sum(uint32_t tmem, int warp, int lane, uint32_t base,
                                                int S, uint16_t* __restrict__ Y, int M, int ncols,
                                                int m0, int c0, int acc = 0, int mt = 1) {
  const int q = warp & 3;
  if ((((warp - 2) >> 2) & 1) != 0) return;
  const int cc = ((warp - 2) >> 3) * 32;
  const int r = q * 32 + lane;
  const int m = m0 + r;
  uint16_t* yrow = Y + static_cast<int64_t>(m) * ncols + c0;
  const bool vec = (ncols & 7) == 0;
#pragma unroll 1
  for (int col = cc; col < BN; col += 64) {
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + col, v);
    for (int p = 1; p < S; ++p) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(split_partial_addr(base, BN, (p - 1) * mt + acc + 1, r, col + 4 * c))
                     : "memory");
        v[4 * c] = __float_as_uint(__uint_as_float(v[4 * c]) + __uint_as_float(w.x));
        v[4 * c + 1] = __float_as_uint(__uint_as_float(v[4 * c + 1]) + __uint_as_float(w.y));
        v[4 * c + 2] = __float_as_uint(__uint_as_float(v[4 * c + 2]) + __uint_as_float(w.z));
        v[4 * c + 3] = __float_as_uint(__uint_as_float(v[4 * c + 3]) + __uint_as_float(w.w));
      }
    }
    if (m < M) {
      const int n = min(32, ncols - (c0 + col));
      if (n == 32 && vec) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 o;
          o.x = pack_x2<DT>(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
          o.y = pack_x2<DT>(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
          o.z = pack_x2<DT>(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
          o.w = pack_x2<DT>(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
          *reinterpret_cast<uint4*>(yrow + col + 8 * j) = o;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < n) yrow[col + j] = round_to_dt<DT>(__uint_as_float(v[j]));
        }
      }
    }
  }
}

// ------------------------------------------------------------ the kernel
template <int CODE, int BN, int DT, int MT>
__global__ void __launch_bounds__(GemmCfg<BN, MT>::kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
            const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
            uint16_t* __restrict__ Y, int M, int N, int K,
            const __grid_constant__ CodeValues C) {
  using Cfg = GemmCfg<BN, MT>;
  constexpr int SA = Cfg::kAStages, SB = Cfg::kBStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sA = [&](int s, int h) { return base + s * Cfg::kAStage + h * kGemmATile; };
  auto sP = [&](int s) { return base + s * Cfg::kAStage + MT * kGemmATile; };
  auto sB = [&](int s) { return base + SA * Cfg::kAStage + s * Cfg::kBTile; };
  const uint32_t sBar = base + SA * Cfg::kAStage + SB * Cfg::kBTile;   // 1 KB of barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sBar - base) + 512);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(gbase + (sBar - base) + 516);
  // full: TMA landed; aempty: MMA done with the TMA slot;
  // bfull: dequantized tile written; bempty: MMA done with the B slot
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto aempty_bar = [&](int s) { return sBar + 8u * (SA + s); };
  auto bfull_bar = [&](int s) { return sBar + 8u * (2 * SA + s); };
  auto bempty_bar = [&](int s) { return sBar + 8u * (2 * SA + SB + s); };
  const uint32_t acc_bar = sBar + 8u * (2 * SA + 2 * SB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * (MT * kGemmBM);
  const int KT = K / kGemmBK;
  // split K: this CTA's k-steps kb .. kb + KTl - 1 (the whole range without a split)
  const int S = static_cast<int>(gridDim.z);
  uint32_t rank = 0;
  if (S > 1) asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int kb = static_cast<int>(rank) * KT / S;
  const int KTl = (static_cast<int>(rank) + 1) * KT / S - kb;

  if (threadIdx.x == 0) {
    *abort = 0u;
    for (int s = 0; s < SA; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(aempty_bar(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bfull_bar(s), 8);
      mbar_init(bempty_bar(s), 1);
    }
    mbar_init(acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kGemmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
      int issued = 0;
      for (int i = 0; i < KTl; ++i) {
        const int kt = kb + i;
        const int s = i % SA;
        const uint32_t ph = (i / SA) & 1;
        if (!mbar_wait(aempty_bar(s), ph ^ 1, abort)) break;
        mbar_arrive_expect_tx(full_bar(s), MT * kGemmATile + Cfg::kPTile);
        tma_load_2d(sA(s, 0), &tmap_x, kt * kGemmBK, m0, full_bar(s));
        if (MT == 2) tma_load_2d(sA(s, 1), &tmap_x, kt * kGemmBK, m0 + kGemmBM, full_bar(s));
        tma_load_2d(sP(s), &tmap_w, kt * (kGemmBK / 2), n0, full_bar(s));
        issued = i + 1;
      }
      // wind-down: make sure no copy is still landing in this CTA's smem
      for (int i = (issued > SA ? issued - SA : 0); i < issued; ++i)
        mbar_wait_drain(full_bar(i % SA), (i / SA) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<DT>(kGemmBM, BN);
      for (int i = 0; i < KTl; ++i) {
        const int sa = i % SA, sb = i % SB;
        if (!mbar_wait(full_bar(sa), (i / SA) & 1, abort)) break;
        if (!mbar_wait(bfull_bar(sb), (i / SB) & 1, abort)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kGemmBK / 16; ++k) {
          const uint64_t bdesc = smem_desc_sw128(sB(sb) + 32 * k);
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          mma_bf16(tmem, smem_desc_sw128(sA(sa, 0) + 32 * k), bdesc, idesc, acc);
          if (MT == 2) mma_bf16(tmem + 256, smem_desc_sw128(sA(sa, 1) + 32 * k), bdesc, idesc, acc);
        }
        mma_commit(aempty_bar(sa));
        mma_commit(bempty_bar(sb));
      }
      mma_commit(acc_bar);  // fires once every MMA issued above has completed
    }
  } else {
    // ---------------- dequantize producers: two groups of 8 warps take
    // alternate k-steps; thread r of a group rebuilds W row r
    const int idx = threadIdx.x - 64;
    const int grp = idx >> 8;
    const int r = idx & 255;
    const bool active = r < BN;
    const int n = n0 + r;
    const bool row_ok = active && n < N;
    const int kblocks = K / kBlock;
    const int64_t row_block0 = static_cast<int64_t>(n) * kblocks;
    // scales are read 16 k-steps at a time, one group ahead
    const bool vec_q = sv.double_quant && (kblocks & 15) == 0;
    auto load_group = [&](ScaleGroup& g, int kt0) {
      g.q = make_uint4(0, 0, 0, 0);
      g.s2a = g.s2b = 0.f;
      g.split = 16;
      if (!row_ok || kt0 >= KT || !sv.double_quant) return;
      const int64_t b0 = row_block0 + kt0;
      if (vec_q) {
        g.q = __ldg(reinterpret_cast<const uint4*>(sv.absmax_q + b0));
      } else {
        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t v = kt0 + j < KT
              ? static_cast<uint32_t>(static_cast<uint8_t>(__ldg(sv.absmax_q + b0 + j))) : 0u;
          const uint32_t sh = v << (8 * (j & 3));
          if (j < 4) w0 |= sh; else if (j < 8) w1 |= sh; else if (j < 12) w2 |= sh; else w3 |= sh;
        }
        g.q = make_uint4(w0, w1, w2, w3);
      }
      g.s2a = __ldg(sv.scale2 + (b0 >> 8));
      const int64_t nextd = ((b0 >> 8) + 1) << 8;   // first block of the next 256
      g.split = static_cast<int>(nextd - b0 < 16 ? nextd - b0 : 16);
      if (g.split < 16 && kt0 + g.split < KT) g.s2b = __ldg(sv.scale2 + (nextd >> 8));
    };
    const float off = sv.double_quant ? __ldg(sv.offset) : 0.f;
    ScaleGroup gcur, gnext;
    int g16 = kb & ~15;  // first k-step of the group of 16 in gcur
    load_group(gcur, g16);
    load_group(gnext, g16 + 16);
    for (int i = grp; i < KTl; i += Cfg::kGroups) {
      const int kt = kb + i;
      const int sa = i % SA, sb = i % SB;
      const int j = kt & 15;
      if ((kt & ~15) != g16) {  // first k-step of this thread in a new group of 16
        g16 += 16;
        gcur = gnext;
        load_group(gnext, g16 + 16);
      }
      float sc;
      if (sv.double_quant) {
        const uint32_t qw = j < 8 ? (j < 4 ? gcur.q.x : gcur.q.y) : (j < 12 ? gcur.q.z : gcur.q.w);
        const float q = static_cast<float>(static_cast<int8_t>((qw >> (8 * (j & 3))) & 0xFFu));
        sc = __fmaf_rn(q, j < gcur.split ? gcur.s2a : gcur.s2b, off);
      } else {
        sc = row_ok ? __ldg(sv.absmax + row_block0 + kt) : 0.f;
      }
      RowTable<CODE> T;
      build_table<CODE, DT>(T, sc, C);
      // B slot sb is free once the MMAs of the previous round on it are done
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bempty_bar(sb), ((i / SB) & 1) ^ 1, abort) &&
                                       mbar_wait(full_bar(sa), (i / SA) & 1, abort)))
        break;
      if (active) {
        const uint8_t* prow = gbase + (sP(sa) - base) + r * 32;
        const int sw = (r >> 2) & 1;  // 32-byte swizzle of the TMA tile
        const uint4 p0 = *reinterpret_cast<const uint4*>(prow + ((0 ^ sw) << 4));
        const uint4 p1 = *reinterpret_cast<const uint4*>(prow + ((1 ^ sw) << 4));
        const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        uint8_t* brow = gbase + (sB(sb) - base) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // chunk c = elements 8c..8c+7 = packed word c
          uint32_t o[4];
          dequant_word<CODE>(T, words[c], o);
          *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bfull_bar(sb));
    }
    // ---------------- epilogue: TMEM -> bf16 -> Y
    if (S == 1 && warp < 18 && __all_sync(0xFFFFFFFFu, mbar_wait(acc_bar, 0, abort))) {
      tc_fence_after();
      store_accumulators<BN, DT, MT>(tmem, warp, lane, Y, M, N, m0, n0);
    }
  }
  if constexpr (MT == 1 && BN % 32 == 0) {
   if (S > 1) {
    // split K: every thread of the cluster passes both barriers
    __syncwarp();
    const bool epi = warp >= 2 && warp < 18;
    bool ok = true;
    if (epi) ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_bar, 0, abort));
    tc_fence_before();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (epi && ok && rank > 0) {
      tc_fence_after();
      send_partials<BN>(tmem, warp, lane, base, rank);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (epi && ok && rank == 0) {
      tc_fence_after();
      store_split_sum<BN, DT>(tmem, warp, lane, base, S, Y, M, N, m0, n0);
    }
   }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait_drain(acc_bar, 0);  // every MMA of this CTA is done
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kGemmTmemCols)
                 : "memory");
  }
}

// Pick BN so that the number of 256 x BN tiles fills whole waves of the SMs.
// BN for a shape: the candidate with the best (wave efficiency x relative
// rate of a full wave at that BN).  The rates were measured on a B300 at
// M = 2048 and 4096 on a 14336 x 4096 weight (wave rate relative to BN =
// 256): narrow tiles lose more per wave than their better wave fill gains.
inline int gemm_pick_bn(int64_t M, int64_t N, int sms) {
  const int cands[5] = {256, 224, 192, 160, 128};
  const double rate[5] = {1.00, 0.93, 0.93, 0.78, 0.68};
  const int64_t mt = (M + 2 * kGemmBM - 1) / (2 * kGemmBM);
  int best = 256;
  double best_score = -1.0;
  for (int i = 0; i < 5; ++i) {
    const int bn = cands[i];
    const int64_t tiles = mt * ((N + bn - 1) / bn);
    const int64_t rounds = (tiles + sms - 1) / sms;
    // useful columns / columns the rounds could have computed
    const double eff = static_cast<double>(N) * mt / (static_cast<double>(rounds) * sms * bn);
    const double score = eff * rate[i];
    if (score > best_score + 1e-9) { best_score = score; best = bn; }
  }
  return best;
}

// K split of a one-accumulator launch: the largest S <= 4 with S x tiles
// CTAs in one wave, at least 8 k-steps per CTA, and the fp32 partials of
// ranks 1 .. S-1 (partial_bytes each) within rank 0's idle rings
// (room_bytes, everything below the barrier area).
inline int gemm_split_k(int64_t tiles, int64_t kt, int sms, int64_t partial_bytes,
                        int64_t room_bytes) {
  int S = 1;
  while (S < 4 && tiles * (S + 1) <= sms && kt / (S + 1) >= 8 &&
         S * partial_bytes <= room_bytes)
    ++S;
  return S;
}

template <int CODE, int BN, int DT, int MT = 2>
inline nf4q_status gemm_launch_bn(const CUtensorMap& tx, const nf4q_weight* wq, const ScaleView& sv,
                                  const CodeValues& C, int64_t M, void* Y, cudaStream_t stream,
                                  int sms) {
  using Cfg = GemmCfg<BN, MT>;
  const int64_t N = wq->rows, K = wq->cols;
  EncodeTiledFn enc = encode_tiled_fn();
  CUtensorMap tw;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {kGemmBK / 2, BN};
  cuuint32_t es[2] = {1, 1};
  nf4q_status st = cu_check(
      enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq->packed, dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
      "cuTensorMapEncodeTiled (GEMM weight)");
  if (st != NF4Q_OK) return st;
  // Opt in to the kernel's dynamic shared memory, once per device.
  static bool attr_set[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if ((st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) != NF4Q_OK) return st;
  if (dev < 0 || dev >= 64) return NF4Q_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(gemm_kernel<CODE, BN, DT, MT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cfg::kSmem)),
                      "cudaFuncSetAttribute (GEMM)");
      if (st != NF4Q_OK) return st;
      attr_set[dev] = true;
    }
  }
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + MT * kGemmBM - 1) / (MT * kGemmBM));
  const int S = (MT == 1 && BN % 32 == 0)
                    ? gemm_split_k(tiles, K / kGemmBK, sms, int64_t{kGemmBM} * BN * 4,
                                   int64_t{Cfg::kAStages} * Cfg::kAStage +
                                       int64_t{Cfg::kBStages} * Cfg::kBTile)
                    : 1;
  dim3 grid(static_cast<unsigned>((N + BN - 1) / BN),
            static_cast<unsigned>((M + MT * kGemmBM - 1) / (MT * kGemmBM)),
            static_cast<unsigned>(S));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = static_cast<unsigned>(S);
  return launch("gemm_kernel", gemm_kernel<CODE, BN, DT, MT>, grid, dim3(Cfg::kThreads), Cfg::kSmem,
                stream, attr, S > 1 ? 1u : 0u, tx, tw, sv, static_cast<uint16_t*>(Y),
                static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), C);
}

// BN of a one-accumulator launch (128-row tiles, mt of them along M), or 0
// when no width fits one wave.  Each CTA rebuilds BN weight rows per
// k-step, so within one wave the time grows with BN: the smallest candidate
// whose tiles fit the SMs.  Weights narrow enough for the K split (at most
// half the SMs' worth of 128-wide tiles) keep BN = 128 and split.
inline int gemm_pick_bn1(int64_t mt, int64_t N, int sms) {
  if (mt * ((N + 127) / 128) * 2 <= sms) return 128;
  const int cands[6] = {80, 112, 128, 160, 208, 256};
  for (int bn : cands)
    if (mt * ((N + bn - 1) / bn) <= sms) return bn;
  return 0;
}

template <int CODE, int DT>
inline nf4q_status gemm_launch_code(const CUtensorMap& tx, const nf4q_weight* wq,
                                    const ScaleView& sv, const CodeValues& C, int64_t M, void* Y,
                                    cudaStream_t stream, int bn, int sms) {
  // One accumulator per CTA (128-row tiles, with the deeper TMA ring the
  // smaller stages allow, W tiles as narrow as one wave allows) whenever
  // such tiles fit one wave: for M <= 128 always (several waves of 128-wide
  // tiles otherwise), above that while they give more CTAs than 256-row
  // tiles do (M = 256 on a 14336-row weight: 138 CTAs instead of 64)
  const int64_t mt1 = (M + kGemmBM - 1) / kGemmBM;
  const int bn1 = gemm_pick_bn1(mt1, wq->rows, sms);
  if (M <= kGemmBM || bn1 != 0) {
    switch (bn1) {
      case 80: return gemm_launch_bn<CODE, 80, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
      case 112: return gemm_launch_bn<CODE, 112, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
      case 160: return gemm_launch_bn<CODE, 160, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
      case 208: return gemm_launch_bn<CODE, 208, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
      case 256: return gemm_launch_bn<CODE, 256, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
      default: return gemm_launch_bn<CODE, 128, DT, 1>(tx, wq, sv, C, M, Y, stream, sms);
    }
  }
  switch (bn) {
    case 224: return gemm_launch_bn<CODE, 224, DT>(tx, wq, sv, C, M, Y, stream, sms);
    case 192: return gemm_launch_bn<CODE, 192, DT>(tx, wq, sv, C, M, Y, stream, sms);
    case 160: return gemm_launch_bn<CODE, 160, DT>(tx, wq, sv, C, M, Y, stream, sms);
    case 128: return gemm_launch_bn<CODE, 128, DT>(tx, wq, sv, C, M, Y, stream, sms);
    default: return gemm_launch_bn<CODE, 256, DT>(tx, wq, sv, C, M, Y, stream, sms);
  }
}

inline nf4q_status gemm_launch(const nf4q_weight* wq, const ScaleView& sv,
                               const CodeValues& C, const void* X, int64_t M, void* Y,
                               cudaStream_t stream, int sms) {
  const int64_t N = wq->rows, K = wq->cols;
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NF4Q_ERR_UNSUPPORTED;
  if ((M + 2 * kGemmBM - 1) / (2 * kGemmBM) > 65535) return NF4Q_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled: driver entry point not found");
  if (ensure_context() != NF4Q_OK) return NF4Q_ERR_CUDA;
  CUtensorMap tx;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {kGemmBK, kGemmBM};
  cuuint32_t es[2] = {1, 1};
  const int dt = wq->compute_dtype;
  const nf4q_status st = cu_check(
      enc(&tx, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
          const_cast<void*>(X), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
      "cuTensorMapEncodeTiled (GEMM activations)");
  if (st != NF4Q_OK) return st;
  const int bn = gemm_pick_bn(M, N, sms);
  if (dt == 0)
    return wq->code == 0 ? gemm_launch_code<0, 0>(tx, wq, sv, C, M, Y, stream, bn, sms)
                         : gemm_launch_code<1, 0>(tx, wq, sv, C, M, Y, stream, bn, sms);
  return wq->code == 0 ? gemm_launch_code<0, 1>(tx, wq, sv, C, M, Y, stream, bn, sms)
                       : gemm_launch_code<1, 1>(tx, wq, sv, C, M, Y, stream, bn, sms);
}

}  // namespace nf4q
