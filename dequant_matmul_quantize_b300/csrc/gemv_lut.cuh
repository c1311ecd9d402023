// nf4_gemv for decode shapes, block-scale folded ("bitsandbytes tutorial",
// sec. 3.4: 4-bit storage, 16-bit compute; sec. 七 myth 5: decode is bound by
// moving the packed weights):
//
//   y[m, n] = sum_b  s_{n,b} * sum_{k in b} x[m, k] * c[code(n, k)]
//
// with c the 16 code values and s_{n,b} the scale of 64-block b of row n.
// The inner sum runs on the tensor cores (mma.sync m16n8k16, fp16 operands,
// fp32 accumulate) with the code VALUES as the A operand - the same table
// for every block - and the block scale is applied to each block's fp32
// partial sum afterwards.  So the per-weight work is only a table lookup,
// with no per-block table to build:
//
//   * A byte of packed codes holds two neighbouring weights; the lookup
//     takes the whole byte: a 256-entry table in shared memory gives the
//     fp16x2 pair (c[hi nibble], c[lo nibble]), which is exactly one
//     A-fragment register.  The table is replicated 32 times so that lane l
//     always reads bank l (no conflicts whatever the codes); entry v of
//     replica l sits at 0x10000 + 256 v + 4 l, so a single byte permute
//     (PRMT) forms the address from the packed word and a per-lane constant.
//   * x becomes fp16: for a bf16 compute dtype each row m of x is scaled by
//     a power of two 2^-F_m (F_m from the row's largest |x|) so that every
//     value keeps its 8 significant bits; the factor 2^F_m is folded back
//     together with the block scale.
//
// What this computes differs from the dequantize-then-multiply reference
// only by rounding: the reference multiplies x by w_hat = bf16(c * s), this
// kernel by c * s with c rounded to fp16 (relative error below 3.3e-4 for
// the NF4 and FP4 values, 2^-11 at most for any value).  Per term the
// difference is at most 2^-8 + 2^-11 of |x * w_hat| for bf16 and 2^-10 for
// fp16; it has the sign of the rounding of each w_hat and so averages out
// over a dot product.  (The bit-faithful variant, which rebuilds w_hat
// exactly inside the contraction, is gemv_mma.cuh.)
//
// Work split.  One CTA per SM (the table takes 64 KB), 16 warps, each with
// its own TMA ring of boxes of 16 rows x BB 64-blocks of packed codes (BB = 8:
// two 2 KB boxes per stage, two stages; BB = 4: one box, three stages; the
// 128-byte swizzle).  Each CTA takes a contiguous range of 16-row tiles (the
// ranges differ by at most one tile), and its boxes, in row-major order over
// those tiles, are cut into equal contiguous runs, one per warp: every warp
// streams ceil or floor of the CTA's boxes / 16, with no barrier between
// warps.  A tile whose boxes fall to several warps is finished by the last
// of them to arrive (a shared-memory counter), which adds the partial sums
// in warp order, so y is deterministic.  One launch may cover up to four
// weights that share x and K (a group: q, k and v of an attention block;
// gate and up of an MLP): their tiles are numbered one after the other.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace nf4q {

constexpr int kLutWarps = 16;
constexpr int kLutThreads = kLutWarps * 32;
constexpr uint32_t kLutBoxBytes = 16 * 128;   // one TMA box: 16 rows x 256 packed columns
constexpr uint32_t kLutTable = 0x10000;       // shared address of the table
constexpr uint32_t kLutRing = 0x20000;        // shared address of the rings
constexpr uint32_t kLutSmemTop = 0x38000;     // end of the layout
constexpr uint32_t kLutMaxBase = 0x1000;      // dynamic shared memory must start below
constexpr uint32_t kLutRing8Low = 0x8000;     // BB = 8: the rings' last 32 KB
// Shared memory for staged x: [kLutMaxBase, kLutTable) with BB = 4,
// [kLutMaxBase, kLutRing8Low) with BB = 8.
constexpr uint32_t kLutXBytes4 = kLutTable - kLutMaxBase;
constexpr uint32_t kLutXBytes8 = kLutRing8Low - kLutMaxBase;
constexpr int kLutMaxM = 8;
constexpr int kLutMaxGroup = 4;

template <int BB>
struct LutCfg {
  static constexpr int kStages = BB == 8 ? 2 : 3;
  static constexpr uint32_t kStageBytes = (BB / 4) * kLutBoxBytes;
  static_assert(BB == 4 || BB == 8, "4 or 8 blocks per box");
  static_assert(kLutWarps * kStages * kStageBytes ==
                    (BB == 8 ? (kLutSmemTop - kLutRing) + (kLutTable - kLutRing8Low)
                             : kLutSmemTop - kLutRing),
                "ring layout");
};

// The unused upper half of each 256-byte table row is a 128-byte "piece";
// pieces hold the control data.
__device__ __forceinline__ uint32_t lut_piece(int p) { return kLutTable + 256u * p + 128u; }
constexpr int kLutPieceBars = 0;    // per warp 32 B (up to 3 stages x 8 B)     (4 pieces)
constexpr int kLutPieceScale = 4;   // per warp BB * 16 floats (BB / 2 pieces)  (<= 64)
constexpr int kLutPieceRed = 68;    // per warp 2 partial-sum slots x 512 B     (128 pieces)
// Chunk mode (M = 1, 8-block boxes, chunked scales): per warp a 16-block
// scale slot (8 pieces, pieces 4 .. 131) and 2 partial-sum slots of 64 B
// (one piece, 132 .. 147)
constexpr int kLutPieceRedCm = 132;
constexpr int kLutPieceMisc = 196;  // F factors, tile counters, scratch       (5 pieces)

// fp16 bits of the 16 code values, built on the host.
struct __align__(16) HalfCodes {
  uint16_t h[16];
};

// The weights of one launch (1 .. 4, same K, code, double quant and compute
// dtype): their tensor maps, scale state, outputs, rows, and the first tile
// of each (16-row tiles numbered over the group; off[count] = all tiles).
struct __align__(64) LutGroup {
  CUtensorMap tmap[kLutMaxGroup];
  ScaleView sv[kLutMaxGroup];
  uint16_t* y[kLutMaxGroup];
  int N[kLutMaxGroup];
  int off[kLutMaxGroup + 1];
  int count;
  int map3d;  // 1: tmap is the 3-D view {128 bytes, rows, 128-byte columns} (K % 256 == 0)
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128_lut(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t prmt_lut(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Bounded wait for a stage, letting the warp sleep inside try_wait (a
// suspend-time hint of 20 us) instead of spinning on issue slots that the
// other warps of the SM need; gives up after the usual time limit.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_device_error, 1u);
      return false;
    }
  }
  return true;
}

// d = A (16x16) . B (16x8) + 0, fp16 operands, fp32 accumulate (first MMA of
// a block) and d += A . B (the others).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory layout of staged x (fp16): row m, 64-block j is a 128-byte
// piece at xbase + (m * kbx + j) * 128; element i of the block sits at byte
// (2 i + 16 m) mod 128, so that the eight rows a quarter-warp reads fall on
// distinct banks.
__device__ __forceinline__ uint32_t lut_x_addr(uint32_t xbase, int kbx, int m, int j, int byte) {
  return xbase + static_cast<uint32_t>((m * kbx + j) * 128) +
         static_cast<uint32_t>((byte + 16 * m) & 127);
}

// Launch: grid = min(SM count, 16-row tiles), 512 threads, kLutSmemTop bytes
// of dynamic shared memory (the layout uses absolute shared addresses and
// checks that the dynamic area starts below kLutMaxBase).  kbx = 64-blocks of
// staged x per row (a multiple of BB, >= K/64).  Requires M <= 8,
// M * kbx * 128 <= the x room of BB, and the run arithmetic within 32 bits
// (checked on the host).  Launched as a programmatic dependent of the
// previous kernel.  early != 0: the caller guarantees that no kernel still
// running when this one starts writes the weights or their scales, so
// their first stages are loaded before the wait for that kernel.
template <int DT, bool DQ, int BB, bool EP, bool M1>
__global__ void __launch_bounds__(kLutThreads, 1)
gemv_lut_kernel(const __grid_constant__ LutGroup G, const uint16_t* __restrict__ x, int K,
                int M_arg, int kbx, const __grid_constant__ HalfCodes hc, int early) {
  const int M = M1 ? 1 : M_arg;  // M1: compiled for a single row of x
  using Cfg = LutCfg<BB>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ __align__(1024) uint8_t lsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t base = smem_u32(lsm);
  if (base > kLutMaxBase) {  // never expected; the layout would not fit
    if (threadIdx.x == 0) atomicOr(&g_device_error, 2u);
    return;
  }
  const uint32_t xbase = kLutMaxBase;
  const int KB = K / kBlock;
  const int nbox = (KB + BB - 1) / BB;
  const int T = G.off[G.count];
  // this CTA's tiles [ct0, ct1); its Bc boxes (tile-major) go to Wc warps,
  // warp w taking boxes [w Bc / Wc, (w + 1) Bc / Wc): one box each when
  // Bc < 16.  (The host keeps T * grid and 16 Bc below 2^31.)
  const int ct0 = static_cast<int>(blockIdx.x) * T / static_cast<int>(gridDim.x);
  const int ct1 = static_cast<int>(blockIdx.x + 1) * T / static_cast<int>(gridDim.x);
  const int Bc = nbox > 0 ? (ct1 - ct0) * nbox : 0;
  const int Wc = min(kLutWarps, Bc);
  auto run_start = [&](int w) { return Bc >= kLutWarps ? (w * Bc) >> 4 : w; };
  const int wb0 = warp < Wc ? run_start(warp) : 0;
  const int total = warp < Wc ? run_start(warp + 1) - wb0 : 0;
  const int tile0 = nbox > 0 ? ct0 + wb0 / nbox : ct0;  // first box: (tile0, bx0)
  const int bx0 = wb0 - (tile0 - ct0) * nbox;
  // The tiles this warp may share with others are its first and its last.
  // For each: the first and last warps whose runs reach into it (wf, wl,
  // found by walking from this warp), and wf's slot for it (0 if the tile
  // is wf's first tile), packed as wf | wl << 4 | slot << 8.  All of this
  // reads only the launch parameters, so it runs before the wait for the
  // previous kernel.
  auto share_of = [&](int tile) -> uint32_t {
    const int fb = (tile - ct0) * nbox, lb = fb + nbox - 1;
    int wf = warp, wl = warp;
    while (wf > 0 && run_start(wf) > fb) --wf;
    while (wl + 1 < Wc && run_start(wl + 1) <= lb) ++wl;
    return static_cast<uint32_t>(wf | (wl << 4) | ((run_start(wf) == fb ? 0 : 1) << 8));
  };
  uint32_t share_first = 0, share_last = 0;
  if (total > 0) {
    const int tile_last = tile0 + (bx0 + total - 1) / nbox;
    share_first = share_of(tile0);
    share_last = tile_last == tile0 ? share_first : share_of(tile_last);
  }
  // the weight a (group-wide) tile belongs to
  auto mat_of = [&](int tile) {
    int m = 0;
#pragma unroll
    for (int i = 1; i < kLutMaxGroup; ++i) m += (i < G.count && tile >= G.off[i]) ? 1 : 0;
    return m;
  };

  const uint32_t barw = lut_piece(kLutPieceBars + warp / 4) + 32u * (warp % 4);
  auto bar_of = [&](int st) { return barw + 8u * st; };
  auto stage_addr = [&](int st) -> uint32_t {
    const int i = warp * NS + st;
    if (BB == 4) return kLutRing + static_cast<uint32_t>(i) * Cfg::kStageBytes;
    return i < 24 ? kLutRing + static_cast<uint32_t>(i) * Cfg::kStageBytes
                  : kLutRing8Low + static_cast<uint32_t>(i - 24) * Cfg::kStageBytes;
  };

  // stage st <- box bb (BB blocks) of tile `tile`
  auto issue_at = [&](int tile, int bb, int st) {
    const int m = mat_of(tile);
    const int row0 = (tile - G.off[m]) * 16;
    const uint32_t bar = bar_of(st);
    const uint32_t dst = stage_addr(st);
    mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
    if (G.map3d) {
      tma_load_3d(dst, &G.tmap[m], 0, row0, bb * (BB / 4), bar);
    } else {
#pragma unroll
      for (int h = 0; h < BB / 4; ++h)
        tma_load_2d(dst + h * kLutBoxBytes, &G.tmap[m], (bb * (BB / 4) + h) * 128, row0, bar);
    }
  };

  // Programmatic dependent launch: the next kernel on the stream may start
  // as soon as SMs free up; this one reads no global memory before the
  // kernels it depends on have finished (griddepcontrol.wait below) - it
  // only asks L2 to prefetch.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // 1. barriers
  if (lane == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(bar_of(st), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }

  // 2. the byte-pair table: in pass k thread i writes replicas 4 (i & 7) ..
  //    + 3 of entry 64 k + i / 8, so that each quarter-warp stores one
  //    entry's 128 bytes (all 32 banks)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 64 * k + (threadIdx.x >> 3);
    const uint32_t v = static_cast<uint32_t>(hc.h[e >> 4]) |
                       (static_cast<uint32_t>(hc.h[e & 15]) << 16);
    sts128(kLutTable + 256u * e + 16u * (threadIdx.x & 7), make_uint4(v, v, v, v));
  }

  // stream positions (tile, box): consumer, scale loader (one box ahead),
  // producer (NS boxes ahead, lane 0); each advances one box at a time
  auto advance = [&](int& tile, int& bx) {
    if (++bx == nbox) {
      bx = 0;
      ++tile;
    }
  };

  // The first NS boxes of each warp (unless they are loaded outright below,
  // `early`), and x, go to L2 while the kernels this one depends on finish:
  // an L2 prefetch is safe even if the data were still being written (L2 is
  // the point of coherence).
  if (threadIdx.x == 0) bulk_prefetch_l2(x, static_cast<uint32_t>(M) * K * 2u);
  if (lane == 0 && !early) {
    int f_tile = tile0, f_bx = bx0;
    for (int q = 0; q < min(NS, total); ++q) {
      const int m = mat_of(f_tile);
      if (G.map3d) {
        tma_prefetch_3d(&G.tmap[m], 0, (f_tile - G.off[m]) * 16, f_bx * (BB / 4));
      } else {
#pragma unroll
        for (int h = 0; h < BB / 4; ++h)
          tma_prefetch_2d(&G.tmap[m], (f_bx * (BB / 4) + h) * 128, (f_tile - G.off[m]) * 16);
      }
      advance(f_tile, f_bx);
    }
  }

  // the first NS stage copies of the warp (lane 0)
  int p_tile = tile0, p_bx = bx0;
  auto issue_first = [&]() {
    if (lane == 0) {
      for (int q = 0; q < min(NS, total); ++q) {
        issue_at(p_tile, p_bx, q);
        advance(p_tile, p_bx);
      }
    }
  };

  // Chunked scale loads (EP: double quant with K / 64 a multiple of 16).  A
  // chunk is 16 blocks of the tile's 16 rows; both lanes of row r hold its
  // 16 int8 scale codes (one 16-byte load) and its scale2 (16 blocks
  // aligned to 16 never straddle a 256-block group).  A chunk is loaded one
  // ahead of the one in use, in the order the warp meets them (row-major
  // over its run of boxes); the first two go out with the first stage
  // copies, before x is staged, so that their latency hides behind it.
  const int nch = KB / 16;  // chunks per row
  struct Chunk {
    uint4 q;
    float s2;
  };
  auto chunk_load = [&](int tile, int ci) -> Chunk {
    Chunk c{make_uint4(0, 0, 0, 0), 0.f};
    if (EP && tile < T) {
      const int m = mat_of(tile);
      const int row = (tile - G.off[m]) * 16 + (lane & 15);
      if (row < G.N[m]) {
        const int64_t b0 = static_cast<int64_t>(row) * KB + 16 * ci;
        c.q = __ldg(reinterpret_cast<const uint4*>(G.sv[m].absmax_q + b0));
        c.s2 = __ldg(G.sv[m].scale2 + (b0 >> 8));
      }
    }
    return c;
  };
  auto chunk_next = [&](int& tile, int& ci) {
    if (++ci == nch) {
      ci = 0;
      ++tile;
    }
  };
  Chunk E0{make_uint4(0, 0, 0, 0), 0.f}, E1 = E0;
  int e_tile = tile0, e_ci = (bx0 * BB) / 16;  // next chunk to load
  float offs[kLutMaxGroup];  // the weights' double-quant offsets
  auto load_first = [&]() {
#pragma unroll
    for (int i = 0; i < kLutMaxGroup; ++i)
      offs[i] = (EP && i < G.count) ? __ldg(G.sv[i].offset) : 0.f;
    if (EP && total > 0) {
      E0 = chunk_load(e_tile, e_ci);
      chunk_next(e_tile, e_ci);
      E1 = chunk_load(e_tile, e_ci);
      chunk_next(e_tile, e_ci);
    }
  };
  // M = 1 and at most 16384 staged columns: one read of x, kept in
  // registers (4 x 16 bytes per thread) from the maximum to the conversion.
  const int n8 = K / 8;  // 16-byte groups per row
  const bool x1 = M1 && kbx * 8 <= 4 * kLutThreads;
  uint4 xv[4];
  auto load_x = [&]() {
    if (x1) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = threadIdx.x + r * kLutThreads;
        xv[r] = i < n8 ? __ldg(reinterpret_cast<const uint4*>(x) + i) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  // x is read only after the wait for the kernel this one follows.  By
  // default its loads go out first after the wait, ahead of the weight
  // stream.  `early`: the weights and their scales were written before that
  // kernel began (the caller's guarantee), so their first stages and chunks
  // load while it finishes, and x after it.  (One call site for the stage
  // and chunk loads: two cost registers on the default path.)
  if (!early) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    load_x();
  }
  issue_first();
  load_first();
  if (early) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    load_x();
  }

  // 3. x -> fp16 with a power-of-two scale per row (bf16), staged
  const uint32_t misc = lut_piece(kLutPieceMisc);  // F of each row of x
  // per-warp maxima [16 warps][8 rows] (4 pieces)
  auto fscr_addr = [&](int w, int m) {
    const int i = w * kLutMaxM + m;
    return lut_piece(kLutPieceMisc + 1 + i / 32) + 4u * (i % 32);
  };
  int F1 = 0;  // the F of the single row (x1)
  if (x1) {
    float mx = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t wv[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mx = fmaxf(mx, fmaxf(fabsf(bf16lo_to_f32(wv[k])), fabsf(bf16hi_to_f32(wv[k]))));
    }
    if (DT == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      if (lane == 0) sts32(fscr_addr(warp, 0), __float_as_uint(mx));
      __syncthreads();
      mx = 0.f;
      for (int w = 0; w < kLutWarps; ++w)
        mx = fmaxf(mx, __uint_as_float(lds32(fscr_addr(w, 0))));
      // F = exponent of mx minus 14: mx * 2^-F lies in [2^14, 2^15)
      if (mx > 0.f && mx == mx) {
        const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;
        F1 = max(-126, min(127, e - 14));
      }
      if (threadIdx.x == 0) sts32(misc, static_cast<uint32_t>(F1));
    }
    const float sc = __uint_as_float(static_cast<uint32_t>(127 - F1) << 23);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = threadIdx.x + r * kLutThreads;
      if (i < kbx * 8) {  // 16-byte groups of staged x; past K they are 0
        uint4 out = xv[r];
        if (DT == 0) {
          out.x = pack_f16x2(bf16lo_to_f32(xv[r].x) * sc, bf16hi_to_f32(xv[r].x) * sc);
          out.y = pack_f16x2(bf16lo_to_f32(xv[r].y) * sc, bf16hi_to_f32(xv[r].y) * sc);
          out.z = pack_f16x2(bf16lo_to_f32(xv[r].z) * sc, bf16hi_to_f32(xv[r].z) * sc);
          out.w = pack_f16x2(bf16lo_to_f32(xv[r].w) * sc, bf16hi_to_f32(xv[r].w) * sc);
        }
        sts128(lut_x_addr(xbase, kbx, 0, i >> 3, 16 * (i & 7)), out);
      }
    }
  }
  if (DT == 0 && !x1) {
    for (int m = 0; m < M; ++m) {
      float mx = 0.f;
      for (int i = threadIdx.x; i < n8; i += kLutThreads) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(m) * K) + i);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mx = fmaxf(mx, fmaxf(fabsf(bf16lo_to_f32(wv[k])), fabsf(bf16hi_to_f32(wv[k]))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      if (lane == 0) sts32(fscr_addr(warp, m), __float_as_uint(mx));
    }
  }
  if (!x1) __syncthreads();
  if (DT == 0 && !x1 && threadIdx.x < M) {
    float mx = 0.f;
    for (int w = 0; w < kLutWarps; ++w)
      mx = fmaxf(mx, __uint_as_float(lds32(fscr_addr(w, threadIdx.x))));
    // F = exponent of mx minus 14: mx * 2^-F lies in [2^14, 2^15)
    int F = 0;
    if (mx > 0.f && mx == mx) {
      const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;
      F = max(-126, min(127, e - 14));
    }
    sts32(misc + 4u * threadIdx.x, static_cast<uint32_t>(F));
  }
  if (!x1) __syncthreads();
  if (!x1) {
    // convert / copy: thread -> 8 consecutive values of one row
    const int groups = M * kbx * 8;  // 16-byte groups of staged x
    for (int i = threadIdx.x; i < groups; i += kLutThreads) {
      const int m = i / (kbx * 8), rem = i - m * kbx * 8;
      const int j = rem >> 3, c = rem & 7;  // block j, values 8c .. 8c+7
      const int k0 = j * kBlock + 8 * c;
      uint4 out = make_uint4(0, 0, 0, 0);
      if (k0 < K) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(m) * K + k0));
        if (DT == 0) {
          const int F = static_cast<int>(lds32(misc + 4u * m));
          const float sc = __uint_as_float(static_cast<uint32_t>(127 - F) << 23);
          out.x = pack_f16x2(bf16lo_to_f32(v.x) * sc, bf16hi_to_f32(v.x) * sc);
          out.y = pack_f16x2(bf16lo_to_f32(v.y) * sc, bf16hi_to_f32(v.y) * sc);
          out.z = pack_f16x2(bf16lo_to_f32(v.z) * sc, bf16hi_to_f32(v.z) * sc);
          out.w = pack_f16x2(bf16lo_to_f32(v.w) * sc, bf16hi_to_f32(v.w) * sc);
        } else {
          out = v;
        }
      }
      sts128(lut_x_addr(xbase, kbx, m, j, 16 * c), out);
    }
  }

  // split-tile counters, one per warp (the first warp of the tile), zeroed
  // before the barrier below
  auto tile_ctr = [&](int w) { return misc + 64u + 4u * static_cast<uint32_t>(w); };
  if (threadIdx.x < kLutWarps) sts32(tile_ctr(threadIdx.x), 0u);

  // per-lane fold factors 2^F for its D columns 2t, 2t+1
  float f0 = 0.f, f1 = 0.f;
  {
    const int m0 = 2 * t, m1 = 2 * t + 1;
    if (DT == 0 && x1) {
      if (m0 < M) f0 = __uint_as_float(static_cast<uint32_t>(127 + F1) << 23);
    } else if (DT == 0) {
      if (m0 < M) f0 = __uint_as_float(static_cast<uint32_t>(127 + static_cast<int>(lds32(misc + 4u * m0))) << 23);
      if (m1 < M) f1 = __uint_as_float(static_cast<uint32_t>(127 + static_cast<int>(lds32(misc + 4u * m1))) << 23);
    } else {
      f0 = m0 < M ? 1.f : 0.f;
      f1 = m1 < M ? 1.f : 0.f;
    }
  }
  __syncthreads();  // table and x are complete

  // 4. block scales.  Lane l computes tile row r = l & 15 and the NBL = BB/2
  //    blocks from NBL (l >> 4) of a box and keeps them in the warp's scale
  //    slot (BB / 2 pieces, one per 128-byte line): the scales of 4
  //    consecutive blocks cb of row r are one 16-byte group, group
  //    ((r >> 1) + 4 (r & 1)) mod 8 of line (r & 1) + 2 cb.  So a writer
  //    stores its 4 scales at once (BB = 8; with BB = 4 its 2, the halves of
  //    an odd row's group swapped), and a reader loads the scales of tile
  //    rows 2g and 2g + 1 for 4 blocks with two 16-byte loads - the eight
  //    rows of either parity sit on distinct banks.  With M = 1 the slot
  //    holds s * 2^F of the single row of x.  Without the 16-block chunks
  //    below: with K / 64 a multiple of 4 the codes of a lane's blocks are
  //    one aligned 16- or 32-bit word and share their scale2 (they never
  //    straddle a multiple of 256), otherwise byte loads; the loads run two
  //    boxes ahead of their use.
  constexpr int NBL = BB / 2;
  const int srow = lane & 15, hw = lane >> 4, sjb = NBL * hw;
  const bool kb4 = (KB & 3) == 0;
  struct Raw {
    uint32_t q;       // NBL int8 codes (block j in byte j)
    float s[NBL];     // scale2 of each block (double quant) or its fp32 absmax
    uint32_t okm;     // bit j: block j exists
    float off;        // the weight's double-quant offset
  };
  auto scale_load = [&](int tile, int bb, Raw& r) {
    const int m = mat_of(tile);
    const ScaleView& sv = G.sv[m];
    const int row = (tile - G.off[m]) * 16 + srow;
    const int jb = bb * BB + sjb;
    r.q = 0;
    r.off = 0.f;
#pragma unroll
    for (int j = 0; j < NBL; ++j) r.s[j] = 0.f;
    r.okm = 0;
    if (row < G.N[m]) {
      const int nj = max(0, min(NBL, KB - jb));
      r.okm = (1u << nj) - 1u;
    }
    if (r.okm) {
      const int64_t b0 = static_cast<int64_t>(row) * KB + jb;
      if (DQ) {
        r.off = __ldg(sv.offset);
        if (kb4) {
          if (NBL == 4)
            r.q = __ldg(reinterpret_cast<const uint32_t*>(sv.absmax_q + b0));
          else
            r.q = __ldg(reinterpret_cast<const uint16_t*>(sv.absmax_q + b0));
          const float s2 = __ldg(sv.scale2 + (b0 >> 8));
#pragma unroll
          for (int j = 0; j < NBL; ++j) r.s[j] = s2;
        } else {
#pragma unroll
          for (int j = 0; j < NBL; ++j)
            if ((r.okm >> j) & 1u) {
              r.q |= static_cast<uint32_t>(static_cast<uint8_t>(__ldg(sv.absmax_q + b0 + j)))
                     << (8 * j);
              r.s[j] = __ldg(sv.scale2 + ((b0 + j) >> 8));
            }
        }
      } else {
#pragma unroll
        for (int j = 0; j < NBL; ++j)
          if ((r.okm >> j) & 1u) r.s[j] = __ldg(sv.absmax + b0 + j);
      }
    }
  };
  // chunk mode: the slot holds a whole 16-block chunk, written when a box
  // starts one (every other box), and the partial sums of split tiles are
  // the 8 rows' pairs of the single column
  constexpr bool CM = M1 && EP && BB == 8;
  const uint32_t slot0 = lut_piece(kLutPieceScale + (CM ? 8 : BB / 2) * warp);
  auto slot_group = [](int r) { return static_cast<uint32_t>(((r >> 1) + 4 * (r & 1)) & 7); };
  // where this lane writes its NBL scales
  const uint32_t slot_w =
      slot0 + 256u * static_cast<uint32_t>((srow & 1) + (BB == 8 ? 2 * hw : 0)) +
      16u * slot_group(srow) + (BB == 4 ? 8u * static_cast<uint32_t>(hw ^ (srow & 1)) : 0u);
  auto slot_put = [&](const float (&v)[NBL]) {
    if constexpr (NBL == 4)
      sts128(slot_w, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                __float_as_uint(v[2]), __float_as_uint(v[3])));
    else
      sts64(slot_w, __float_as_uint(v[0]), __float_as_uint(v[1]));
  };
  // with M = 1 the slot holds s * 2^F of row 0 of x (the same for every lane)
  const float fs =
      M != 1 ? 1.f
             : (DT == 0 ? __uint_as_float(static_cast<uint32_t>(127 + static_cast<int>(lds32(misc))) << 23)
                        : 1.f);
  auto scale_store = [&](const Raw& r) {
    float v[NBL];
#pragma unroll
    for (int j = 0; j < NBL; ++j) {
      float sc = 0.f;  // rows past N and blocks past K get scale 0
      if ((r.okm >> j) & 1u)
        sc = DQ ? __fmaf_rn(static_cast<float>(static_cast<int8_t>((r.q >> (8 * j)) & 0xFFu)),
                            r.s[j], r.off)
                : r.s[j];
      v[j] = sc * fs;
    }
    slot_put(v);
  };

  // The factor 2^F (M = 1) is folded into scale2 and the offsets, which is
  // exact: s * 2^F and (q scale2 + offset) 2^F round alike.
#pragma unroll
  for (int i = 0; i < kLutMaxGroup; ++i) offs[i] *= fs;
  float s2c = 0.f, offc = 0.f;  // scale2 * 2^F and offset * 2^F of chunk E0
  auto chunk_use = [&](int tile) {
    float off = offs[0];
#pragma unroll
    for (int i = 1; i < kLutMaxGroup; ++i)
      if (i < G.count && tile >= G.off[i]) off = offs[i];
    offc = off;
    s2c = E0.s2 * fs;
  };
  if (EP && total > 0) chunk_use(tile0);
  auto word_of = [](const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  };
  // scales of box bb of `tile` into the slot, from the chunk registers; a
  // box that starts a chunk moves to the next chunk (except the warp's
  // first box).  An int8 code q becomes a float through the bit pattern
  // 2^23 + (q + 128): exact.
  auto scale_store_ep = [&](int tile, int bb, bool first) {
    if (!first && ((bb * BB) & 15) == 0) {
      E0 = E1;
      E1 = chunk_load(e_tile, e_ci);
      chunk_next(e_tile, e_ci);
      chunk_use(tile);
    }
    const int o = (bb * BB) & 15;  // first block of the box in the chunk
    const uint32_t qw = word_of(E0.q, (o >> 2) + (NBL == 4 ? hw : 0)) ^ 0x80808080u;
    float v[NBL];
#pragma unroll
    for (int j = 0; j < NBL; ++j) {
      const uint32_t sel = 0x7650u + static_cast<uint32_t>(NBL == 4 ? j : 2 * hw + j);
      const float qv = __fsub_rn(__uint_as_float(prmt_lut(qw, 0x4B000000u, sel)), 8388736.f);
      v[j] = __fmaf_rn(qv, s2c, offc);
    }
    slot_put(v);
  };
  // chunk mode: lane (r, h) writes blocks 8h .. 8h + 7 of row r, two 16-byte
  // groups (blocks 4c .. 4c + 3 at line (r & 1) + 2c)
  const uint32_t slot_cm = slot0 + 256u * static_cast<uint32_t>((srow & 1) + 4 * hw) +
                           16u * slot_group(srow);
  auto scale_chunk_cm = [&](int tile, int bb, bool first) {
    if (((bb * BB) & 15) != 0 && !first) return;  // second box of a chunk
    if (!first) {
      E0 = E1;
      E1 = chunk_load(e_tile, e_ci);
      chunk_next(e_tile, e_ci);
      chunk_use(tile);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t qw = (hw ? (c ? E0.q.w : E0.q.z) : (c ? E0.q.y : E0.q.x)) ^ 0x80808080u;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float qv =
            __fsub_rn(__uint_as_float(prmt_lut(qw, 0x4B000000u, 0x7650u + j)), 8388736.f);
        v[j] = __fmaf_rn(qv, s2c, offc);
      }
      sts128(slot_cm + 512u * c, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                           __float_as_uint(v[2]), __float_as_uint(v[3])));
    }
  };

  // 5. per-lane constants.  MMA row g is tile row 2g, MMA row g + 8 is tile
  //    row 2g + 1, so that the four rows a half-warp reads in one load sit
  //    on distinct banks under the 128-byte swizzle: row r's 16-byte chunk c
  //    is at chunk c ^ (r & 7), and this lane's 8 bytes of block j are chunk
  //    2j + (t >> 1), half t & 1.
  const uint32_t SB0 = 256u * g + 32u * (g & 3) + 16u * (t >> 1) + 8u * (t & 1);
  const uint32_t SB1 = (SB0 + 128u) ^ 16u;
  const int mx_row = min(g, M - 1);
  const uint32_t xrow = xbase + static_cast<uint32_t>(mx_row * kbx * 128);
  const uint32_t xo0 = static_cast<uint32_t>((32 * t + 16 * mx_row) & 127);
  const uint32_t xo1 = static_cast<uint32_t>((32 * t + 16 + 16 * mx_row) & 127);
  // table address = [lane * 4, code byte, 0x01, 0]: the table sits at 0x10000
  const uint32_t L = kLutTable | (static_cast<uint32_t>(lane) << 2);
  // the slot groups of tile rows 2g (line 0 + 2 cb) and 2g + 1 (line 1 + 2 cb)
  const uint32_t slot_ra = slot0 + 16u * slot_group(2 * g);
  const uint32_t slot_rb = slot0 + 256u + 16u * slot_group(2 * g + 1);

  // raw scales (without EP): box q + 1 in rA, box q + 2 in rB while box q
  // is consumed
  Raw rA, rB;
  int s_tile = tile0, s_bx = bx0;
  if (EP) {
    if (total > 0) {
      if constexpr (CM)
        scale_chunk_cm(s_tile, s_bx, true);
      else
        scale_store_ep(s_tile, s_bx, true);
      advance(s_tile, s_bx);
    }
  } else {
    if (total > 0) {
      scale_load(s_tile, s_bx, rA);
      scale_store(rA);
      advance(s_tile, s_bx);
    }
    if (total > 1) {
      scale_load(s_tile, s_bx, rA);
      advance(s_tile, s_bx);
    }
    if (total > 2) {
      scale_load(s_tile, s_bx, rB);
      advance(s_tile, s_bx);
    }
  }

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool dead = false;
  int waited_q = -1;  // last box whose stage wait succeeded (waits go in order)
  int issued_n = min(NS, total);
  int c_tile = tile0, c_bx = bx0, u_bx = bx0;  // u_bx: first box of the unit
  int st = 0;
  uint32_t ph = 0;

  for (int q = 0; q < total; ++q) {
    __syncwarp();
    if (!dead) {
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_sleep(bar_of(st), ph));
      if (!ok) dead = true;
      else waited_q = q;
    }
    const uint32_t stage = stage_addr(st);
    const uint32_t w0 = stage + SB0, w1 = stage + SB1;
    const uint32_t xbox = xrow + static_cast<uint32_t>(c_bx * BB * 128);
    uint4 sva = make_uint4(0, 0, 0, 0), svb = sva;  // scales of rows 2g, 2g + 1, 4 blocks
    // unrolled 4 blocks at a time for M = 1 (fewer live registers; ~1 %
    // faster there, ~0.5 % slower at M = 2)
    constexpr int kJUnroll = M1 ? 4 : BB;
#pragma unroll kJUnroll
    for (int j = 0; j < BB; ++j) {
      if ((j & 3) == 0) {
        // chunk mode: the second box of a chunk reads its upper half
        const uint32_t so = 512u * (j >> 2) + (CM ? 1024u * (c_bx & 1) : 0u);
        sva = lds128_lut(slot_ra + so);
        svb = lds128_lut(slot_rb + so);
      }
      const uint32_t hb = kLutBoxBytes * (j >> 2);  // second TMA box of an 8-block stage
      const uint2 wg = lds64((w0 + hb) ^ (32u * (j & 3)));
      const uint2 wh = lds64((w1 + hb) ^ (32u * (j & 3)));
      // x: values 16t .. 16t+15 of block j of row g; lanes whose column
      // g is past M load nothing (their outputs are never stored), so a
      // load moves only the M rows' bytes, and their B registers keep
      // whatever they hold (they feed only D columns that are never read:
      // no zero fill)
      uint4 xa, xb;
      asm("" : "=r"(xa.x), "=r"(xa.y), "=r"(xa.z), "=r"(xa.w), "=r"(xb.x), "=r"(xb.y), "=r"(xb.z),
               "=r"(xb.w));
      if (g < M) {
        xa = lds128_lut(xbox + 128u * j + xo0);
        xb = lds128_lut(xbox + 128u * j + xo1);
      }
      const uint32_t xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const uint32_t wr[2][2] = {{wg.x, wg.y}, {wh.x, wh.y}};
      float d[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // MMA i: bytes 2i, 2i+1 of the lane's 8 bytes (word i / 2, bytes 2(i&1), +1)
        const uint32_t sel0 = 0x7604u | (static_cast<uint32_t>(2 * (i & 1)) << 4);
        const uint32_t sel1 = 0x7604u | (static_cast<uint32_t>(2 * (i & 1) + 1) << 4);
        const uint32_t a0 = lds32(prmt_lut(wr[0][i >> 1], L, sel0));
        const uint32_t a1 = lds32(prmt_lut(wr[1][i >> 1], L, sel0));
        const uint32_t a2 = lds32(prmt_lut(wr[0][i >> 1], L, sel1));
        const uint32_t a3 = lds32(prmt_lut(wr[1][i >> 1], L, sel1));
        if (i == 0)
          mma_f16_first(d, a0, a1, a2, a3, xr[2 * i], xr[2 * i + 1]);
        else
          mma_f16_acc(d, a0, a1, a2, a3, xr[2 * i], xr[2 * i + 1]);
      }
      // s of tile rows 2g and 2g + 1 for block j (BB = 4: an odd row's
      // group holds blocks 2, 3, 0, 1)
      const float sa = __uint_as_float(word_of(sva, j & 3));
      const float sb = __uint_as_float(word_of(svb, BB == 4 ? (j & 3) ^ 2 : (j & 3)));
      // (M > 1: the rows' factors 2^F are applied once, when y is stored)
      acc[0] = __fmaf_rn(d[0], sa, acc[0]);
      acc[2] = __fmaf_rn(d[2], sb, acc[2]);
      if (M != 1) {
        acc[1] = __fmaf_rn(d[1], sa, acc[1]);
        acc[3] = __fmaf_rn(d[3], sb, acc[3]);
      }
    }
    __syncwarp();
    if (lane == 0 && !dead && q + NS < total) {
      fence_proxy_async_smem();
      issue_at(p_tile, p_bx, st);
      advance(p_tile, p_bx);
      ++issued_n;
    }
    // scales of the next box into the slot (every lane is done with this
    // box's); raw loads for box q + 3
    if (q + 1 < total) {
      if (EP) {
        if constexpr (CM)
          scale_chunk_cm(s_tile, s_bx, false);
        else
          scale_store_ep(s_tile, s_bx, false);
        advance(s_tile, s_bx);
      } else {
        scale_store(rA);
        rA = rB;
        if (q + 3 < total) {
          scale_load(s_tile, s_bx, rB);
          advance(s_tile, s_bx);
        }
      }
    }
    if (++st == NS) {
      st = 0;
      ph ^= 1u;
    }
    // end of a unit (the warp's boxes of one tile): a tile the warp covers
    // whole is stored; otherwise the partial sum goes to the warp's slot
    // (0 for the first tile of its run, 1 for the last) and the last of the
    // tile's warps to arrive adds the slots in warp order and stores y
    if (c_bx == nbox - 1 || q == total - 1) {
      const int m = mat_of(c_tile);
      const int Nm = G.N[m];
      uint16_t* __restrict__ ym = G.y[m];
      const int row = (c_tile - G.off[m]) * 16 + 2 * g;
      // y = the sum times 2^F of the row of x (M > 1; with M = 1 it is in
      // the scales): a power of two, so this equals scaling every term
      auto store = [&](const float (&v)[4]) {
        const int c0 = 2 * t, c1 = 2 * t + 1;
        const float g0 = M != 1 ? f0 : 1.f, g1 = M != 1 ? f1 : 1.f;
        if (row < Nm) {
          if (c0 < M) ym[static_cast<int64_t>(c0) * Nm + row] = round_to_dt<DT>(v[0] * g0);
          if (c1 < M) ym[static_cast<int64_t>(c1) * Nm + row] = round_to_dt<DT>(v[1] * g1);
        }
        if (row + 1 < Nm) {
          if (c0 < M) ym[static_cast<int64_t>(c0) * Nm + row + 1] = round_to_dt<DT>(v[2] * g0);
          if (c1 < M) ym[static_cast<int64_t>(c1) * Nm + row + 1] = round_to_dt<DT>(v[3] * g1);
        }
      };
      if (u_bx == 0 && c_bx == nbox - 1) {
        store(acc);
      } else {
        auto red_addr = [&](int w, int par, int l) {
          return lut_piece(kLutPieceRed + 8 * w + 4 * par + (l >> 3)) + 16u * (l & 7);
        };
        // chunk mode: lane (g, 0) holds rows 2g, 2g + 1 of the one column
        auto red_addr_cm = [&](int w, int par) {
          return lut_piece(kLutPieceRedCm + w) + 64u * par + 8u * g;
        };
        const uint32_t sh = c_tile == tile0 ? share_first : share_last;
        const int wf = static_cast<int>(sh & 15u), wl = static_cast<int>((sh >> 4) & 15u);
        // slots: every warp after wf has this tile as its first
        auto slot_of = [&](int w) { return w > wf ? 0 : static_cast<int>(sh >> 8); };
        if constexpr (CM) {
          if (t == 0)
            sts64(red_addr_cm(warp, c_tile == tile0 ? 0 : 1), __float_as_uint(acc[0]),
                  __float_as_uint(acc[2]));
        } else {
          sts128(red_addr(warp, c_tile == tile0 ? 0 : 1, lane),
                 make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                            __float_as_uint(acc[2]), __float_as_uint(acc[3])));
        }
        __threadfence_block();
        __syncwarp();
        uint32_t before = 0;
        if (lane == 0) before = atom_add_shared(tile_ctr(wf), 1u);
        before = __shfl_sync(0xFFFFFFFFu, before, 0);
        if (before == static_cast<uint32_t>(wl - wf)) {
          __threadfence_block();
          float v[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (CM) {
            if (t == 0) {
              for (int w = wf; w <= wl; ++w) {
                const uint2 r = lds64(red_addr_cm(w, slot_of(w)));
                v[0] += __uint_as_float(r.x);
                v[2] += __uint_as_float(r.y);
              }
            }
          } else {
            for (int w = wf; w <= wl; ++w) {
              const uint4 r = lds128_lut(red_addr(w, slot_of(w), lane));
              v[0] += __uint_as_float(r.x);
              v[1] += __uint_as_float(r.y);
              v[2] += __uint_as_float(r.z);
              v[3] += __uint_as_float(r.w);
            }
          }
          store(v);
        }
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      u_bx = 0;
    }
    advance(c_tile, c_bx);
  }
  // drain copies still landing (only after a wait gave up)
  if (lane == 0 && dead) {
    for (int s2 = 0; s2 < NS; ++s2) {
      const int n_st = issued_n > s2 ? (issued_n - s2 + NS - 1) / NS : 0;
      const int w_st = waited_q >= s2 ? (waited_q - s2) / NS + 1 : 0;
      if (n_st > w_st) mbar_wait_drain(bar_of(s2), static_cast<uint32_t>((n_st - 1) & 1));
    }
  }
}

}  // namespace nf4q
