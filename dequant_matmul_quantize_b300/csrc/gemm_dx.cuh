// nf4_gemm_dx: dX [M x K] = dY [M x N] . w_hat [N x K] on the 5th-generation
// tensor cores - the input gradient of y = x . w_hat^T through a frozen
// 4-bit weight, the backward pass of QLoRA's base layer ("bitsandbytes
// tutorial", sec. 5.4: the NF4 weight stays frozen and only the LoRA
// adapters train, so the base layer needs dX but no dW).
//
// The contraction runs over the weight's rows n, so the dequantized weight
// is the B operand in MN-major form: a stage holds 64 rows n of w_hat and
// BN output columns k.  Row n of a stage covers BN / 64 whole 64-blocks of
// that row, each rebuilt from its packed bytes and scale by one thread with
// the register byte tables of lut.cuh (the same bit-exact w_hat as
// nf4_dequantize), and written as one 128-byte row of the 128-byte-swizzled
// MN-major layout: chunk c (columns 64c .. 64c+63) of the tile is 64 rows of
// 128 bytes, 8-row groups 1024 bytes apart, chunks 8 KB apart.  Everything
// else is the forward kernel's pipeline (gemm.cuh):
//   warp 0      TMA: two dY tiles (128 x 64, K-major over n, 128-byte
//               swizzle) and the packed tile (64 rows x BN/2 bytes) of a
//               stage, one mbarrier with the byte count;
//   warp 1      512 TMEM columns; one lane issues the 2 x 4 MMAs of a stage
//               (128 x BN x 16, B transposed = MN-major);
//   warps 2..   dequantize producers, groups of 8 warps on alternate stages;
//               afterwards warps 2..17 drain the accumulators.
// Rows n >= N and columns k >= K of the last tiles get scale 0 (w_hat = 0);
// the TMA zero-fills dY beyond N, so they add nothing.  Every wait is
// bounded as in the forward kernel.
//
// When 128 x 128 tiles (one accumulator, MT = 1) fit one wave, a CTA owns
// 128 rows of dY, and if the tiles still leave SMs idle the contraction
// over n is split across a thread-block cluster (S <= 4 CTAs, stages
// [r NT / S, (r + 1) NT / S) for rank r) whose fp32 partials are summed in
// rank order in rank 0's shared memory, as in the forward kernel's split K.
#pragma once

#include "gemm.cuh"

namespace nf4q {

constexpr int kDxRows = 64;  // contraction rows n per stage

template <int BN, int MT = 2>
struct GemmDxCfg {
  static constexpr int kChunks = BN / 64;              // 64-column chunks (blocks) per row
  static constexpr int kBTile = kDxRows * BN * 2;      // dequantized w_hat tile
  static constexpr int kPTile = kDxRows * BN / 2;      // packed tile
  static constexpr int kAStages = MT == 2 ? 4 : 8;
  static constexpr int kAStage = MT * kGemmATile + kPTile;
  static constexpr int kBStages =
      (kAStages * kAStage + 3 * kBTile + 2048 <= 232448 - 1024) ? 3 : 2;
  static constexpr size_t kSmem = 1024 + kAStages * kAStage + kBStages * kBTile + 1024;
  static constexpr int kGroups = kBStages;
  static constexpr int kThreads = 64 + kGroups * 256;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN: whole 64-blocks, MMA N <= 256");
  static_assert(kPTile % 1024 == 0 && kBTile % 1024 == 0, "1 KB alignment of tiles");
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(MT == 1 || MT == 2, "one or two accumulators");
};

// MN-major operand in the 128-byte swizzled layout: the leading byte offset
// is the distance between 64-element chunks along MN (8 KB: 64 rows of 128
// bytes), the stride byte offset the distance between 8-row groups along
// the contraction (1 KB).  Other fields as smem_desc_sw128.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((kDxRows * 128) >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// SP: the split epilogue is compiled in (always with one accumulator; with
// two only in the instantiation that splits, which keeps the others free of
// its register pressure).
template <int CODE, int BN, int DT, int MT, bool SP>
__global__ void __launch_bounds__(GemmDxCfg<BN, MT>::kThreads, 1)
gemm_dx_kernel(const __grid_constant__ CUtensorMap tmap_dy,
               const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
               uint16_t* __restrict__ dX, int M, int N, int K,
               const __grid_constant__ CodeValues C) {
  using Cfg = GemmDxCfg<BN, MT>;
  constexpr int SA = Cfg::kAStages, SB = Cfg::kBStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sA = [&](int s, int h) { return base + s * Cfg::kAStage + h * kGemmATile; };
  auto sP = [&](int s) { return base + s * Cfg::kAStage + MT * kGemmATile; };
  auto sB = [&](int s) { return base + SA * Cfg::kAStage + s * Cfg::kBTile; };
  const uint32_t sBar = base + SA * Cfg::kAStage + SB * Cfg::kBTile;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sBar - base) + 512);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(gbase + (sBar - base) + 516);
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto aempty_bar = [&](int s) { return sBar + 8u * (SA + s); };
  auto bfull_bar = [&](int s) { return sBar + 8u * (2 * SA + s); };
  auto bempty_bar = [&](int s) { return sBar + 8u * (2 * SA + SB + s); };
  const uint32_t acc_bar = sBar + 8u * (2 * SA + 2 * SB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = blockIdx.x * BN, m0 = blockIdx.y * (MT * kGemmBM);
  const int NT = (N + kDxRows - 1) / kDxRows;  // stages
  // split of the contraction: this CTA's stages t0 .. t0 + nst - 1
  const int S = static_cast<int>(gridDim.z);
  uint32_t rank = 0;
  if (S > 1) asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int t0 = static_cast<int>(rank) * NT / S;
  const int nst = (static_cast<int>(rank) + 1) * NT / S - t0;

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
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_dy)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
      int issued = 0;
      for (int i = 0; i < nst; ++i) {
        const int t = t0 + i;
        const int s = i % SA;
        if (!mbar_wait(aempty_bar(s), ((i / SA) & 1) ^ 1, abort)) break;
        mbar_arrive_expect_tx(full_bar(s), MT * kGemmATile + Cfg::kPTile);
        tma_load_2d(sA(s, 0), &tmap_dy, t * kDxRows, m0, full_bar(s));
        if (MT == 2) tma_load_2d(sA(s, 1), &tmap_dy, t * kDxRows, m0 + kGemmBM, full_bar(s));
        tma_load_2d(sP(s), &tmap_w, k0 / 2, t * kDxRows, full_bar(s));
        issued = i + 1;
      }
      for (int i = (issued > SA ? issued - SA : 0); i < issued; ++i)
        mbar_wait_drain(full_bar(i % SA), (i / SA) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<DT>(kGemmBM, BN) | (1u << 16);  // B MN-major
      for (int i = 0; i < nst; ++i) {
        const int sa = i % SA, sb = i % SB;
        if (!mbar_wait(full_bar(sa), (i / SA) & 1, abort)) break;
        if (!mbar_wait(bfull_bar(sb), (i / SB) & 1, abort)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kDxRows / 16; ++k) {
          // rows 16k .. 16k+15 of the stage: two 8-row groups of 1 KB
          const uint64_t bdesc = smem_desc_sw128_mn(sB(sb) + 2048 * k);
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          mma_bf16(tmem, smem_desc_sw128(sA(sa, 0) + 32 * k), bdesc, idesc, acc);
          if (MT == 2) mma_bf16(tmem + 256, smem_desc_sw128(sA(sa, 1) + 32 * k), bdesc, idesc, acc);
        }
        mma_commit(aempty_bar(sa));
        mma_commit(bempty_bar(sb));
      }
      mma_commit(acc_bar);
    }
  } else {
    // ---------------- dequantize producers: thread (r, c) of a group
    // rebuilds block c of row t * 64 + r in each of its stages t
    const int idx = threadIdx.x - 64;
    const int grp = idx >> 8;
    const int r = idx & 63;
    const int c = (idx & 255) >> 6;
    const bool active = c < Cfg::kChunks;
    const int kblocks = K / kBlock;
    const int kb = k0 / kBlock + c;  // block column
    const bool col_ok = active && kb < kblocks;
    const float off = sv.double_quant ? __ldg(sv.offset) : 0.f;
    // The scale inputs of this thread's block in stage t, loaded one own
    // stage ahead and turned into the scale only when used, so no
    // instruction waits on the load before then.  Outside the weight
    // (rows >= N, blocks >= K / 64) the scale is 0.
    struct RawScale {
      int q;       // int8 code of the double-quantized scale
      float s;     // its scale2, or the fp32 absmax without double quant
      bool ok;
    };
    auto load_scale = [&](int t) -> RawScale {
      RawScale v{0, 0.f, false};
      const int n = t * kDxRows + r;
      if (!col_ok || t >= NT || n >= N) return v;
      const int64_t b = static_cast<int64_t>(n) * kblocks + kb;
      v.ok = true;
      if (sv.double_quant) {
        v.q = __ldg(sv.absmax_q + b);
        v.s = __ldg(sv.scale2 + (b >> 8));
      } else {
        v.s = __ldg(sv.absmax + b);
      }
      return v;
    };
    RawScale next = load_scale(grp < nst ? t0 + grp : NT);
    for (int i = grp; i < nst; i += Cfg::kGroups) {
      const int t = t0 + i;
      const int sa = i % SA, sb = i % SB;
      const RawScale cur = next;
      next = load_scale(i + Cfg::kGroups < nst ? t + Cfg::kGroups : NT);
      const float sc = !cur.ok ? 0.f
                     : (sv.double_quant ? __fmaf_rn(static_cast<float>(cur.q), cur.s, off) : cur.s);
      RowTable<CODE> T;
      build_table<CODE, DT>(T, sc, C);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bempty_bar(sb), ((i / SB) & 1) ^ 1, abort) &&
                                       mbar_wait(full_bar(sa), (i / SA) & 1, abort)))
        break;
      if (active) {
        // packed row r: BN / 2 bytes, of which this block is the 16-byte
        // chunks 2c and 2c + 1, stored by the TMA at chunk ^ (r % 8) for
        // 128-byte rows (BN = 256) and chunk ^ ((r / 2) % 4) for 64-byte rows
        // (BN = 128); 96-byte rows (BN = 192) are unswizzled
        const uint8_t* prow = gbase + (sP(sa) - base) + r * (BN / 2);
        const int swz = r & 7;
        const int pswz = BN == 256 ? swz : (BN == 128 ? ((r >> 1) & 3) : 0);
        const int pc0 = (2 * c) ^ pswz, pc1 = (2 * c + 1) ^ pswz;
        const uint4 p0 = *reinterpret_cast<const uint4*>(prow + (pc0 << 4));
        const uint4 p1 = *reinterpret_cast<const uint4*>(prow + (pc1 << 4));
        const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        uint8_t* brow = gbase + (sB(sb) - base) + c * (kDxRows * 128) + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = columns 8j .. 8j+7 of the block
          uint32_t o[4];
          dequant_word<CODE>(T, words[j], o);
          *reinterpret_cast<uint4*>(brow + ((j ^ swz) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bfull_bar(sb));
    }
    if (S == 1 && warp < 18 && __all_sync(0xFFFFFFFFu, mbar_wait(acc_bar, 0, abort))) {
      tc_fence_after();
      store_accumulators<BN, DT, MT>(tmem, warp, lane, dX, M, K, m0, k0);
    }
  }
  if constexpr (SP && BN % 32 == 0) {
   if (S > 1) {
    // split of the contraction: every thread of the cluster passes both
    // barriers (as in the forward kernel); with two accumulators each rank
    // sends both (rows m0 .. m0 + 127 and m0 + 128 .. m0 + 255)
    __syncwarp();
    const bool epi = warp >= 2 && warp < 18;
    bool ok = true;
    if (epi) ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_bar, 0, abort));
    tc_fence_before();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (epi && ok && rank > 0) {
      tc_fence_after();
#pragma unroll 1
      for (int a = 0; a < MT; ++a)
        send_partials<BN>(tmem + 256u * a, warp, lane, base, rank, a, MT);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (epi && ok && rank == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int a = 0; a < MT; ++a)
        store_split_sum<BN, DT>(tmem + 256u * a, warp, lane, base, S, dX, M, K,
                                m0 + kGemmBM * a, k0, a, MT);
    }
   }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait_drain(acc_bar, 0);
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kGemmTmemCols)
                 : "memory");
  }
}

// BN (output columns per CTA) for a shape: the forward kernel's wave rule
// over the widths with whole 64-blocks.
inline int gemm_dx_pick_bn(int64_t M, int64_t K, int sms) {
  const int cands[3] = {256, 192, 128};
  const double rate[3] = {1.00, 0.93, 0.68};
  const int64_t mt = (M + 2 * kGemmBM - 1) / (2 * kGemmBM);
  int best = 256;
  double best_score = -1.0;
  for (int i = 0; i < 3; ++i) {
    const int bn = cands[i];
    const int64_t tiles = mt * ((K + bn - 1) / bn);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const double eff = static_cast<double>(K) * mt / (static_cast<double>(rounds) * sms * bn);
    const double score = eff * rate[i];
    if (score > best_score + 1e-9) { best_score = score; best = bn; }
  }
  return best;
}

template <int CODE, int BN, int DT, int MT = 2, bool SP = (MT == 1)>
inline nf4q_status gemm_dx_launch_bn(const CUtensorMap& tdy, const nf4q_weight* wq,
                                     const ScaleView& sv, const CodeValues& C, int64_t M,
                                     void* dX, cudaStream_t stream, int sms) {
  using Cfg = GemmDxCfg<BN, MT>;
  const int64_t N = wq->rows, K = wq->cols;
  EncodeTiledFn enc = encode_tiled_fn();
  CUtensorMap tw;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {BN / 2, kDxRows};
  cuuint32_t es[2] = {1, 1};
  // 128- and 64-byte rows take the swizzle of their width, which makes the
  // producers' 16-byte reads conflict-free; 96-byte rows (BN = 192) have no
  // matching swizzle and are read with 2-way conflicts
  nf4q_status st = cu_check(
      enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq->packed, dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          BN == 256 ? CU_TENSOR_MAP_SWIZZLE_128B
                    : (BN == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
      "cuTensorMapEncodeTiled (dX weight)");
  if (st != NF4Q_OK) return st;
  static bool attr_set[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if ((st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) != NF4Q_OK) return st;
  if (dev < 0 || dev >= 64) return NF4Q_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(gemm_dx_kernel<CODE, BN, DT, MT, SP>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cfg::kSmem)),
                      "cudaFuncSetAttribute (dX GEMM)");
      if (st != NF4Q_OK) return st;
      attr_set[dev] = true;
    }
  }
  const int64_t tiles = ((K + BN - 1) / BN) * ((M + MT * kGemmBM - 1) / (MT * kGemmBM));
  const int S = (SP && BN % 32 == 0)
                    ? gemm_split_k(tiles, (N + kDxRows - 1) / kDxRows, sms,
                                   int64_t{MT} * kGemmBM * BN * 4,
                                   int64_t{Cfg::kAStages} * Cfg::kAStage +
                                       int64_t{Cfg::kBStages} * Cfg::kBTile)
                    : 1;
  dim3 grid(static_cast<unsigned>((K + BN - 1) / BN),
            static_cast<unsigned>((M + MT * kGemmBM - 1) / (MT * kGemmBM)),
            static_cast<unsigned>(S));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = static_cast<unsigned>(S);
  return launch("gemm_dx_kernel", gemm_dx_kernel<CODE, BN, DT, MT, SP>, grid, dim3(Cfg::kThreads),
                Cfg::kSmem, stream, attr, S > 1 ? 1u : 0u, tdy, tw, sv,
                static_cast<uint16_t*>(dX), static_cast<int>(M), static_cast<int>(N),
                static_cast<int>(K), C);
}

template <int CODE, int DT>
inline nf4q_status gemm_dx_launch_code(const CUtensorMap& tdy, const nf4q_weight* wq,
                                       const ScaleView& sv, const CodeValues& C, int64_t M,
                                       void* dX, cudaStream_t stream, int bn, int sms) {
  // 128 x 128 tiles with one accumulator (then the split) when they fit one
  // wave: at M = 256 on a 4096-column weight 64 CTAs x 2 instead of 16.
  // When that wave leaves no room for a split but 256 x 128 tiles would
  // (M = 512 on such a weight: 128 CTAs walking all rows of w_hat), the two
  // accumulators share each dequantized tile and the split halves the walk.
  const int64_t t1 = ((M + kGemmBM - 1) / kGemmBM) * ((wq->cols + 127) / 128);
  const int64_t t2 = ((M + 2 * kGemmBM - 1) / (2 * kGemmBM)) * ((wq->cols + 127) / 128);
  if (t1 <= sms && t1 * 2 > sms && t2 * 2 <= sms)
    return gemm_dx_launch_bn<CODE, 128, DT, 2, true>(tdy, wq, sv, C, M, dX, stream, sms);
  if (t1 <= sms) return gemm_dx_launch_bn<CODE, 128, DT, 1>(tdy, wq, sv, C, M, dX, stream, sms);
  switch (bn) {
    case 192: return gemm_dx_launch_bn<CODE, 192, DT>(tdy, wq, sv, C, M, dX, stream, sms);
    case 128: return gemm_dx_launch_bn<CODE, 128, DT>(tdy, wq, sv, C, M, dX, stream, sms);
    default: return gemm_dx_launch_bn<CODE, 256, DT>(tdy, wq, sv, C, M, dX, stream, sms);
  }
}

// dX = dY . w_hat after the entry point's checks: M, rows, cols > 0; dY's
// row pitch ld_dy >= rows elements, a multiple of 8 (16 bytes).
inline nf4q_status gemm_dx_launch(const nf4q_weight* wq, const ScaleView& sv,
                                  const CodeValues& C, const void* dY, int64_t ld_dy, int64_t M,
                                  void* dX, cudaStream_t stream, int sms) {
  const int64_t N = wq->rows, K = wq->cols;
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NF4Q_ERR_UNSUPPORTED;
  if ((M + 2 * kGemmBM - 1) / (2 * kGemmBM) > 65535) return NF4Q_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled: driver entry point not found");
  if (ensure_context() != NF4Q_OK) return NF4Q_ERR_CUDA;
  CUtensorMap tdy;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_dy) * 2};
  cuuint32_t box[2] = {kDxRows, kGemmBM};
  cuuint32_t es[2] = {1, 1};
  const int dt = wq->compute_dtype;
  const nf4q_status st = cu_check(
      enc(&tdy, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
          const_cast<void*>(dY), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
      "cuTensorMapEncodeTiled (dY)");
  if (st != NF4Q_OK) return st;
  const int bn = gemm_dx_pick_bn(M, K, sms);
  if (dt == 0)
    return wq->code == 0 ? gemm_dx_launch_code<0, 0>(tdy, wq, sv, C, M, dX, stream, bn, sms)
                         : gemm_dx_launch_code<1, 0>(tdy, wq, sv, C, M, dX, stream, bn, sms);
  return wq->code == 0 ? gemm_dx_launch_code<0, 1>(tdy, wq, sv, C, M, dX, stream, bn, sms)
                       : gemm_dx_launch_code<1, 1>(tdy, wq, sv, C, M, dX, stream, bn, sms);
}

}  // namespace nf4q
