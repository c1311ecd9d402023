// nf4_gemm: Y [M x N] = X [M x K] . w_hat^T on the 5th-generation tensor
// cores ("bitsandbytes tutorial", sec. 3.4: the 4-bit weight is dequantized
// to bf16 and an ordinary bf16 matmul with fp32 accumulation follows).
//
// One CTA computes a 128 x 256 tile of Y with tcgen05.mma (kind::f16, bf16
// operands, fp32 accumulator in tensor memory), K in steps of 64:
//   warp 0      TMA producer: the X tile (128 x 64 bf16, 128-byte swizzle)
//               and the packed W tile (256 rows x 32 bytes, 32-byte swizzle)
//               of each stage, one mbarrier with the transaction byte count.
//   warp 1      allocates 256 TMEM columns; one lane issues the four
//               128x256x16 MMAs of a stage and commits them to the stage's
//               "empty" barrier, and after the last stage to "acc_full".
//   warps 2..9  dequantize: thread r rebuilds row r of the W tile,
//               w_hat = bf16(code[nibble] * s_b) exactly as nf4_dequantize,
//               into the K-major 128-byte-swizzled layout the MMA reads,
//               then fence.proxy.async and arrive on the stage's "b_full".
//               After the main loop the same warps drain TMEM (tcgen05.ld),
//               round to bf16 and store Y.
// Every wait is bounded (about 2 s of %globaltimer); a wait that gives up
// sets bit 0 of the device error word and the CTA winds down: it waits
// (bounded) for its own TMA copies and MMAs, frees its TMEM and returns.
// No multicast: every CTA loads its own tiles.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace nf4q {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;
constexpr int kGemmStages = 3;
constexpr int kGemmThreads = 320;
constexpr int kGemmATile = kGemmBM * kGemmBK * 2;    // 16 KB
constexpr int kGemmBTile = kGemmBN * kGemmBK * 2;    // 32 KB
constexpr int kGemmPTile = kGemmBN * kGemmBK / 2;    // 8 KB
constexpr int kGemmTmemCols = 256;
constexpr size_t kGemmSmemBytes =
    1024 + kGemmStages * (kGemmATile + kGemmBTile + kGemmPTile) + 1024 + 16 * 32 * 4;

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Bounded wait for the phase of the given parity.  Gives up (false) after
// the time limit, or as soon as another thread of the CTA has given up
// (`abort` in shared memory), so a stuck CTA winds down quickly.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort = 1u;
      atomicOr(&g_device_error, 1u);
      return false;
    }
  }
}

// Bounded wait that ignores the CTA abort flag: used before the CTA exits,
// to let its own TMA copies and MMAs finish.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_device_error, 1u);
      return;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0,
                                            int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

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
__host__ __device__ constexpr uint32_t make_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
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

// ------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
            const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
            uint16_t* __restrict__ Y, int M, int N, int K,
            const __grid_constant__ CodeValues C) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = sA + kGemmStages * kGemmATile;
  const uint32_t sP = sB + kGemmStages * kGemmBTile;
  const uint32_t sBar = sP + kGemmStages * kGemmPTile;   // 1 KB of barriers
  uint8_t* gB = gbase + (sB - base);
  const uint8_t* gP = gbase + (sP - base);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sBar - base) + 512);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(gbase + (sBar - base) + 516);
  float* s_code = reinterpret_cast<float*>(gbase + (sBar - base) + 1024);
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto bfull_bar = [&](int s) { return sBar + 8u * (kGemmStages + s); };
  auto empty_bar = [&](int s) { return sBar + 8u * (2 * kGemmStages + s); };
  const uint32_t acc_bar = sBar + 8u * (3 * kGemmStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kGemmBN, m0 = blockIdx.y * kGemmBM;
  const int KT = K / kGemmBK;

  for (int i = threadIdx.x; i < 16 * 32; i += blockDim.x) s_code[i] = C.v[i >> 5];
  if (threadIdx.x == 0) {
    *abort = 0u;
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(bfull_bar(s), 8);
      mbar_init(empty_bar(s), 1);
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
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kGemmStages;
        const uint32_t ph = (kt / kGemmStages) & 1;
        if (!mbar_wait(empty_bar(s), ph ^ 1, abort)) break;
        mbar_arrive_expect_tx(full_bar(s), kGemmATile + kGemmPTile);
        tma_load_2d(sA + s * kGemmATile, &tmap_x, kt * kGemmBK, m0, full_bar(s));
        tma_load_2d(sP + s * kGemmPTile, &tmap_w, kt * (kGemmBK / 2), n0, full_bar(s));
        issued = kt + 1;
      }
      // wind-down: make sure no copy is still landing in this CTA's smem
      for (int kt = (issued > kGemmStages ? issued - kGemmStages : 0); kt < issued; ++kt)
        mbar_wait_drain(full_bar(kt % kGemmStages), (kt / kGemmStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kGemmBM, kGemmBN);
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kGemmStages;
        const uint32_t ph = (kt / kGemmStages) & 1;
        if (!mbar_wait(full_bar(s), ph, abort)) break;
        if (!mbar_wait(bfull_bar(s), ph, abort)) break;
        tc_fence_after();
        const uint32_t a0 = sA + s * kGemmATile, b0 = sB + s * kGemmBTile;
#pragma unroll
        for (int k = 0; k < kGemmBK / 16; ++k) {
          mma_bf16(tmem, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k), idesc,
                   (kt > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(s));
      }
      mma_commit(acc_bar);  // fires once every MMA issued above has completed
    }
  } else {
    // ---------------- dequantize producers (256 threads, one W row each)
    const int r = threadIdx.x - 64;
    const int n = n0 + r;
    const bool row_ok = n < N;
    const int64_t row_block0 = static_cast<int64_t>(n) * (K / kBlock);
    const float* code = s_code + lane;
    float s_next = (row_ok && KT > 0) ? block_scale(sv, row_block0) : 0.f;
    bool ok = true;
    for (int kt = 0; kt < KT && ok; ++kt) {
      const int s = kt % kGemmStages;
      const uint32_t ph = (kt / kGemmStages) & 1;
      const float sc = s_next;
      if (row_ok && kt + 1 < KT) s_next = block_scale(sv, row_block0 + kt + 1);
      // B slot s is free once the MMAs of the previous round on it are done
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(s), ph ^ 1, abort) &&
                                       mbar_wait(full_bar(s), ph, abort))) {
        ok = false;
        break;
      }
      const uint8_t* prow = gP + s * kGemmPTile + r * 32;
      const int sw = (r >> 2) & 1;  // 32-byte swizzle of the TMA tile
      const uint4 p0 = *reinterpret_cast<const uint4*>(prow + ((0 ^ sw) << 4));
      const uint4 p1 = *reinterpret_cast<const uint4*>(prow + ((1 ^ sw) << 4));
      const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint8_t* brow = gB + s * kGemmBTile + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // chunk c = elements 8c..8c+7 = packed word c
        const uint32_t p = words[c];
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t nib = (p >> (8 * (i >> 1) + ((i & 1) ? 0 : 4))) & 0xFu;
          f[i] = __fmul_rn(code[nib * 32], sc);
        }
        uint4 o;
        o.x = pack_bf16x2(f[0], f[1]);
        o.y = pack_bf16x2(f[2], f[3]);
        o.z = pack_bf16x2(f[4], f[5]);
        o.w = pack_bf16x2(f[6], f[7]);
        *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bfull_bar(s));
    }
    // ---------------- epilogue: TMEM -> bf16 -> Y
    if (__all_sync(0xFFFFFFFFu, mbar_wait(acc_bar, 0, abort))) {
      tc_fence_after();
      const int q = warp & 3;        // TMEM lane quarter this warp may read
      const int h = (warp - 2) >> 2;  // column half
      const int m = m0 + q * 32 + lane;
      for (int cc = 0; cc < 4; ++cc) {
        const int col = h * 128 + cc * 32;
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + col, v);
        if (m < M) {
          uint16_t* yrow = Y + static_cast<int64_t>(m) * N + n0 + col;
          const int ncols = min(32, N - (n0 + col));
          if (ncols == 32 && (N & 7) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
              *reinterpret_cast<uint4*>(yrow + 8 * j) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < ncols) {
                const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]));
                yrow[j] = *reinterpret_cast<const uint16_t*>(&b);
              }
            }
          }
        }
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

// ------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

inline nf4q_status gemm_launch(const nf4q_weight* wq, const ScaleView& sv,
                               const CodeValues& C, const void* X, int64_t M, void* Y,
                               cudaStream_t stream, int /*sms*/) {
  const int64_t N = wq->rows, K = wq->cols;
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NF4Q_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return NF4Q_ERR_CUDA;
  CUtensorMap tx, tw;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {kGemmBK, kGemmBM};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return NF4Q_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[2] = {kGemmBK / 2, kGemmBN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq->packed, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return NF4Q_ERR_CUDA;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmemBytes)) != cudaSuccess)
      return NF4Q_ERR_CUDA;
    attr_set[dev] = true;
  }
  if ((M + kGemmBM - 1) / kGemmBM > 65535) return NF4Q_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>((N + kGemmBN - 1) / kGemmBN),
            static_cast<unsigned>((M + kGemmBM - 1) / kGemmBM));
  gemm_kernel<<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(
      tx, tw, sv, static_cast<uint16_t*>(Y), static_cast<int>(M), static_cast<int>(N),
      static_cast<int>(K), C);
  return cudaGetLastError() == cudaSuccess ? NF4Q_OK : NF4Q_ERR_CUDA;
}

}  // namespace nf4q
