// nf4_gemv, decode shapes (M <= 16): y[m, n] = sum_k x[m, k] * w_hat[n, k]
// ("bitsandbytes tutorial", sec. 3.4, sec. 七 myth 5: bandwidth-bound, the
// dequantization is extra arithmetic on top of moving the packed weights).
//
// At M = 1 a B300 must turn ~45 packed weights per SM clock into bf16 to keep
// up with HBM, i.e. under three instructions per weight, and at M = 16 the
// CUDA cores could not even do the FMAs.  So the contraction runs on the
// tensor cores (mma.sync m16n8k16, bf16 or fp16 in, fp32 accumulate) with the
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
// one: lane (g, t) feeds rows g and g+8, 64-block t of each 256-column
// segment, four columns per MMA; its B fragment is then 64 consecutive x
// values.
//
// Work split.  A CTA owns 16*R rows and a range of 1024-column chunks; its
// four warps take one 256-column segment each of every chunk.  The chunks
// stream through a ring of shared-memory stages filled by TMA (one 2D box
// of 16*R rows x 128 packed bytes per segment, 128-byte swizzle, so the
// eight rows a lane group reads sit in distinct banks); the last warp to
// finish a stage refills it.  Small weights split K over the CTAs of a
// thread-block cluster, whose partial sums meet in the shared memory of
// rank 0 (DSMEM).  Every sum is taken in a fixed order, so y is
// deterministic.
#pragma once

#include "common.cuh"
#include "tma.cuh"
#include "lut.cuh"

namespace nf4q {

constexpr int kGemvRows = 16;       // rows of one MMA tile
constexpr int kGemvSeg = 256;       // columns per warp per stage (128 packed bytes a row)
constexpr int kGemvWarps = 4;       // warps per CTA = segments per stage
constexpr int kGemvMaxStages = 4;
constexpr int kGemvStages = 2;      // stages used (more cost occupancy, measured slower)
constexpr int kGemvMinCtasPerSm = 4;
constexpr int kGemvMaxSplit = 8;    // CTAs of a cluster splitting K (portable limit)
constexpr int kGemvCtrlBytes = 128;  // mbarriers and counters

// d += A (16x16) . B (16x8), bf16 (DT 0) or fp16 (DT 1) operands, fp32 accumulate
template <int DT>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if (DT == 0)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}


template <int R>
struct GemvGeom {
  static constexpr uint32_t kSegBytes = R * kGemvRows * 128;     // one TMA box
  static constexpr uint32_t kStageBytes = kGemvWarps * kSegBytes;
};

// Dynamic shared memory of one CTA: alignment slack, the ring (reused for
// the in-CTA reduction once drained), control words, and the cluster
// reduction slots (written by other CTAs, so never aliased).
inline size_t gemv_smem_bytes(int R, int NT, int stages, int split) {
  const size_t stage = static_cast<size_t>(kGemvWarps) * R * kGemvRows * 128;
  const size_t red = static_cast<size_t>(kGemvWarps) * R * NT * 4 * 32 * sizeof(float);
  const size_t ring = std::max(stage * stages, red);
  return 1024 + ring + kGemvCtrlBytes +
         static_cast<size_t>(split) * R * NT * 4 * 32 * sizeof(float);
}

// Launch: grid = tiles * split CTAs of 128 threads, cluster (split, 1, 1);
// `per` chunks per CTA, `stages` ring stages (<= per, <= kGemvMaxStages).
template <int CODE, int NT, int R, int DT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, ScaleView sv,
                const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int N, int K, int M,
                int per, int stages, const __grid_constant__ CodeValues C) {
  using G = GemvGeom<R>;
  extern __shared__ __align__(1024) uint8_t gsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  uint32_t rank, nrank;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(nrank));
  const int row0 = static_cast<int>(blockIdx.x / nrank) * (kGemvRows * R);
  const int kblocks = K / kBlock;
  const int nseg = (K + kGemvSeg - 1) / kGemvSeg;
  const int nchunks = (nseg + kGemvWarps - 1) / kGemvWarps;
  const int c_begin = static_cast<int>(rank) * per;
  const int nmine = max(0, min(nchunks, c_begin + per) - c_begin);
  const float off = sv.double_quant ? __ldg(sv.offset) : 0.f;
  const uint16_t* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    xrow[nt] = x + static_cast<int64_t>(min(g + 8 * nt, M - 1)) * K;

  const uint32_t base = smem_u32(gsm);
  const uint32_t ring = (base + 1023u) & ~1023u;
  const size_t red_bytes = static_cast<size_t>(kGemvWarps) * R * NT * 4 * 32 * sizeof(float);
  const uint32_t ctrl =
      ring + static_cast<uint32_t>(max(static_cast<size_t>(stages) * G::kStageBytes, red_bytes));
  const uint32_t bars = ctrl;                       // [kGemvMaxStages] mbarriers
  const uint32_t cnt = ctrl + 8 * kGemvMaxStages;   // [kGemvMaxStages] release counts
  const uint32_t issued = cnt + 4 * kGemvMaxStages; // [kGemvMaxStages] loads issued
  const uint32_t cl = ctrl + kGemvCtrlBytes;        // [split][R*NT*4*32] partial sums
  auto u32_at = [&](uint32_t a) { return reinterpret_cast<uint32_t*>(gsm + (a - base)); };

  // one chunk (up to four segments) into a stage; called by one thread
  auto issue = [&](int i, int st) {
    const int c = c_begin + i;
    const int nv = min(kGemvWarps, nseg - kGemvWarps * c);
    const uint32_t bar = bars + 8 * st;
    *u32_at(issued + 4 * st) += 1u;  // before the arrive, which releases it
    mbar_arrive_expect_tx(bar, nv * G::kSegBytes);
    for (int j = 0; j < nv; ++j)
      tma_load_2d(ring + st * G::kStageBytes + j * G::kSegBytes, &tmap_w,
                  (kGemvWarps * c + j) * (kGemvSeg / 2), row0, bar);
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < kGemvMaxStages; ++st) {
      mbar_init(bars + 8 * st, 1);
      *u32_at(cnt + 4 * st) = 0u;
      *u32_at(issued + 4 * st) = 0u;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  // Cluster K split: every CTA of the cluster must be known to run before
  // another writes into its shared memory.  Arrive now, wait just before
  // the first remote store (after the main loop), so the wait costs nothing.
  if (nrank > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (threadIdx.x == 0)
    for (int i = 0; i < min(stages, nmine); ++i) issue(i, i);

  float acc[R][NT][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][nt][i] = 0.f;

  // This lane's blocks: rows row0 + 16r + g (+8), block blk of each chunk
  // (advancing by 16 a chunk); b = row * kblocks + blk fits 31 bits.  The
  // scales are fetched one chunk ahead: [tile][row g, g+8].
  int blk = kGemvWarps * (kGemvWarps * c_begin + warp) + t;
  int bidx[R][2];
  bool rok[R][2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = row0 + 16 * r + g + 8 * h;
      rok[r][h] = row < N;
      bidx[r][h] = (rok[r][h] ? row : 0) * kblocks + blk;
    }
  auto scale_at = [&](int r, int h, int bb, bool in_k) -> float {
    if (!(rok[r][h] && in_k)) return 0.f;
    if (sv.double_quant)
      return __fmaf_rn(static_cast<float>(__ldg(sv.absmax_q + bb)), __ldg(sv.scale2 + (bb >> 8)), off);
    return __ldg(sv.absmax + bb);
  };
  float scur[R][2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h) scur[r][h] = scale_at(r, h, bidx[r][h], blk < kblocks);
  const uint16_t* xp[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) xp[nt] = xrow[nt] + blk * kBlock;
  int st = 0;
  uint32_t ph = 0;
  for (int i = 0; i < nmine; ++i) {
    RowTable<CODE> T[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      build_table<CODE, DT>(T[r][0], scur[r][0], C);
      build_table<CODE, DT>(T[r][1], scur[r][1], C);
    }
    const bool in_k = blk < kblocks;
    // x of this lane's block; blocks past K read block 0 (their weights are zero)
    const uint16_t* xq[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) xq[nt] = in_k ? xp[nt] : xrow[nt];
    blk += kGemvWarps * kGemvWarps;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) xp[nt] += kGemvWarps * kGemvWarps * kBlock;
    if (i + 1 < nmine) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          bidx[r][h] += kGemvWarps * kGemvWarps;
          scur[r][h] = scale_at(r, h, bidx[r][h], blk < kblocks);
        }
    }
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_timed(bars + 8 * st, ph))) break;
    if (kGemvWarps * (c_begin + i) + warp < nseg) {  // warp-uniform: segment inside K
      const uint32_t tile = ring + st * G::kStageBytes + warp * G::kSegBytes;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        // 16-byte chunk (2t + hb) of rows g and g + 8 of each row tile
        const uint32_t chunk = ((2 * t + hb) ^ g) << 4;
        uint32_t wds[R][2][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
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
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(xq[nt] + wi * 8));
            xb[nt][0] = v.x; xb[nt][1] = v.y; xb[nt][2] = v.z; xb[nt][3] = v.w;
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            uint32_t ra[4], rb[4];
            dequant_word<CODE>(T[r][0], wds[r][0][q], ra);
            dequant_word<CODE>(T[r][1], wds[r][1][q], rb);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816<DT>(acc[r][nt], ra[2 * h], rb[2 * h], ra[2 * h + 1], rb[2 * h + 1],
                              xb[nt][2 * h], xb[nt][2 * h + 1]);
          }
        }
      }
    }
    __syncwarp();
    // Release the stage; the fourth warp to do so refills it.  The arriving
    // warp has already used every word it read from the stage (the values
    // fed its MMAs), and shared-memory accesses of a thread complete in
    // order, so a relaxed add suffices; the last arriver's proxy fence then
    // orders the refill after all of them.
    if (lane == 0) {
      const uint32_t prev = atom_add_shared(cnt + 4 * st, 1u);
      if ((prev & (kGemvWarps - 1)) == kGemvWarps - 1 && i + stages < nmine) {
        fence_proxy_async_smem();
        issue(i + stages, st);
      }
    }
    if (++st == stages) { st = 0; ph ^= 1u; }
  }
  __syncthreads();
  // drain: no copy may still be landing when the ring is reused or the CTA
  // exits (only after a timed-out wait can one still be in flight)
  if (threadIdx.x == 0) {
    for (int st = 0; st < stages; ++st) {
      const uint32_t n = *u32_at(issued + 4 * st);
      if (n > 0) mbar_wait_drain(bars + 8 * st, (n - 1) & 1);
    }
  }
  __syncthreads();

  // fixed-order reduction over the warps of the CTA (in the drained ring)
  constexpr int kItems = R * NT * 4 * 32;
  float* red = reinterpret_cast<float*>(gsm + (ring - base));
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        red[warp * kItems + ((r * NT + nt) * 4 + i) * 32 + lane] = acc[r][nt][i];
  __syncthreads();
  auto store_y = [&](int item, float v) {
    const int ln = item & 31, i = (item >> 5) & 3, rn = item >> 7;
    const int nt = rn % NT, r = rn / NT;
    // d0,d1: row g, cols 2t, 2t+1; d2,d3: row g+8
    const int row = row0 + 16 * r + (ln >> 2) + (i < 2 ? 0 : 8);
    const int col = 8 * nt + 2 * (ln & 3) + (i & 1);
    if (row < N && col < M) y[static_cast<int64_t>(col) * N + row] = round_to_dt<DT>(v);
  };
  if (nrank > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int item = threadIdx.x; item < kItems; item += kGemvWarps * 32) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) v += red[w * kItems + item];
    if (nrank == 1) {
      store_y(item, v);
    } else {  // into slot `rank` of the cluster's rank 0
      const uint32_t local = cl + (rank * kItems + item) * 4;
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(local));
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
    }
  }
  if (nrank > 1) {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank == 0) {
      const float* slots = reinterpret_cast<const float*>(gsm + (cl - base));
      for (int item = threadIdx.x; item < kItems; item += kGemvWarps * 32) {
        float v = 0.f;
        for (uint32_t r = 0; r < nrank; ++r) v += slots[r * kItems + item];
        store_y(item, v);
      }
    }
  }
}

}  // namespace nf4q
