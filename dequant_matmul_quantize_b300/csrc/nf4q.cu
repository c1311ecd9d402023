// C-ABI entry points of libnf4q: argument checks on the host, then launches
// of the kernels in the included headers on the caller's stream.  The whole
// library is one translation unit.
#include "nf4q.h"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "dequantize.cuh"
#include "double_quant.cuh"
#include "gemm.cuh"
#include "gemm_dx.cuh"
#include "gemv_lut.cuh"
#include "gemv_mma.cuh"
#include "host.h"
#include "int8.cuh"
#include "quantize.cuh"

namespace nf4q {
namespace {

const HostTables& tables() {
  static HostTables T;
  static std::once_flag once;
  std::call_once(once, [] { T = build_host_tables(); });
  return T;
}

constexpr int kMaxDevices = 64;

int sm_count() {
  static int cache[kMaxDevices] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
inline bool aligned4(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 3u) == 0;
}

// Shape and layout checks shared by every call on a quantized weight.
nf4q_status check_shape(const nf4q_weight* wq) {
  if (!wq) return NF4Q_ERR_INVALID_ARG;
  if (wq->rows < 0 || wq->cols < 0 || wq->cols % kBlock != 0)
    return NF4Q_ERR_INVALID_ARG;
  if (wq->blocksize != kBlock || wq->dq_blocksize != kDqBlock)
    return NF4Q_ERR_INVALID_ARG;
  if (wq->code != NF4Q_CODE_NF4 && wq->code != NF4Q_CODE_FP4)
    return NF4Q_ERR_INVALID_ARG;
  if (wq->double_quant != 0 && wq->double_quant != 1) return NF4Q_ERR_INVALID_ARG;
  if (wq->compute_dtype != NF4Q_DT_BF16 && wq->compute_dtype != NF4Q_DT_F16)
    return NF4Q_ERR_INVALID_ARG;
  // n_b must fit the 32-bit divisor of the exact mean
  if (wq->rows > 0 && wq->cols > 0 &&
      wq->rows > (static_cast<int64_t>(0x7FFFFFFF) * kBlock) / wq->cols)
    return NF4Q_ERR_UNSUPPORTED;
  return NF4Q_OK;
}

// Checks of the stored state a dequantizer reads.
nf4q_status check_scales(const nf4q_weight* wq) {
  if (!wq->packed) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(wq->packed)) return NF4Q_ERR_ALIGNMENT;
  if (wq->double_quant) {
    if (!wq->absmax_q || !wq->scale2 || !wq->offset) return NF4Q_ERR_INVALID_ARG;
    if (!aligned16(wq->absmax_q) || !aligned4(wq->scale2) || !aligned4(wq->offset))
      return NF4Q_ERR_ALIGNMENT;
  } else {
    if (!wq->absmax) return NF4Q_ERR_INVALID_ARG;
    if (!aligned4(wq->absmax)) return NF4Q_ERR_ALIGNMENT;
  }
  return NF4Q_OK;
}

// The GEMV instantiations: code (NF4, FP4) x (NT, R) in {(1, 1), (1, 2),
// (2, 2)} x compute dtype (bf16, fp16).
using GemvKernelFn = void (*)(CUtensorMap, ScaleView, const uint16_t*, uint16_t*, int, int, int,
                              int, int, CodeValues);
template <int CODE, int DT>
GemvKernelFn gemv_kernel_cd(int NT, int R) {
  if (NT == 2) return gemv_mma_kernel<CODE, 2, 2, DT>;
  return R == 2 ? gemv_mma_kernel<CODE, 1, 2, DT> : gemv_mma_kernel<CODE, 1, 1, DT>;
}
GemvKernelFn gemv_kernel(int code, int NT, int R, int dt) {
  if (dt == 0) return code == 0 ? gemv_kernel_cd<0, 0>(NT, R) : gemv_kernel_cd<1, 0>(NT, R);
  return code == 0 ? gemv_kernel_cd<0, 1>(NT, R) : gemv_kernel_cd<1, 1>(NT, R);
}

// The current device (0 .. kMaxDevices-1) or an error status.
nf4q_status current_device(int* dev) {
  nf4q_status st = cuda_check(cudaGetDevice(dev), "cudaGetDevice");
  if (st == NF4Q_OK && (*dev < 0 || *dev >= kMaxDevices)) return NF4Q_ERR_UNSUPPORTED;
  return st;
}

// Opt the GEMV kernels in to their largest dynamic shared memory (once per
// device).
nf4q_status gemv_attr_ready() {
  static bool done[kMaxDevices] = {false};
  static std::mutex mu;
  int dev = 0;
  nf4q_status st = current_device(&dev);
  if (st != NF4Q_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return NF4Q_OK;
  const int bytes = static_cast<int>(gemv_smem_bytes(2, 2, kGemvMaxStages, kGemvMaxSplit));
  const int shapes[3][2] = {{1, 1}, {1, 2}, {2, 2}};  // (NT, R)
  for (int code = 0; code < 2; ++code)
    for (const auto& sh : shapes)
      for (int dt = 0; dt < 2; ++dt)
        if ((st = cuda_check(cudaFuncSetAttribute(gemv_kernel(code, sh[0], sh[1], dt),
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  bytes),
                             "cudaFuncSetAttribute (GEMV)")) != NF4Q_OK)
          return st;
  done[dev] = true;
  return NF4Q_OK;
}

// Opt the block-scale-folded GEMV kernels in to their shared memory (once
// per device).
using LutKernelFn = void (*)(LutGroup, const uint16_t*, int, int, int, HalfCodes, int);

// The folded-GEMV instantiation for a compute dtype, double quant, box size,
// whether the scales are read in 16-block chunks (double quant with K / 64
// a multiple of 16) and whether x has a single row.
template <int DT, bool DQ, int BB>
LutKernelFn gemv_lut_kernel_bb(bool ep, bool m1) {
  if (DQ && ep)
    return m1 ? gemv_lut_kernel<DT, DQ, BB, DQ, true> : gemv_lut_kernel<DT, DQ, BB, DQ, false>;
  return m1 ? gemv_lut_kernel<DT, DQ, BB, false, true> : gemv_lut_kernel<DT, DQ, BB, false, false>;
}
template <int DT, bool DQ>
LutKernelFn gemv_lut_kernel_dq(int bb, bool ep, bool m1) {
  return bb == 8 ? gemv_lut_kernel_bb<DT, DQ, 8>(ep, m1) : gemv_lut_kernel_bb<DT, DQ, 4>(ep, m1);
}
LutKernelFn gemv_lut_kernel_for(int dt, bool dq, int bb, bool ep, bool m1) {
  if (dt == 0)
    return dq ? gemv_lut_kernel_dq<0, true>(bb, ep, m1) : gemv_lut_kernel_dq<0, false>(bb, ep, m1);
  return dq ? gemv_lut_kernel_dq<1, true>(bb, ep, m1) : gemv_lut_kernel_dq<1, false>(bb, ep, m1);
}

nf4q_status gemv_lut_attr_ready() {
  static bool done[kMaxDevices] = {false};
  static std::mutex mu;
  int dev = 0;
  nf4q_status st = current_device(&dev);
  if (st != NF4Q_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return NF4Q_OK;
  const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const int b = static_cast<int>(kLutSmemTop);
  for (int dt = 0; dt < 2; ++dt)
    for (int dq = 0; dq < 2; ++dq)
      for (int bb = 4; bb <= 8; bb += 4)
        for (int v = 0; v < 4; ++v)
          if ((st = cuda_check(cudaFuncSetAttribute(
                   gemv_lut_kernel_for(dt, dq != 0, bb, (v & 1) != 0, (v & 2) != 0), A, b),
                   "cudaFuncSetAttribute (GEMV, folded)")) != NF4Q_OK)
            return st;
  done[dev] = true;
  return NF4Q_OK;
}

// Opt the dequantize kernels in to their dynamic shared memory (once per
// device).
nf4q_status dequantize_attr_ready() {
  static bool done[kMaxDevices] = {false};
  static std::mutex mu;
  int dev = 0;
  nf4q_status st = current_device(&dev);
  if (st != NF4Q_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return NF4Q_OK;
  const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const int b = static_cast<int>(kDequantSmemBytes);
  const char* what = "cudaFuncSetAttribute (dequantize)";
  if ((st = cuda_check(cudaFuncSetAttribute(dequantize_kernel<0, 0>, A, b), what)) != NF4Q_OK ||
      (st = cuda_check(cudaFuncSetAttribute(dequantize_kernel<1, 0>, A, b), what)) != NF4Q_OK ||
      (st = cuda_check(cudaFuncSetAttribute(dequantize_kernel<0, 1>, A, b), what)) != NF4Q_OK ||
      (st = cuda_check(cudaFuncSetAttribute(dequantize_kernel<1, 1>, A, b), what)) != NF4Q_OK)
    return st;
  done[dev] = true;
  return NF4Q_OK;
}

using QuantKernelFn = void (*)(const void*, uint2*, float*, int64_t, QuantParams,
                               DqWorkspace*, float*);

// The quantize instantiation for a code, input dtype (nf4q_in_dtype) and
// fused double-quant pass.
template <int CODE>
QuantKernelFn quantize_kernel_code(int in, int dq) {
  if (in == 1) return dq ? quantize_kernel<CODE, 1, true> : quantize_kernel<CODE, 1, false>;
  if (in == 2) return dq ? quantize_kernel<CODE, 2, true> : quantize_kernel<CODE, 2, false>;
  return dq ? quantize_kernel<CODE, 0, true> : quantize_kernel<CODE, 0, false>;
}
QuantKernelFn quantize_kernel_for(int code, int in, int dq) {
  return code == 0 ? quantize_kernel_code<0>(in, dq) : quantize_kernel_code<1>(in, dq);
}

// Opt the quantize kernels in to their dynamic shared memory (once per device).
nf4q_status quantize_attr_ready() {
  static bool done[kMaxDevices] = {false};
  static std::mutex mu;
  int dev = 0;
  nf4q_status st = current_device(&dev);
  if (st != NF4Q_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return NF4Q_OK;
  const int b0 = static_cast<int>(quantize_smem_bytes(0)), b1 = static_cast<int>(quantize_smem_bytes(1));
  const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
  for (int code = 0; code < 2; ++code)
    for (int in = 0; in < 3; ++in)
      for (int dq = 0; dq < 2; ++dq)
        if ((st = cuda_check(cudaFuncSetAttribute(quantize_kernel_for(code, in, dq), A,
                                                  code == 0 ? b0 : b1),
                             "cudaFuncSetAttribute (quantize)")) != NF4Q_OK)
          return st;
  done[dev] = true;
  return NF4Q_OK;
}

// Resident CTAs per SM of the quantize kernel (registers and shared memory),
// so the grid-stride grid is exactly one full wave.
int quantize_ctas_per_sm(int code) {
  static int cache[kMaxDevices][2] = {{0}};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][code] == 0) {
    int n = 0;
    const size_t smem = quantize_smem_bytes(code);
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, quantize_kernel_for(code, 1, 1), kQuantThreads, smem);
    cache[dev][code] = (e == cudaSuccess && n > 0) ? n : 1;
  }
  return cache[dev][code];
}

ScaleView scale_view(const nf4q_weight* wq) {
  ScaleView sv;
  sv.absmax_q = wq->absmax_q;
  sv.absmax = wq->absmax;
  sv.scale2 = wq->scale2;
  sv.offset = wq->offset;
  sv.double_quant = wq->double_quant;
  return sv;
}

CodeValues code_values(int code) {
  CodeValues C;
  for (int i = 0; i < 16; ++i) C.v[i] = tables().values[code][i];
  return C;
}

// fp16 bits (round to nearest even) of the 16 code values.
HalfCodes half_codes(int code) {
  HalfCodes H;
  for (int i = 0; i < 16; ++i) {
    const __half h = __float2half_rn(tables().values[code][i]);
    std::memcpy(&H.h[i], &h, sizeof(uint16_t));
  }
  return H;
}

int64_t grid_for(int64_t work_items, int64_t per_cta, int64_t cap) {
  int64_t g = (work_items + per_cta - 1) / per_cta;
  return std::max<int64_t>(1, std::min<int64_t>(g, cap));
}

}  // namespace
}  // namespace nf4q

using namespace nf4q;

extern "C" {

int32_t nf4q_version(void) { return (1 << 16) | 0; }

const char* nf4q_status_string(nf4q_status s) {
  switch (s) {
    case NF4Q_OK: return "ok";
    case NF4Q_ERR_INVALID_ARG: return "invalid argument";
    case NF4Q_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case NF4Q_ERR_UNSUPPORTED: return "unsupported configuration";
    case NF4Q_ERR_WORKSPACE: return "workspace missing or too small";
    case NF4Q_ERR_CUDA: return "CUDA error";
    case NF4Q_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int32_t nf4q_last_cuda_error(char* buf, int32_t buf_bytes) {
  const char* text = last_error_text();
  const int32_t n = static_cast<int32_t>(std::strlen(text));
  if (buf && buf_bytes > 0) {
    const int32_t m = std::min(n, buf_bytes - 1);
    std::memcpy(buf, text, static_cast<size_t>(m));
    buf[m] = '\0';
  }
  return n;
}

nf4q_status nf4q_sizes(int64_t rows, int64_t cols, int32_t blocksize,
                       int32_t dq_blocksize, size_t* packed_bytes, int64_t* n_b,
                       int64_t* n_d) {
  if (rows < 0 || cols < 0 || blocksize != kBlock || dq_blocksize != kDqBlock ||
      cols % kBlock != 0)
    return NF4Q_ERR_INVALID_ARG;
  if (cols > 0 && rows > INT64_MAX / cols) return NF4Q_ERR_UNSUPPORTED;  // rows*cols overflows
  const int64_t n = rows * cols;
  const int64_t nb = n / kBlock;
  if (packed_bytes) *packed_bytes = static_cast<size_t>(n / 2);
  if (n_b) *n_b = nb;
  if (n_d) *n_d = (nb + kDqBlock - 1) / kDqBlock;
  return NF4Q_OK;
}

nf4q_status nf4q_code_values(int32_t code, float* out) {
  if (!out || (code != NF4Q_CODE_NF4 && code != NF4Q_CODE_FP4)) return NF4Q_ERR_INVALID_ARG;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  for (int i = 0; i < 16; ++i) out[i] = tables().values[code][i];
  return NF4Q_OK;
}

nf4q_status nf4q_thresholds(int32_t code, float* out, int32_t* count) {
  if (!out || !count || (code != NF4Q_CODE_NF4 && code != NF4Q_CODE_FP4))
    return NF4Q_ERR_INVALID_ARG;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  const int n = tables().nthr[code];
  for (int i = 0; i < n; ++i) out[i] = tables().thr[code][i];
  *count = n;
  return NF4Q_OK;
}


}  // extern "C"

namespace nf4q {
namespace {
// Quantize launch after the argument checks common to both entry points
// (n > 0).  ws != nullptr: fused first double-quant pass into ws (zero on
// entry, left zero by the kernel's last CTA) and wq->offset.
nf4q_status quantize_launch(const void* w, int32_t in_dtype, const nf4q_weight* wq, void* ws,
                            cudaStream_t s) {
  const int64_t n = wq->rows * wq->cols;
  if (!w || !wq->packed || !wq->absmax) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(wq->packed) || !aligned16(wq->absmax))
    return NF4Q_ERR_ALIGNMENT;
  const HostTables& T = tables();
  if (!T.ok) return NF4Q_ERR_UNSUPPORTED;
  QuantParams P;
  const int c = wq->code;
  for (int i = 0; i < kLutEntries; ++i) {
    P.lut_t[i] = T.lut_t[c][i];
    P.lut_lo[i] = T.lut_lo[c][i];
    P.lut_dl[i] = T.lut_dl[c][i];
  }
  for (int i = 0; i < 15; ++i) P.thr[i] = i < T.nthr[c] ? T.thr[c][i] : 2.0f;
  nf4q_status st = quantize_attr_ready();
  if (st != NF4Q_OK) return st;
  const int64_t n_units = n / 16;  // 16 elements per lane and unit
  const int64_t grid = grid_for(n_units, kQuantThreads,
                                static_cast<int64_t>(sm_count()) * quantize_ctas_per_sm(c));
  // a programmatic dependent of the kernel before it (the kernel waits for
  // it before any global access), so that its table build overlaps that
  // kernel's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  return launch("quantize_kernel", quantize_kernel_for(c, in_dtype, ws != nullptr),
                dim3(static_cast<unsigned>(grid)), dim3(kQuantThreads), quantize_smem_bytes(c), s,
                attr, 1, w, reinterpret_cast<uint2*>(wq->packed), wq->absmax, n_units, P,
                static_cast<DqWorkspace*>(ws), wq->offset);
}

// Second double-quant pass: int8 codes and per-256 scales from the mean.
// `dependent`: launched as a programmatic dependent of the kernel before it
// on the stream (which signals griddepcontrol.launch_dependents), so its
// launch overlaps that kernel's tail.
nf4q_status dq_quant_launch(const nf4q_weight* wq, int64_t nb, cudaStream_t s,
                            bool dependent) {
  const int64_t nd = (nb + kDqBlock - 1) / kDqBlock;
  const int64_t g2 = grid_for(nd, kDqQuantThreads / 32, static_cast<int64_t>(sm_count()) * 8);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const float* am = wq->absmax;
  const float* off = wq->offset;
  return launch("dq_quant_kernel", dq_quant_kernel, dim3(static_cast<unsigned>(g2)),
                dim3(kDqQuantThreads), 0, s, attr, dependent ? 1u : 0u, am, nb, off,
                wq->absmax_q, wq->scale2);
}

// Both passes of the double quantization, on a zero workspace record (left
// zero by the first pass's last CTA).
nf4q_status dq_launch(const nf4q_weight* wq, int64_t nb, void* ws, cudaStream_t s) {
  nf4q_status st;
  const int64_t g1 = grid_for(nb / 4, kDqSumThreads, static_cast<int64_t>(sm_count()));
  st = launch("dq_sum_kernel", dq_sum_kernel, dim3(static_cast<unsigned>(g1)),
              dim3(kDqSumThreads), 0, s, nullptr, 0, static_cast<const float*>(wq->absmax), nb,
              static_cast<DqWorkspace*>(ws), wq->offset);
  if (st != NF4Q_OK) return st;
  return dq_quant_launch(wq, nb, s, false);
}
}  // namespace
}  // namespace nf4q

extern "C" {

nf4q_status nf4q_quantize(const void* w, int32_t in_dtype, const nf4q_weight* wq,
                          void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  if (in_dtype != NF4Q_IN_F32 && in_dtype != NF4Q_IN_BF16 && in_dtype != NF4Q_IN_F16)
    return NF4Q_ERR_INVALID_ARG;
  if (wq->rows * wq->cols == 0) return NF4Q_OK;
  return quantize_launch(w, in_dtype, wq, nullptr, static_cast<cudaStream_t>(stream));
}

size_t nf4q_double_quant_workspace_bytes(int64_t n_b) {
  (void)n_b;
  return sizeof(DqWorkspace);
}

nf4q_status nf4q_double_quant(const nf4q_weight* wq, void* workspace,
                              size_t workspace_bytes, void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  const int64_t nb = wq->rows * wq->cols / kBlock;
  if (!wq->absmax_q || !wq->scale2 || !wq->offset) return NF4Q_ERR_INVALID_ARG;
  if (!aligned4(wq->offset) || !aligned4(wq->scale2)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nb == 0) {
    return cuda_check(cudaMemsetAsync(wq->offset, 0, sizeof(float), s),
                      "cudaMemsetAsync (offset)");
  }
  if (!wq->absmax) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(wq->absmax) || !aligned16(wq->absmax_q)) return NF4Q_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < sizeof(DqWorkspace)) return NF4Q_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NF4Q_ERR_ALIGNMENT;
  return dq_launch(wq, nb, workspace, s);
}

nf4q_status nf4q_quantize_dq(const void* w, int32_t in_dtype, const nf4q_weight* wq,
                             void* workspace, size_t workspace_bytes, void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  if (in_dtype != NF4Q_IN_F32 && in_dtype != NF4Q_IN_BF16 && in_dtype != NF4Q_IN_F16)
    return NF4Q_ERR_INVALID_ARG;
  if (wq->double_quant != 1) return NF4Q_ERR_INVALID_ARG;
  if (!wq->absmax_q || !wq->scale2 || !wq->offset) return NF4Q_ERR_INVALID_ARG;
  if (!aligned4(wq->offset) || !aligned4(wq->scale2)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nb = wq->rows * wq->cols / kBlock;
  if (nb == 0)
    return cuda_check(cudaMemsetAsync(wq->offset, 0, sizeof(float), s),
                      "cudaMemsetAsync (offset)");
  if (!aligned16(wq->absmax_q)) return NF4Q_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < sizeof(DqWorkspace)) return NF4Q_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NF4Q_ERR_ALIGNMENT;
  if ((st = quantize_launch(w, in_dtype, wq, workspace, s)) != NF4Q_OK) return st;
  return dq_quant_launch(wq, nb, s, true);
}

nf4q_status nf4q_dequantize(const nf4q_weight* wq, void* out, void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  const int64_t n = wq->rows * wq->cols;
  if (n == 0) return NF4Q_OK;
  if ((st = check_scales(wq)) != NF4Q_OK) return st;
  if (!out) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(out)) return NF4Q_ERR_ALIGNMENT;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  if ((st = dequantize_attr_ready()) != NF4Q_OK) return st;
  const int64_t n_blocks = n / kBlock;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled: driver entry point not found");
  if ((st = ensure_context()) != NF4Q_OK) return st;
  CUtensorMap tout;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kBlock), static_cast<cuuint64_t>(n_blocks)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kBlock * 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlock), 32};
    cuuint32_t es[2] = {1, 1};
    st = cu_check(enc(&tout, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, out, dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled (dequantize output)");
    if (st != NF4Q_OK) return st;
  }
  const int64_t n_tiles = (n_blocks + 31) / 32;
  const int64_t grid = grid_for(n_tiles, kDequantWarps,
                                static_cast<int64_t>(sm_count()) * kDequantCtasPerSm);
  const uint4* pk = reinterpret_cast<const uint4*>(wq->packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  using DequantFn = void (*)(const uint4*, ScaleView, CUtensorMap, int64_t, CodeValues);
  const DequantFn k = wq->compute_dtype == NF4Q_DT_BF16
      ? (wq->code == NF4Q_CODE_NF4 ? dequantize_kernel<0, 0> : dequantize_kernel<1, 0>)
      : (wq->code == NF4Q_CODE_NF4 ? dequantize_kernel<0, 1> : dequantize_kernel<1, 1>);
  return launch("dequantize_kernel", k, dim3(static_cast<unsigned>(grid)), dim3(kDequantThreads),
                kDequantSmemBytes, s, nullptr, 0, pk, scale_view(wq), tout, n_blocks,
                code_values(wq->code));
}

}  // extern "C"

namespace nf4q {
namespace {

// Checks shared by both GEMV entry points.  *done = true when nothing (or
// only the y = 0 of an empty contraction) was to be launched.
nf4q_status gemv_checks(const nf4q_weight* wq, const void* x, int32_t M, void* y,
                        cudaStream_t s, bool* done) {
  *done = true;
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  if (M < 1 || M > NF4Q_GEMV_MAX_M) return NF4Q_ERR_UNSUPPORTED;
  if (wq->rows == 0) return NF4Q_OK;
  if (!x || !y) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return NF4Q_ERR_ALIGNMENT;
  if (wq->cols == 0) {  // empty contraction: y = 0
    return cuda_check(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * wq->rows * 2, s),
                      "cudaMemsetAsync (y of an empty contraction)");
  }
  if ((st = check_scales(wq)) != NF4Q_OK) return st;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  if (wq->rows > (1ll << 30) || wq->cols > (1ll << 30)) return NF4Q_ERR_UNSUPPORTED;
  *done = false;
  return NF4Q_OK;
}

// 2D tensor map of the packed weight [rows x cols/2 bytes], boxes of
// `box_rows` rows x 128 bytes with the 128-byte swizzle.
nf4q_status gemv_weight_map(const nf4q_weight* wq, int box_rows, CUtensorMap* tw) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled: driver entry point not found");
  nf4q_status st = ensure_context();
  if (st != NF4Q_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(wq->cols / 2), static_cast<cuuint64_t>(wq->rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(wq->cols / 2)};
  cuuint32_t box[2] = {kGemvSeg / 2, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return cu_check(enc(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq->packed, dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled (GEMV weight)");
}

// Packed weights of the folded GEMV as a 3-D view {128 bytes, rows, 128-byte
// columns of a row} when K is a multiple of 256 (the view then covers each
// row exactly): one copy brings a stage of 16 rows x (BB / 4) such columns,
// laid out column after column, each the 2 KB of 16 rows in the 128-byte
// swizzle - the layout of BB / 4 separate 2-D boxes, in one operation.
nf4q_status gemv_lut_weight_map(const nf4q_weight* wq, int depth, CUtensorMap* tw) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled: driver entry point not found");
  nf4q_status st = ensure_context();
  if (st != NF4Q_OK) return st;
  cuuint64_t dims[3] = {kGemvSeg / 2, static_cast<cuuint64_t>(wq->rows),
                        static_cast<cuuint64_t>(wq->cols / kGemvSeg)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(wq->cols / 2), kGemvSeg / 2};
  cuuint32_t box[3] = {kGemvSeg / 2, 16, static_cast<cuuint32_t>(depth)};
  cuuint32_t es[3] = {1, 1, 1};
  return cu_check(enc(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq->packed, dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled (folded GEMV weight)");
}

// Staged x of the folded GEMV: 64-blocks per row, a multiple of the box.
int64_t lut_kbx(int64_t K, int bb) { return (K / kBlock + bb - 1) / bb * bb; }

// Box size of the folded GEMV for this call: 8 blocks when x fits the room
// that layout leaves it, else 4; 0 when the folded GEMV does not take the
// call (M > 8, or x does not fit at all).
int lut_box(int64_t K, int32_t M) {
  if (M > kLutMaxM) return 0;
  if (static_cast<int64_t>(M) * lut_kbx(K, 8) * 128 <= kLutXBytes8) return 8;
  if (static_cast<int64_t>(M) * lut_kbx(K, 4) * 128 <= kLutXBytes4) return 4;
  return 0;
}

// The kernel numbers tiles, a CTA's boxes and its warps' runs in 32-bit
// ints: T x grid and (tiles of the largest CTA) x (boxes per row) x 16 must
// stay below 2^31.
bool lut_runs_fit(int64_t T, int64_t K, int bb, int64_t grid) {
  const int64_t nbox = (K / kBlock + bb - 1) / bb;
  return grid > 0 && T * grid < (int64_t{1} << 31) &&
         (T + grid - 1) / grid * nbox * kLutWarps < (int64_t{1} << 31);
}

// The block-scale-folded GEMV (gemv_lut.cuh) over a group of 1..4 weights
// with the same cols, code, double quant and compute dtype, sharing x.
// One CTA per SM (at most one per 16-row tile); the kernel splits each
// CTA's tiles into equal runs of boxes over its warps.  flags: the
// nf4q_gemv_multi_ex flags (NF4Q_GEMV_WEIGHTS_STATIC).
nf4q_status gemv_lut_launch(const nf4q_weight* const* wq, int count, const void* x, int32_t M,
                            void* const* y, cudaStream_t s, int32_t flags) {
  nf4q_status st = gemv_lut_attr_ready();
  if (st != NF4Q_OK) return st;
  const int K = static_cast<int>(wq[0]->cols);
  const int bb = lut_box(K, M);
  LutGroup G;
  std::memset(&G, 0, sizeof(G));
  G.count = count;
  G.map3d = K % kGemvSeg == 0 ? 1 : 0;
  int64_t T = 0;
  for (int i = 0; i < count; ++i) {
    G.off[i] = static_cast<int>(T);
    G.N[i] = static_cast<int>(wq[i]->rows);
    G.sv[i] = scale_view(wq[i]);
    G.y[i] = static_cast<uint16_t*>(y[i]);
    st = G.map3d ? gemv_lut_weight_map(wq[i], bb / 4, &G.tmap[i])
                 : gemv_weight_map(wq[i], 16, &G.tmap[i]);
    if (st != NF4Q_OK) return st;
    T += (wq[i]->rows + 15) / 16;
  }
  for (int i = count; i <= kLutMaxGroup; ++i) G.off[i] = static_cast<int>(T);
  const int64_t grid = std::min<int64_t>(sm_count(), T);
  if (!lut_runs_fit(T, K, bb, grid)) return NF4Q_ERR_UNSUPPORTED;
  const auto k = gemv_lut_kernel_for(wq[0]->compute_dtype == NF4Q_DT_BF16 ? 0 : 1,
                                     wq[0]->double_quant != 0, bb, (K / kBlock) % 16 == 0,
                                     M == 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  return launch("gemv_lut_kernel", k, dim3(static_cast<unsigned>(grid)), dim3(kLutThreads),
                kLutSmemTop, s, attr, 1, G, static_cast<const uint16_t*>(x), K,
                static_cast<int>(M), static_cast<int>(lut_kbx(K, bb)),
                half_codes(wq[0]->code), (flags & NF4Q_GEMV_WEIGHTS_STATIC) ? 1 : 0);
}

// The bit-faithful GEMV (gemv_mma.cuh): w_hat rebuilt exactly inside the
// contraction.
nf4q_status gemv_exact_launch(const nf4q_weight* wq, const void* x, int32_t M, void* y,
                              cudaStream_t s) {
  nf4q_status st;
  const int N = static_cast<int>(wq->rows), K = static_cast<int>(wq->cols);
  if ((st = gemv_attr_ready()) != NF4Q_OK) return st;
  // M <= 4: one 8-column MMA tile and 16 rows per CTA; M = 5..8: 32 rows,
  // so each x fragment (by then up to eight distinct rows of x) serves twice
  // as many weights; M > 8: two column tiles and 32 rows.  FP4, whose lookup
  // is cheaper, takes 32 rows from M = 2 when those tiles alone give every SM
  // its four CTAs (measured on 28672 x 8192: 69.1 -> 57.2 us at M = 4); with
  // fewer rows the K split it would need costs more than it saves.
  const int code = wq->code == NF4Q_CODE_NF4 ? 0 : 1;
  const bool fp4_wide = code == 1 && M > 1 &&
                        (N + 2 * kGemvRows - 1) / (2 * kGemvRows) >=
                            static_cast<int64_t>(kGemvMinCtasPerSm) * sm_count();
  const int NT = M > 8 ? 2 : 1, R = M > 4 || fp4_wide ? 2 : 1;
  const int64_t tiles = (N + kGemvRows * R - 1) / (kGemvRows * R);
  const int nseg = (K + kGemvSeg - 1) / kGemvSeg;
  const int nchunks = (nseg + kGemvWarps - 1) / kGemvWarps;
  // K split over a cluster: the smallest that gives every SM at least four
  // CTAs (16 warps); the ring has two stages, which leaves room for eight
  // CTAs per SM (measured best on 4096^2 .. 28672x8192 weights).
  int split = 1;
  while (split < std::min(kGemvMaxSplit, nchunks) &&
         tiles * split < static_cast<int64_t>(kGemvMinCtasPerSm) * sm_count())
    split *= 2;
  const int per = (nchunks + split - 1) / split;
  split = (nchunks + per - 1) / per;  // CTAs that get chunks
  const int stages = std::min(kGemvStages, per);
  const size_t smem = gemv_smem_bytes(R, NT, stages, split);
  CUtensorMap tw;
  if ((st = gemv_weight_map(wq, kGemvRows * R, &tw)) != NF4Q_OK) return st;
  if (tiles * split > 0x7FFFFFFF) return NF4Q_ERR_UNSUPPORTED;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  uint16_t* yp = static_cast<uint16_t*>(y);
  const ScaleView sv = scale_view(wq);
  const CodeValues C = code_values(wq->code);
  return launch("gemv_mma_kernel", gemv_kernel(code, NT, R, wq->compute_dtype),
                dim3(static_cast<unsigned>(tiles * split)), dim3(kGemvWarps * 32), smem, s, attr,
                split > 1 ? 1u : 0u, tw, sv, xp, yp, N, K, static_cast<int>(M), per, stages, C);
}

// One weight: the folded kernel where it applies (M <= NF4Q_GEMV_FOLD_MAX_M,
// x fits its staging room, run arithmetic in 32 bits), else the exact one.
nf4q_status gemv_one(const nf4q_weight* wq, const void* x, int32_t M, void* y, cudaStream_t s,
                     int32_t flags) {
  bool done = false;
  nf4q_status st = gemv_checks(wq, x, M, y, s, &done);
  if (st != NF4Q_OK || done) return st;
  if (M <= NF4Q_GEMV_FOLD_MAX_M && lut_box(wq->cols, M) &&
      lut_runs_fit((wq->rows + 15) / 16, wq->cols, lut_box(wq->cols, M),
                   std::min<int64_t>(sm_count(), (wq->rows + 15) / 16)))
    return gemv_lut_launch(&wq, 1, x, M, &y, s, flags);
  return gemv_exact_launch(wq, x, M, y, s);
}

}  // namespace
}  // namespace nf4q

extern "C" {

nf4q_status nf4q_gemv(const nf4q_weight* wq, const void* x, int32_t M, void* y,
                      void* stream) {
  return nf4q::gemv_one(wq, x, M, y, static_cast<cudaStream_t>(stream), 0);
}

nf4q_status nf4q_gemv_multi(const nf4q_weight* const* wq, int32_t count, const void* x,
                            int32_t M, void* const* y, void* stream) {
  return nf4q_gemv_multi_ex(wq, count, x, M, y, 0, stream);
}

nf4q_status nf4q_gemv_multi_ex(const nf4q_weight* const* wq, int32_t count, const void* x,
                               int32_t M, void* const* y, int32_t flags, void* stream) {
  if ((flags & ~NF4Q_GEMV_WEIGHTS_STATIC) != 0) return NF4Q_ERR_INVALID_ARG;
  if (!wq || !y || count < 1 || count > kLutMaxGroup) return NF4Q_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    if (!wq[i]) return NF4Q_ERR_INVALID_ARG;
    nf4q_status st = check_shape(wq[i]);
    if (st != NF4Q_OK) return st;
    if (wq[i]->cols != wq[0]->cols || wq[i]->code != wq[0]->code ||
        wq[i]->double_quant != wq[0]->double_quant ||
        wq[i]->compute_dtype != wq[0]->compute_dtype)
      return NF4Q_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one launch when the folded GEMV takes the call and every weight is
  // non-empty; else the weights one by one
  bool one = lut_box(wq[0]->cols, M) != 0 && wq[0]->cols > 0;
  for (int i = 0; i < count && one; ++i) {
    bool done = false;
    nf4q_status st = gemv_checks(wq[i], x, M, y[i], s, &done);
    if (st != NF4Q_OK) return st;
    one = !done;
  }
  if (!one) {
    for (int i = 0; i < count; ++i) {
      nf4q_status st = nf4q::gemv_one(wq[i], x, M, y[i], s, flags);
      if (st != NF4Q_OK) return st;
    }
    return NF4Q_OK;
  }
  int64_t tiles = 0;
  for (int i = 0; i < count; ++i) tiles += (wq[i]->rows + 15) / 16;
  if (tiles > 0x7FFFFFFF) return NF4Q_ERR_UNSUPPORTED;
  return gemv_lut_launch(wq, count, x, M, y, s, flags);
}

nf4q_status nf4q_gemv_exact(const nf4q_weight* wq, const void* x, int32_t M, void* y,
                            void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool done = false;
  nf4q_status st = gemv_checks(wq, x, M, y, s, &done);
  if (st != NF4Q_OK || done) return st;
  return gemv_exact_launch(wq, x, M, y, s);
}

nf4q_status nf4q_gemm(const nf4q_weight* wq, const void* X, int64_t M, void* Y,
                      void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  if (M < 0) return NF4Q_ERR_INVALID_ARG;
  if (M == 0 || wq->rows == 0) return NF4Q_OK;
  if (!X || !Y) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Y)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (wq->cols == 0) {
    return cuda_check(cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * wq->rows * 2, s),
                      "cudaMemsetAsync (Y of an empty contraction)");
  }
  if ((st = check_scales(wq)) != NF4Q_OK) return st;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  return gemm_launch(wq, scale_view(wq), code_values(wq->code), X, M, Y, s, sm_count());
}

nf4q_status nf4q_matmul_dx(const nf4q_weight* wq, const void* dY, int64_t ld_dy, int64_t M,
                           void* dX, void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  if (M < 0 || ld_dy < wq->rows || ld_dy % 8 != 0) return NF4Q_ERR_INVALID_ARG;
  if (M == 0 || wq->cols == 0) return NF4Q_OK;
  if (!dY || !dX) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(dY) || !aligned16(dX)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (wq->rows == 0) {  // empty contraction: dX = 0
    return cuda_check(cudaMemsetAsync(dX, 0, static_cast<size_t>(M) * wq->cols * 2, s),
                      "cudaMemsetAsync (dX of an empty contraction)");
  }
  if ((st = check_scales(wq)) != NF4Q_OK) return st;
  if (!tables().ok) return NF4Q_ERR_UNSUPPORTED;
  return gemm_dx_launch(wq, scale_view(wq), code_values(wq->code), dY, ld_dy, M, dX, s,
                        sm_count());
}

nf4q_status nf4q_matmul(const nf4q_weight* wq, const void* X, int64_t M, void* Y,
                        void* stream) {
  // M = 9..16 on weights with at least NF4Q_MATMUL_GEMM_ROWS rows: the GEMM,
  // whose tiles then still fit one wave of the SMs (measured on a B300,
  // 28672x8192: 72.4 us against 74.6..88.3 us for the GEMV; on 4096- to
  // 14336-row weights the GEMV stays ahead or even)
  const bool gemm_wins = M > 8 && wq && wq->rows >= NF4Q_MATMUL_GEMM_ROWS;
  if (M >= 1 && M <= NF4Q_GEMV_MAX_M && !gemm_wins)
    return nf4q_gemv(wq, X, static_cast<int32_t>(M), Y, stream);
  return nf4q_gemm(wq, X, M, Y, stream);
}

nf4q_status nf4q_device_error(uint32_t* flags, int32_t clear) {
  if (!flags) return NF4Q_ERR_INVALID_ARG;
  nf4q_status st = cuda_check(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (st != NF4Q_OK) return st;
  st = cuda_check(cudaMemcpyFromSymbol(flags, g_device_error, sizeof(uint32_t)),
                  "cudaMemcpyFromSymbol (device error word)");
  if (st != NF4Q_OK || !clear) return st;
  const uint32_t zero = 0;
  return cuda_check(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t)),
                    "cudaMemcpyToSymbol (device error word)");
}

// ---------------------------------------------------------------- no-alloc
// Static scratch of nf4q_double_quant_noalloc, zero when the module loads and
// left zero by every call.  In host code the symbol is only a handle: its
// device address comes from cudaGetSymbolAddress, looked up once per device
// with that device current.
static __device__ __align__(256) unsigned char g_dq_noalloc_scratch[256] = {};
static_assert(sizeof(DqWorkspace) <= 256, "double-quant record must fit the static scratch");

namespace {
// The scratch's device address in the current context, looked up with
// cudaGetSymbolAddress the first time a device is used and again whenever the
// current context is not the one the cached address belongs to (a device
// reset, or another context made current on the device).
void* noalloc_scratch(nf4q_status* st) {
  static void* addr[kMaxDevices] = {nullptr};
  static unsigned long long ctx_of[kMaxDevices] = {0};
  static std::mutex mu;
  int dev = 0;
  if ((*st = current_device(&dev)) != NF4Q_OK) return nullptr;
  if ((*st = ensure_context()) != NF4Q_OK) return nullptr;
  unsigned long long ctx = 0;
  if ((*st = current_context_id(&ctx)) != NF4Q_OK) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx_of[dev] != ctx) {
    void* p = nullptr;
    *st = cuda_check(cudaGetSymbolAddress(&p, g_dq_noalloc_scratch), "cudaGetSymbolAddress");
    if (*st != NF4Q_OK) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *st = NF4Q_OK;
  return addr[dev];
}
}  // namespace

nf4q_status nf4q_double_quant_noalloc(const nf4q_weight* wq, void* stream) {
  nf4q_status st = check_shape(wq);
  if (st != NF4Q_OK) return st;
  const int64_t nb = wq->rows * wq->cols / kBlock;
  if (!wq->absmax_q || !wq->scale2 || !wq->offset) return NF4Q_ERR_INVALID_ARG;
  if (!aligned4(wq->offset) || !aligned4(wq->scale2)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nb == 0) {
    return cuda_check(cudaMemsetAsync(wq->offset, 0, sizeof(float), s),
                      "cudaMemsetAsync (offset)");
  }
  if (!wq->absmax) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(wq->absmax) || !aligned16(wq->absmax_q)) return NF4Q_ERR_ALIGNMENT;
  void* ws = noalloc_scratch(&st);
  if (st != NF4Q_OK) return st;
  return dq_launch(wq, nb, ws, s);
}


// ---------------------------------------------------------------- LLM.int8()
namespace {
nf4q_status check_int8_weight(const nf4q_int8_weight* wq) {
  if (!wq || wq->rows < 0 || wq->cols < 0 || wq->cols % 16 != 0) return NF4Q_ERR_INVALID_ARG;
  // the kernels step int column indices by up to a few thousand past cols
  if (wq->rows > 0x7FFFFFFF || wq->cols > (1ll << 30)) return NF4Q_ERR_UNSUPPORTED;
  return NF4Q_OK;
}
}  // namespace

nf4q_status nf4q_int8_quantize_weight(const void* w, int32_t in_dtype,
                                      const nf4q_int8_weight* wq, void* stream) {
  nf4q_status st = check_int8_weight(wq);
  if (st != NF4Q_OK) return st;
  if (in_dtype != NF4Q_IN_BF16 && in_dtype != NF4Q_IN_F16) return NF4Q_ERR_INVALID_ARG;
  if (wq->rows == 0) return NF4Q_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!wq->scale) return NF4Q_ERR_INVALID_ARG;
  if (!aligned4(wq->scale)) return NF4Q_ERR_ALIGNMENT;
  if (wq->cols == 0)
    return cuda_check(cudaMemsetAsync(wq->scale, 0, sizeof(float) * wq->rows, s),
                      "cudaMemsetAsync (int8 scales of empty rows)");
  if (!w || !wq->q) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(wq->q)) return NF4Q_ERR_ALIGNMENT;
  const auto k = in_dtype == NF4Q_IN_BF16 ? int8_quant_weight_kernel<1>
                                          : int8_quant_weight_kernel<2>;
  return launch("int8_quant_weight_kernel", k, dim3(static_cast<unsigned>(wq->rows)),
                dim3(kI8Threads), 0, s, nullptr, 0, static_cast<const uint16_t*>(w), wq->q,
                wq->scale, static_cast<int>(wq->cols));
}

size_t nf4q_int8_workspace_bytes(int64_t M, int64_t cols) {
  if (M < 0 || cols < 0) return 0;
  return int8_workspace_layout(M, cols).total;
}

nf4q_status nf4q_int8_matmul(const nf4q_int8_weight* wq, const void* X, int64_t M,
                             float threshold, void* Y, void* workspace,
                             size_t workspace_bytes, void* stream) {
  nf4q_status st = check_int8_weight(wq);
  if (st != NF4Q_OK) return st;
  if (M < 0) return NF4Q_ERR_INVALID_ARG;
  if (M == 0 || wq->rows == 0) return NF4Q_OK;
  if (M > 0x7FFFFFFF || (M + 15) / 16 > 65535) return NF4Q_ERR_UNSUPPORTED;
  if (!X || !Y) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Y)) return NF4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t N = wq->rows, K = wq->cols;
  if (K == 0)
    return cuda_check(cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * N * 2, s),
                      "cudaMemsetAsync (Y of an empty contraction)");
  if (!wq->q || !wq->scale) return NF4Q_ERR_INVALID_ARG;
  if (!aligned16(wq->q) || !aligned4(wq->scale)) return NF4Q_ERR_ALIGNMENT;
  const Int8Workspace L = int8_workspace_layout(M, K);
  if (!workspace || workspace_bytes < L.total) return NF4Q_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NF4Q_ERR_ALIGNMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* flags = ws + L.flags;
  int32_t* count = reinterpret_cast<int32_t*>(ws + L.count);
  int32_t* list = reinterpret_cast<int32_t*>(ws + L.list);
  float* sx = reinterpret_cast<float*>(ws + L.sx);
  uint16_t* xq = reinterpret_cast<uint16_t*>(ws + L.xq);
  const uint16_t* x = static_cast<const uint16_t*>(X);
  const int Mi = static_cast<int>(M), Ni = static_cast<int>(N), Ki = static_cast<int>(K);
  const float thr = threshold > 0.f ? threshold : 0.f;  // NaN -> 0: no decomposition
  // the activation side: flags, ordered outlier list, row scales and codes
  if (M <= 16) {
    st = launch("int8_act_small_kernel", int8_act_small_kernel, dim3(1), dim3(1024), 0, s,
                nullptr, 0, x, Mi, Ki, thr, flags, list, count, sx, xq);
  } else {
    st = launch("int8_outlier_flags_kernel", int8_outlier_flags_kernel,
                dim3(static_cast<unsigned>((K + 255) / 256)), dim3(kI8Threads), 0, s, nullptr, 0,
                x, Mi, Ki, thr, flags);
    if (st == NF4Q_OK)
      st = launch("int8_outlier_list_kernel", int8_outlier_list_kernel, dim3(1), dim3(1024), 0, s,
                  nullptr, 0, static_cast<const uint8_t*>(flags), Ki, list, count);
    if (st == NF4Q_OK)
      st = launch("int8_quant_act_kernel", int8_quant_act_kernel,
                  dim3(static_cast<unsigned>(M)), dim3(kI8Threads), 0, s, nullptr, 0, x,
                  static_cast<const uint8_t*>(flags), Ki, sx, xq);
  }
  if (st != NF4Q_OK) return st;
  const int nt = M > 8 ? 2 : 1;
  const dim3 grid(static_cast<unsigned>((N + kI8Rows - 1) / kI8Rows),
                  static_cast<unsigned>((M + 8 * nt - 1) / (8 * nt)));
  const auto k = nt == 2 ? int8_mm_kernel<2> : int8_mm_kernel<1>;
  return launch("int8_mm_kernel", k, grid, dim3(kI8Threads), 0, s, nullptr, 0,
                static_cast<const int8_t*>(wq->q), static_cast<const float*>(wq->scale), x,
                static_cast<const uint16_t*>(xq), static_cast<const float*>(sx),
                static_cast<const int32_t*>(list), static_cast<const int32_t*>(count),
                static_cast<uint16_t*>(Y), Ni, Ki, Mi);
}

}  // extern "C"
