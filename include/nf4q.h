/*
 * nf4q - NF4 / FP4 blockwise weight quantization with double quantization,
 * and the "4-bit stored, 16-bit computed" matmul, for NVIDIA B300 (sm_103a).
 *
 * Plain C ABI.  Every pointer in a compute call is a DEVICE pointer unless
 * the comment says "host"; every `stream` is a cudaStream_t passed as void*
 * (NULL = the legacy default stream).  Sizes are element counts unless they
 * end in `_bytes`.
 *
 * Where the operations come from (web pages about the bitsandbytes library):
 *   - "bitsandbytes tutorial" (mlqm.cn/news/394670)
 *       sec. 2.3  data-free absmax quantization, one scale per block
 *       sec. 3.2  NF4: 16 levels spaced by the normal density
 *       sec. 3.3  double quantization: the block scales quantized again
 *       sec. 3.4  compute dtype: 4-bit storage, dequantize to bf16, matmul
 *       sec. 四   config keys: quant type nf4|fp4, double quant, compute dtype
 *       sec. 5.4  QLoRA: the 4-bit base is frozen, LoRA adapters train
 *   - "bitsandbytes introduction" (modelers.csdn.net), sec. 一 item 7 and
 *       sec. 三 examples 1-2: NF4 and FP4 4-bit types
 *   - "bitsandbytes: quantifier un modèle PyTorch sans quitter PyTorch"
 *       (hysenlabs.com): blockwise quantization, Linear4bit layers
 *
 * Ownership: the caller allocates every buffer (including workspaces) and
 * keeps it alive until the work enqueued on `stream` has finished.  The
 * library never allocates device memory, never synchronizes the stream and
 * never calls exit/abort or executes a device trap.  Inputs marked const are
 * never written.  Outputs must not alias inputs.
 *
 * Errors: arguments are checked on the host before anything is launched
 * (a failing check launches nothing).  A failing CUDA call (a launch, a
 * memset, the tensor-map encoder) is reported as NF4Q_ERR_CUDA, and its text
 * is kept for nf4q_last_cuda_error().  The status of a launch is that
 * launch's own: the thread's sticky CUDA "last error", which other code on
 * the thread may have set, is never read.  Every entry point may be called
 * from any host thread.  Device-side bounded waits that give up set a sticky flag
 * read with nf4q_device_error().
 *
 * Layout of a quantized weight W [rows x cols] (row-major, cols contiguous,
 * the nn.Linear [out, in] convention):
 *   packed    uint8 [rows*cols/2]: element 2i -> bits 7..4 of byte i,
 *             element 2i+1 -> bits 3..0 (4-bit code, see below)
 *   absmax    fp32  [n_b]  n_b = rows*cols/64, max |w| of each run of 64
 *             consecutive elements (cols % 64 == 0, so a block never
 *             straddles two rows)
 *   absmax_q  int8  [n_b]  double-quantized absmax
 *   scale2    fp32  [n_d]  n_d = ceil(n_b/256), one per 256 absmax values
 *   offset    fp32  [1]    mean of absmax (see nf4q_double_quant)
 * Codes: NF4 - index 0..15 of the 16 ascending NF4 levels (0 is code 7,
 * +1 is code 15); FP4 - (sign << 3) | j, j indexing the E2M1 magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}/6.
 */
#ifndef NF4Q_H_
#define NF4Q_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden visibility; the entry points below are
 * the only exported symbols. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
  NF4Q_OK = 0,
  NF4Q_ERR_INVALID_ARG = 1,  /* null pointer, bad size, unsupported blocksize */
  NF4Q_ERR_ALIGNMENT = 2,    /* a pointer is not 16-byte aligned */
  NF4Q_ERR_UNSUPPORTED = 3,  /* valid but not implemented (e.g. M range) */
  NF4Q_ERR_WORKSPACE = 4,    /* workspace null or too small */
  NF4Q_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  NF4Q_ERR_TIMEOUT = 6       /* a bounded device wait gave up */
} nf4q_status;

typedef enum { NF4Q_CODE_NF4 = 0, NF4Q_CODE_FP4 = 1 } nf4q_code;
/* dtype of the weight given to nf4q_quantize / nf4q_quantize_dq */
typedef enum { NF4Q_IN_F32 = 0, NF4Q_IN_BF16 = 1, NF4Q_IN_F16 = 2 } nf4q_in_dtype;
/* Compute dtype (tutorial sec. 四, bnb_4bit_compute_dtype): the type of the
 * dequantized weights, of x and of y.  w_hat = round(fp32(code_value * s_b))
 * to this type (nearest, ties to even; fp16 overflows to infinity). */
typedef enum { NF4Q_DT_BF16 = 0, NF4Q_DT_F16 = 1 } nf4q_compute_dtype;

/* Views into caller-owned device buffers describing one quantized weight. */
typedef struct {
  uint8_t* packed;      /* [rows*cols/2]                                    */
  int8_t* absmax_q;     /* [n_b]  used when double_quant == 1               */
  float* absmax;        /* [n_b]  written by nf4q_quantize; the stored scale
                           when double_quant == 0                           */
  float* scale2;        /* [n_d]  used when double_quant == 1               */
  float* offset;        /* [1]    used when double_quant == 1               */
  int64_t rows;         /* N (output features)                              */
  int64_t cols;         /* K (input features), K % 64 == 0                  */
  int32_t blocksize;    /* must be 64                                       */
  int32_t dq_blocksize; /* must be 256                                      */
  int32_t code;         /* nf4q_code                                        */
  int32_t double_quant; /* 1: dequantizers use absmax_q/scale2/offset;
                           0: they use the fp32 absmax                      */
  int32_t compute_dtype; /* nf4q_compute_dtype of nf4q_dequantize's output
                            and of x / y of nf4q_gemv, _gemm, _matmul;
                            0 (bf16) for callers that zero the struct       */
} nf4q_weight;

/* Library version, (major << 16) | minor. */
int32_t nf4q_version(void);

/* Human-readable name of a status (static string, never NULL). */
const char* nf4q_status_string(nf4q_status s);

/* HOST ONLY.  The last CUDA failure of a call on the CALLING THREAD: the
 * failing runtime or driver call and the error's name and text, e.g.
 * "dequantize_kernel: cudaErrorInvalidValue (1): invalid argument"; "" if no
 * call on this thread has returned NF4Q_ERR_CUDA.  Copies at most
 * buf_bytes - 1 characters and a terminating NUL into buf (buf may be NULL
 * when buf_bytes is 0) and returns the length of the whole text.  The text
 * stays until the next failure on the same thread. */
int32_t nf4q_last_cuda_error(char* buf, int32_t buf_bytes);

/* HOST ONLY.  Buffer sizes of a [rows x cols] weight: packed bytes, number of
 * 64-blocks n_b and of 256-blocks n_d.  Any output pointer may be NULL.
 * NF4Q_ERR_INVALID_ARG for negative sizes, cols not a multiple of 64 or other
 * block sizes; NF4Q_ERR_UNSUPPORTED when rows*cols does not fit in int64_t
 * (nothing is written then). */
nf4q_status nf4q_sizes(int64_t rows, int64_t cols, int32_t blocksize,
                       int32_t dq_blocksize, size_t* packed_bytes,
                       int64_t* n_b, int64_t* n_d);

/* HOST ONLY.  The 16 code values (float32, indexed by code) the kernels use,
 * built by the library itself: NF4 from its definition (Phi^-1 of 8 points
 * evenly spaced from 0.9677083 down to 0.5 for the positive side, of 7 for
 * the negative side, plus 0, normalized by the largest; tutorial sec. 3.2),
 * FP4 from the E2M1 magnitudes. `out` is a host array of 16 floats. */
nf4q_status nf4q_code_values(int32_t code, float* out);

/* HOST ONLY.  The decision thresholds of the encoder: the largest float32 not
 * above the exact midpoint of each pair of neighbouring levels (15 for NF4,
 * 7 magnitude thresholds for FP4).  `out` is a host array of at least 15
 * floats; `*count` receives 15 or 7. */
nf4q_status nf4q_thresholds(int32_t code, float* out, int32_t* count);

/* Blockwise quantization (tutorial sec. 2.3 absmax, sec. 3.2 NF4; FP4 per the
 * introduction page, sec. 一 item 7).
 *   w      device, [rows x cols] row-major, fp32, bf16 or fp16 per `in_dtype`
 *          (widened to fp32 exactly), 16-byte aligned.  Values must be finite.
 *   wq     host struct; wq->packed and wq->absmax are written (both 16-byte
 *          aligned); rows, cols, blocksize, code are read.
 * Per 64-block: absmax = max|w| (fp32); wn = fp32(w / absmax) (IEEE
 * division; 0 when absmax == 0); code = the nearest level, an exact tie
 * going to the lower NF4 index / the smaller FP4 magnitude; two codes per
 * byte, first element in the high nibble. */
nf4q_status nf4q_quantize(const void* w, int32_t in_dtype,
                          const nf4q_weight* wq, void* stream);

/* Workspace bytes nf4q_double_quant needs for n_b absmax values (>= 64). */
size_t nf4q_double_quant_workspace_bytes(int64_t n_b);

/* Double quantization of the scales (tutorial sec. 3.3).
 *   reads wq->absmax [n_b]; writes wq->absmax_q [n_b], wq->scale2 [n_d],
 *   wq->offset [1].  absmax must be 16-byte aligned.
 *   workspace: device, >= nf4q_double_quant_workspace_bytes(n_b) bytes,
 *   16-byte aligned, zero-filled before its first use (one cudaMemset).
 *   Every call leaves it zero-filled again (the kernel that reads the sums
 *   clears them), so successive calls on one stream reuse it without
 *   clearing; a workspace that is not zero gives a wrong offset.  Calls whose
 *   work overlaps on the GPU (other streams) need workspaces of their own.
 * offset = the float32 nearest to the exact mean of all absmax values (ties
 * to even; the sum is exact for any inputs); c = fp32(absmax - offset); per
 * 256-block scale2 = fp32(max|c| / 127); absmax_q = clamp(rint_even(
 * fp32(c / scale2)), -127, 127), 0 where scale2 == 0. */
nf4q_status nf4q_double_quant(const nf4q_weight* wq, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Blockwise quantization followed by double quantization, in one call (the
 * stored form with double quant on, tutorial sec. 2.3, 3.2 and 3.3).  The
 * results are bit for bit those of nf4q_quantize followed by
 * nf4q_double_quant on the same arguments; the first double-quant pass (the
 * exact mean) runs inside the quantize kernel, so only the per-256 pass is a
 * second launch.
 *   w, in_dtype  as for nf4q_quantize.
 *   wq   wq->double_quant must be 1; writes packed, absmax, absmax_q,
 *        scale2 and offset (alignments as for the two calls).
 *   workspace  as for nf4q_double_quant (zero on entry, left zero). */
nf4q_status nf4q_quantize_dq(const void* w, int32_t in_dtype, const nf4q_weight* wq,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Dequantization to the compute dtype (tutorial sec. 3.4).
 *   out: device [rows x cols] of wq->compute_dtype (bf16 or fp16), 16-byte
 *   aligned.
 * s_b = fmaf(absmax_q[b], scale2[b/256], offset) with double quant, else
 * absmax[b]; out = round(fp32(code_value[code] * s_b)) to the compute dtype
 * (nearest, ties to even). */
nf4q_status nf4q_dequantize(const nf4q_weight* wq, void* out, void* stream);

/* Decode-shaped matmul, 1 <= M <= 16 (tutorial sec. 3.4, sec. 七 myth 5:
 * memory-bandwidth bound): y[m, n] = sum_k x[m, k] * w_hat[n, k], fp32
 * accumulation, output rounded to the compute dtype.
 *   x: device [M x cols], y: device [M x rows], both of wq->compute_dtype
 *   (bf16 or fp16) and 16-byte aligned.
 * For M <= NF4Q_GEMV_FOLD_MAX_M (when M * cols <= 30720, the staging room
 * for x) the block scale is folded:
 * y = sum_b s_b * sum_{k in b} x_k * code_value[code_k],
 * with the code values rounded to fp16 and x converted to fp16 after a
 * power-of-two scaling per row (exact for every bf16 x within 2^31 of its
 * row's largest |x|).  This differs from x . w_hat^T only by the rounding of
 * w_hat = bf16(code_value * s_b) and of the code values: at most 2^-8 + 2^-11
 * of |x_k w_hat_k| per term (fp16 compute dtype: 2^-10), signed like those
 * roundings.
 * Other calls, and nf4q_gemv_exact always, use w_hat itself (measured on a
 * B300: the folded kernel is faster up to M = 6 wherever x fits - by up to
 * 40 % at M = 1 and 25 % at M = 5..6 on 14336 x 4096 - and within 0.5 us
 * behind on 4096 x 4096 NF4; beyond M = 6 x fits only for short rows). */
#define NF4Q_GEMV_FOLD_MAX_M 6
nf4q_status nf4q_gemv(const nf4q_weight* wq, const void* x, int32_t M,
                      void* y, void* stream);

/* nf4q_gemv over a group of 1..4 weights that share x (q, k and v of an
 * attention block, gate and up of an MLP): y[i] = x . w_hat_i^T for each,
 * in one launch of the block-scale-folded GEMV when M <= 8 and x fits its
 * staging room (numerics as the folded nf4q_gemv above, for any such M);
 * else the weights go one by one through nf4q_gemv.  wq: host array of `count` weight pointers, all with the same
 * cols, code, double_quant and compute_dtype (NF4Q_ERR_INVALID_ARG
 * otherwise); y: host array of `count` device outputs [M x rows_i].  Other
 * arguments and errors as nf4q_gemv. */
nf4q_status nf4q_gemv_multi(const nf4q_weight* const* wq, int32_t count, const void* x,
                            int32_t M, void* const* y, void* stream);

/* nf4q_gemv_multi with flags (0 = nf4q_gemv_multi itself; any bit other than
 * those below: NF4Q_ERR_INVALID_ARG).
 *
 * NF4Q_GEMV_WEIGHTS_STATIC: the caller guarantees that no kernel that may
 * still be running when this call's kernel starts writes the weights -
 * their packed codes and every scale array (absmax, absmax_q, scale2,
 * offset) - i.e. they were last written before the kernel preceding this
 * call on the stream began.  That holds for weights quantized once and
 * reused, as in a decode loop.  The folded kernel, which starts while the
 * preceding kernel finishes (programmatic dependent launch), then loads its
 * first weight tiles and scales before waiting for that kernel; x is still
 * read only after it.  The results are bit-identical to the call without the
 * flag; the flag only moves loads earlier, so a caller that breaks the
 * guarantee may get results computed from partly written weights.  The
 * bit-faithful kernel (weights that go one by one through the exact path)
 * ignores the flag. */
#define NF4Q_GEMV_WEIGHTS_STATIC 1
nf4q_status nf4q_gemv_multi_ex(const nf4q_weight* const* wq, int32_t count, const void* x,
                               int32_t M, void* const* y, int32_t flags, void* stream);

/* nf4q_gemv with w_hat rebuilt bit for bit inside the contraction: y =
 * x . w_hat^T with w_hat exactly as nf4q_dequantize produces it, fp32
 * accumulation (only the order of the additions differs from an exact
 * dot product).  Same arguments and errors as nf4q_gemv. */
nf4q_status nf4q_gemv_exact(const nf4q_weight* wq, const void* x, int32_t M,
                            void* y, void* stream);

/* Prefill-shaped matmul on the tcgen05 tensor cores, M >= 1 (intended for
 * M >= 64).  Same contraction and output as nf4q_gemv: Y [M x rows] =
 * X [M x cols] . w_hat^T, compute-dtype operands (bf16 or fp16), fp32
 * accumulate, compute-dtype output.
 *   X, Y: device, of wq->compute_dtype, 16-byte aligned. */
nf4q_status nf4q_gemm(const nf4q_weight* wq, const void* X, int64_t M,
                      void* Y, void* stream);

/* Dispatch on M: nf4q_gemv for M <= NF4Q_GEMV_MAX_M, nf4q_gemm above, and
 * nf4q_gemm also for M = 9..16 on weights of at least NF4Q_MATMUL_GEMM_ROWS
 * rows (the crossover measured on a B300). */
#define NF4Q_GEMV_MAX_M 16
#define NF4Q_MATMUL_GEMM_ROWS 20000
nf4q_status nf4q_matmul(const nf4q_weight* wq, const void* X, int64_t M,
                        void* Y, void* stream);

/* Input gradient through the frozen 4-bit weight - the backward pass of a
 * QLoRA base layer, whose 4-bit weight stays frozen while LoRA adapters
 * train ("bitsandbytes tutorial" sec. 5.4; "bitsandbytes introduction",
 * core techniques item 3): dX [M x cols] =
 * dY [M x rows] . w_hat, on the tcgen05 tensor cores; w_hat exactly as
 * nf4q_dequantize writes it, compute-dtype operands, fp32 accumulate,
 * compute-dtype output.
 *   dY: device, of wq->compute_dtype, row-major with row pitch ld_dy
 *       elements (ld_dy >= rows, a multiple of 8), 16-byte aligned; only the
 *       first `rows` elements of a row are read.
 *   dX: device, [M x cols] row-major, of wq->compute_dtype, 16-byte aligned.
 * M == 0 or cols == 0 launches nothing; rows == 0 writes dX = 0.  Other
 * errors as nf4q_gemm. */
nf4q_status nf4q_matmul_dx(const nf4q_weight* wq, const void* dY, int64_t ld_dy,
                           int64_t M, void* dX, void* stream);

/* Sticky device error flags of the current device (bit 0: a GEMM pipeline
 * wait gave up).  Synchronizes the device; `clear` != 0 resets the flags. */
nf4q_status nf4q_device_error(uint32_t* flags, int32_t clear);

/* Double quantization without a caller-supplied workspace: the same
 * computation and outputs as nf4q_double_quant, for callers that must not
 * allocate device memory at all - e.g. code that runs with every byte of
 * device memory already handed to a fixed pool, or that cannot afford
 * cudaMalloc's implicit device synchronization on a latency-critical path,
 * and so has nowhere to get the small workspace from.  (The bitsandbytes
 * pages have no counterpart; this is an interface convenience only.)
 *   Scratch: a 256-byte array in the library's static device memory, present
 *   on every GPU the library is loaded on until the process exits.  The call
 *   allocates nothing and calls no allocating routine.
 *   Limit: the scratch holds one double-quant record, which serves any tensor
 *   the library accepts; the only size limit is the library-wide one of every
 *   double-quant call, n_b = rows*cols/64 <= 2^31 - 1 (NF4Q_ERR_UNSUPPORTED
 *   beyond it).
 *   Set-up: the first call on each device looks up the scratch's device
 *   address (cudaGetSymbolAddress) with that device current, and caches it
 *   with the id of the current context; a call in another context (after a
 *   cudaDeviceReset, for example) looks it up again.  Make the first call in
 *   a context before any stream capture.
 *   Sharing: every call on a device uses the same scratch, which is zero
 *   when the library's device code loads and which every call leaves zero
 *   (as a caller's workspace for nf4q_double_quant).  Calls whose work overlaps on
 *   the GPU (other streams, other threads) race on it and must be serialized
 *   by the caller.  Other arguments and errors as nf4q_double_quant. */
nf4q_status nf4q_double_quant_noalloc(const nf4q_weight* wq, void* stream);

/* ------------------------------------------------------------------------
 * LLM.int8(): vector-wise int8 quantization and the mixed-precision
 * decomposition matmul ("bitsandbytes tutorial" sec. 3.1: the outlier
 * feature dimensions of the activations are computed in FP16, the rest in
 * INT8, and the two results are added; sec. 四: llm_int8_threshold, default
 * 6.0; "bitsandbytes introduction", core techniques item 2: weights and
 * activations in 8 bits, vector-wise, outlier feature vectors in 16 bits).
 *
 * An int8 weight W [rows x cols] (the nn.Linear [out, in] convention):
 *   q      int8 [rows*cols] row-major codes, 16-byte aligned
 *   scale  fp32 [rows]  s_n = max_k |W[n, k]|, 4-byte aligned
 *   code   q = rint(RN(127 * w / s_n)) (RN: the float32 rounding of the
 *          quotient; rint: half to even), 0 in a row with s_n = 0
 * cols must be a multiple of 16 (16-byte rows). */
typedef struct {
  int8_t* q;
  float* scale;
  int64_t rows;
  int64_t cols;
} nf4q_int8_weight;

#define NF4Q_INT8_DEFAULT_THRESHOLD 6.0f

/* Quantize W (device, fp16 or bf16 per `in_dtype`, row-major, 16-byte
 * aligned) into wq->q / wq->scale.  One CTA per row.  Every int8 call
 * refuses cols > 2^30 and rows > 2^31 - 1 with NF4Q_ERR_UNSUPPORTED. */
nf4q_status nf4q_int8_quantize_weight(const void* w, int32_t in_dtype,
                                      const nf4q_int8_weight* wq, void* stream);

/* HOST ONLY.  Workspace bytes of nf4q_int8_matmul for M activation rows of
 * `cols` elements.  Layout from the (16-byte aligned) start, each section
 * starting at a multiple of 256 bytes after the previous one:
 *   flags  uint8 [cols]    1 where the column is an outlier
 *   count  int32 [1]       number of outlier columns (a 256-byte section)
 *   list   int32 [cols]    the outlier columns, ascending (first `count`)
 *   sx     fp32  [M]       activation row scales
 *   xq     fp16  [M*cols]  activation codes as fp16 integers
 * Section sizes are rounded up to multiples of 256 bytes. */
size_t nf4q_int8_workspace_bytes(int64_t M, int64_t cols);

/* Y [M x rows] = the decomposition matmul of X [M x cols] with the int8
 * weight, fp16 in and out:
 *   outlier columns  O = {k : max_m |X[m, k]| > threshold}; threshold <= 0
 *                    (or NaN) turns the decomposition off
 *   activation codes per row m: sx_m = max |X[m, k]| over k not in O,
 *                    xq = rint(RN(127 * x / sx_m)), 0 in O and when sx_m = 0
 *   Y[m, n] = fp16( C[m, n] * sx_m * s_n / 127^2
 *                   + sum_{k in O} X[m, k] * w_hat[n, k] )
 *   with C the sum of xq * q over k not in O (products of codes, fp32
 *   accumulation: exact while partial sums stay below 2^24) and
 *   w_hat = fp16(RN(RN(q * s_n) / 127)), the 16-bit weight the code gives
 *   back.
 *   X, Y: device fp16, row-major, 16-byte aligned.  The workspace (device,
 *   16-byte aligned, nf4q_int8_workspace_bytes(M, cols) bytes) holds the
 *   activation side after the call.  Streams the weight once per 16 rows of
 *   X (decode-shaped; M is not limited).  M == 0 or rows == 0 launches
 *   nothing; cols == 0 writes Y = 0. */
nf4q_status nf4q_int8_matmul(const nf4q_int8_weight* wq, const void* X, int64_t M,
                             float threshold, void* Y, void* workspace,
                             size_t workspace_bytes, void* stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* NF4Q_H_ */
