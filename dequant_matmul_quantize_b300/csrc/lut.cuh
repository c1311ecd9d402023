// Exact bf16 (or fp16) dequantization of packed 4-bit codes with register
// tables.
//
// For one (row, 64-block) the 16 values w_hat_j = bf16(fp32(code_j * s_b))
// - bit for bit what nf4_dequantize writes ("bitsandbytes tutorial", sec.
// 3.4) - are built once and split into a table of high bytes and one of low
// bytes (4 + 4 registers of 4 one-byte entries; FP4 keeps the 8 magnitudes,
// 2 + 2 registers, and takes the sign from bit 3).  Four codes are then
// looked up with byte permutes (prmt) on the low 3 bits of each nibble, a
// select on bit 3, and two permutes that interleave high and low bytes into
// two bf16x2 registers.  About 2.6 integer-pipe instructions per weight.
#pragma once

#include "common.cuh"

namespace nf4q {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t lop_select(uint32_t if1, uint32_t if0, uint32_t m) {
  uint32_t r;  // (if1 & m) | (if0 & ~m)
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(r) : "r"(if1), "r"(if0), "r"(m));
  return r;
}

// (c0 * s, c1 * s) for a pair of code values, each product rounded to
// nearest: one packed f32x2 multiply.
__device__ __forceinline__ uint64_t mul2_rn(uint64_t c01, uint64_t ss) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(c01), "l"(ss));
  return d;
}

// Byte tables of one (row, block): H[i] / L[i] hold the high / low bytes of
// w_hat for codes 4i .. 4i+3 (NF4 uses 4+4 registers; FP4 2+2, magnitudes).
template <int CODE>
struct RowTable {
  uint32_t H[CODE == 0 ? 4 : 2];
  uint32_t L[CODE == 0 ? 4 : 2];
};

template <int CODE, int DT = 0>
__device__ __forceinline__ void build_table(RowTable<CODE>& T, float s, const CodeValues& C) {
  uint64_t ss;
  asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(s));
  const uint64_t* cv = reinterpret_cast<const uint64_t*>(C.v);
#pragma unroll
  for (int i = 0; i < (CODE == 0 ? 4 : 2); ++i) {
    const uint64_t d0 = mul2_rn(cv[2 * i], ss), d1 = mul2_rn(cv[2 * i + 1], ss);
    uint32_t p0, p1;  // bf16x2 (fp16x2) of codes 4i, 4i+1 and 4i+2, 4i+3
    if (DT == 0) {
      asm("{\n .reg .f32 a, b;\n mov.b64 {a, b}, %1;\n cvt.rn.bf16x2.f32 %0, b, a;\n}"
          : "=r"(p0) : "l"(d0));
      asm("{\n .reg .f32 a, b;\n mov.b64 {a, b}, %1;\n cvt.rn.bf16x2.f32 %0, b, a;\n}"
          : "=r"(p1) : "l"(d1));
    } else {
      asm("{\n .reg .f32 a, b;\n mov.b64 {a, b}, %1;\n cvt.rn.f16x2.f32 %0, b, a;\n}"
          : "=r"(p0) : "l"(d0));
      asm("{\n .reg .f32 a, b;\n mov.b64 {a, b}, %1;\n cvt.rn.f16x2.f32 %0, b, a;\n}"
          : "=r"(p1) : "l"(d1));
    }
    T.H[i] = prmt(p0, p1, 0x7531);
    T.L[i] = prmt(p0, p1, 0x6420);
  }
}

// Four codes -> two bf16x2 registers.  `sel` holds the four nibbles with
// bit 3 cleared (low 16 bits), `m` the per-byte 0xFF/0x00 mask of bit 3.
// Byte j of a lookup belongs to nibble j; nibble 2i+1 is element 2i of the
// word (high nibble first), so the interleave puts elements (0,1) and (2,3)
// of these four into the low/high halves of the two outputs.
template <int CODE>
__device__ __forceinline__ void lookup4(const RowTable<CODE>& T, uint32_t sel, uint32_t m,
                                        uint32_t& r01, uint32_t& r23) {
  uint32_t h, l;
  if (CODE == 0) {
    h = lop_select(prmt(T.H[2], T.H[3], sel), prmt(T.H[0], T.H[1], sel), m);
    l = lop_select(prmt(T.L[2], T.L[3], sel), prmt(T.L[0], T.L[1], sel), m);
  } else {  // FP4: magnitude lookup, bit 3 flips the sign
    h = prmt(T.H[0], T.H[1], sel) ^ (m & 0x80808080u);
    l = prmt(T.L[0], T.L[1], sel);
  }
  r01 = prmt(l, h, 0x4051);
  r23 = prmt(l, h, 0x6273);
}

// One packed word (8 consecutive codes of one row) -> four bf16x2 registers
// holding elements (0,1), (2,3), (4,5), (6,7).
template <int CODE>
__device__ __forceinline__ void dequant_word(const RowTable<CODE>& T, uint32_t w,
                                             uint32_t (&r)[4]) {
  const uint32_t s7 = w & 0x77777777u;
  // the two shifts as multiplies, which run on the FMA pipe
  const uint32_t w4 = w * 16u;
  const uint32_t s7h = __umulhi(s7, 0x10000u);  // s7 >> 16
  lookup4<CODE>(T, s7, prmt(w, w4, 0x9D8C), r[0], r[1]);
  lookup4<CODE>(T, s7h, prmt(w, w4, 0xBFAE), r[2], r[3]);
}

}  // namespace nf4q
