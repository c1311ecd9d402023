// Host-side construction of the code tables the kernels use.
//
// NF4: "bitsandbytes tutorial" (mlqm.cn/news/394670), sec. 3.2 - 16 levels
// spaced by the density of the standard normal distribution.  The levels are
// Phi^-1 of 8 points evenly spaced from 0.9677083 down to 0.5 (0.5 itself
// dropped) on the positive side, -Phi^-1 of 7 such points on the negative
// side, and 0, divided by the largest, sorted ascending and rounded to
// float32.  Phi^-1 is obtained here by Newton's method on Phi(x) =
// erfc(-x/sqrt(2))/2 (C library erfc), in double precision.
//
// FP4: the E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} / 6 with a sign bit
// ("bitsandbytes introduction", sec. 一 item 7 and sec. 三 example 2).
//
// Encoder decision points: for neighbouring levels c_j < c_{j+1} the exact
// midpoint (c_j + c_{j+1}) / 2 (exact in double) is rounded DOWN to float32.
// For a float32 value v, "v > T_j" then holds exactly when v is nearer to
// c_{j+1} than to c_j, and an exact tie stays with c_j.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

namespace nf4q {

constexpr int kLutEntries = 259;   // bin index 1..257 is ever produced
constexpr double kNf4Offset = 0.9677083;

struct HostTables {
  float values[2][16];   // [code kind][code]
  float thr[2][15];      // decision points (NF4: 15 on wn; FP4: 7 on |wn|)
  int nthr[2];
  // Bin table of the fast encoder: entry b holds the only decision point
  // within reach of bin b (or 2.0f when there is none), with the number of
  // decision points below the bin stored in its low 4 bits.
  float lut[2][kLutEntries];
  float lut_scale[2], lut_bias[2];
  bool ok;
};

namespace detail {

inline double phi(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

inline double phi_inv(double p) {  // p in (0.5, 1)
  const double inv_sqrt_2pi = 0.39894228040143267794;
  double x = 1.0;
  for (int it = 0; it < 100; ++it) {
    double f = phi(x) - p;
    double d = inv_sqrt_2pi * std::exp(-0.5 * x * x);
    double nx = x - f / d;
    if (nx == x) break;
    x = nx;
  }
  return x;
}

inline float round_down_f32(double v) {
  float f = static_cast<float>(v);
  if (static_cast<double>(f) > v) f = std::nextafter(f, -INFINITY);
  return f;
}

inline void sort16(double* v) {
  for (int i = 1; i < 16; ++i)
    for (int j = i; j > 0 && v[j - 1] > v[j]; --j) {
      double t = v[j]; v[j] = v[j - 1]; v[j - 1] = t;
    }
}

}  // namespace detail

// Fill one bin table.  Bin b receives every value v with
// rn_int(v * scale + bias) == b, i.e. v in [(b - .5 - bias)/scale,
// (b + .5 - bias)/scale]; a margin of a quarter bin absorbs rounding.
inline bool build_lut(const float* thr, int n, float scale, float bias,
                      float* lut) {
  const double m = 0.25 / scale;
  for (int b = 0; b < kLutEntries; ++b) {
    double lo = (b - 0.5 - bias) / scale - m;
    double hi = (b + 0.5 - bias) / scale + m;
    int base = 0, inside = -1, count_inside = 0;
    for (int j = 0; j < n; ++j) {
      if (thr[j] < lo) ++base;
      else if (thr[j] <= hi) { inside = j; ++count_inside; }
    }
    if (count_inside > 1 || base > 15) return false;
    float t = inside >= 0 ? thr[inside] : 2.0f;
    uint32_t bits;
    std::memcpy(&bits, &t, 4);
    bits = (bits & ~0xFu) | static_cast<uint32_t>(base);
    std::memcpy(&lut[b], &bits, 4);
  }
  return true;
}

inline HostTables build_host_tables() {
  HostTables T;
  std::memset(&T, 0, sizeof(T));
  // ---- NF4
  const double start = kNf4Offset, stop = 0.5;
  double v[16];
  int k = 0;
  const double step_pos = (stop - start) / 8.0;   // 9 points, last dropped
  for (int i = 0; i < 8; ++i) v[k++] = detail::phi_inv(i * step_pos + start);
  v[k++] = 0.0;
  const double step_neg = (stop - start) / 7.0;   // 8 points, last dropped
  for (int i = 0; i < 7; ++i) v[k++] = -detail::phi_inv(i * step_neg + start);
  double mx = v[0];
  for (int i = 0; i < 16; ++i) mx = v[i] > mx ? v[i] : mx;
  for (int i = 0; i < 16; ++i) v[i] /= mx;
  detail::sort16(v);
  for (int i = 0; i < 16; ++i) T.values[0][i] = static_cast<float>(v[i]);
  for (int j = 0; j < 15; ++j)
    T.thr[0][j] = detail::round_down_f32(
        (static_cast<double>(T.values[0][j]) + T.values[0][j + 1]) * 0.5);
  T.nthr[0] = 15;
  // ---- FP4
  const double mags[8] = {0, 0.5, 1, 1.5, 2, 3, 4, 6};
  for (int j = 0; j < 8; ++j) {
    T.values[1][j] = static_cast<float>(mags[j] / 6.0);
    T.values[1][8 + j] = -T.values[1][j];
  }
  for (int j = 0; j < 7; ++j)
    T.thr[1][j] = detail::round_down_f32(
        (static_cast<double>(T.values[1][j]) + T.values[1][j + 1]) * 0.5);
  T.nthr[1] = 7;
  // ---- bin tables: NF4 over wn in [-1, 1], FP4 over |wn| in [0, 1]
  T.lut_scale[0] = 128.0f; T.lut_bias[0] = 129.0f;
  T.lut_scale[1] = 256.0f; T.lut_bias[1] = 1.0f;
  T.ok = build_lut(T.thr[0], 15, 128.0f, 129.0f, T.lut[0]) &&
         build_lut(T.thr[1], 7, 256.0f, 1.0f, T.lut[1]);
  return T;
}

}  // namespace nf4q
