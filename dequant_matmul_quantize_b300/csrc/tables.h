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
// c_{j+1} than to c_j, and an exact tie stays with c_j.  (FP4 applies its 7
// points to |v|.)
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
  // Bin tables of the fast encoder, over the signed normalized value for
  // both codes: entry b holds the only decision point within reach of bin b
  // (2.0f when there is none), the code just below it and the change of code
  // across it.
  float lut_t[2][kLutEntries];
  int32_t lut_lo[2][kLutEntries];
  int32_t lut_dl[2][kLutEntries];
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

// Exact code of a float32 value under the decision points (host copy of the
// rule the kernels implement; used to label the bins).
inline int code_of(const HostTables& T, int code, double v) {
  if (code == 0) {
    int c = 0;
    for (int j = 0; j < 15; ++j) c += v > T.thr[0][j] ? 1 : 0;
    return c;
  }
  const double a = v < 0 ? -v : v;
  int m = 0;
  for (int j = 0; j < 7; ++j) m += a > T.thr[1][j] ? 1 : 0;
  return m | ((v < 0 && m) ? 8 : 0);
}

// Fill the bin tables of one code.  Bin b receives every value v with
// rn_int(v * 128 + 129) == b, i.e. v in [(b - 129.5)/128, (b - 128.5)/128];
// a margin of a quarter bin on both sides absorbs rounding.  The decision
// points on the signed value are +-T_j (FP4) or T_j (NF4); all are more than
// two bins apart, so a bin holds at most one.
inline bool build_lut(HostTables& T, int code) {
  double pts[15];
  int np = 0;
  if (code == 0) {
    for (int j = 0; j < 15; ++j) pts[np++] = T.thr[0][j];
  } else {
    for (int j = 6; j >= 0; --j) pts[np++] = -static_cast<double>(T.thr[1][j]);
    for (int j = 0; j < 7; ++j) pts[np++] = T.thr[1][j];
  }
  const double m = 0.25 / 128.0;
  for (int b = 0; b < kLutEntries; ++b) {
    const double lo = (b - 129.5) / 128.0 - m, hi = (b - 128.5) / 128.0 + m;
    int inside = -1, count = 0;
    for (int j = 0; j < np; ++j)
      if (pts[j] >= lo && pts[j] <= hi) { inside = j; ++count; }
    if (count > 1) return false;
    if (inside < 0) {
      T.lut_t[code][b] = 2.0f;
      T.lut_lo[code][b] = code_of(T, code, 0.5 * (lo + hi));
      T.lut_dl[code][b] = 0;
    } else {
      const double p = pts[inside];
      const float pf = static_cast<float>(p);
      T.lut_t[code][b] = pf;
      const int below = code_of(T, code, std::nextafter(p, -1e9));
      const int above = code_of(T, code, std::nextafter(p, 1e9));
      T.lut_lo[code][b] = below;
      T.lut_dl[code][b] = above - below;
    }
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
  // ---- bin tables over the signed normalized value
  T.ok = build_lut(T, 0) && build_lut(T, 1);
  return T;
}

}  // namespace nf4q
