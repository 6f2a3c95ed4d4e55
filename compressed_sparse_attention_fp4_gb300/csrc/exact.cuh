// exact.cuh -- exact indexer scores for the candidates an error bound cannot
// decide.
//
// A head dot d = sum_c q_c k_c of fp32-representable factors (bf16 x E4M3,
// or fp32 x fp32) is summed exactly in fixed point and rounded once to fp64
// (round-to-nearest-even); the score is then s = sum_h w_h * ReLU(d_h) in
// fp64, heads in ascending order, with separate (unfused) multiply and add.
// This is the exact ranking value the library's selections are defined on.
//
// Fixed point: every factor is sig * 2^exp with an integer significand (<=
// 24 bits), so every product is an integer P (< 2^48) times 2^E.  Pass 1
// finds the span of the products; if the sum fits in 62 bits it is
// accumulated in one int64, if it fits in 126 bits in one 128-bit integer
// (kept in registers: the usual case of fp32 keys, whose smallest products
// sit far below the largest), else in an 11-limb (704-bit) two's-complement
// integer, which covers the whole fp32 x fp32 range.
#pragma once

#include <climits>

#include "common.cuh"

namespace csa2 {

struct Factor {
  int32_t sig;   // signed significand
  int32_t exp;   // value = sig * 2^exp
};

__device__ inline Factor factor_f32(float x) {
  uint32_t u = __float_as_uint(x);
  int32_t E = int32_t((u >> 23) & 0xFF);
  int32_t m = int32_t(u & 0x7FFFFF);
  Factor f;
  f.sig = (E == 0) ? m : (m | 0x800000);
  f.exp = (E == 0) ? -149 : E - 150;
  if (u >> 31) f.sig = -f.sig;
  return f;
}

__device__ inline Factor factor_e4m3(uint32_t c) {
  int32_t e = int32_t((c >> 3) & 0xF), m = int32_t(c & 7);
  Factor f;
  f.sig = (e == 0) ? m : (8 + m);
  f.exp = (e == 0) ? -9 : e - 10;
  if (c & 0x80) f.sig = -f.sig;
  return f;
}

constexpr int kLimbs = 11;

// value += sign * P * 2^sh in an NL-limb two's-complement integer.
__device__ inline void limb_add(uint64_t* L, uint64_t P, int sh, bool neg) {
  int li = sh >> 6, bo = sh & 63;
  uint64_t lo = P << bo;
  uint64_t hi = bo ? (P >> (64 - bo)) : 0;
  if (!neg) {
    uint64_t old = L[li];
    L[li] = old + lo;
    uint64_t c = L[li] < old;
    int k = li + 1;
    if (k < kLimbs) {
      uint64_t o2 = L[k];
      uint64_t t = o2 + hi;
      uint64_t c2 = t < o2;
      uint64_t t2 = t + c;
      c2 |= (t2 < t);
      L[k] = t2;
      c = c2;
      for (k = k + 1; k < kLimbs && c; ++k) { L[k] += 1; c = (L[k] == 0); }
    }
  } else {
    uint64_t old = L[li];
    L[li] = old - lo;
    uint64_t bw = old < lo;
    int k = li + 1;
    if (k < kLimbs) {
      uint64_t o2 = L[k];
      uint64_t t = o2 - hi;
      uint64_t b2 = o2 < hi;
      uint64_t t2 = t - bw;
      b2 |= (t < bw);
      L[k] = t2;
      bw = b2;
      for (k = k + 1; k < kLimbs && bw; ++k) { bw = (L[k] == 0); L[k] -= 1; }
    }
  }
}

// Round the limb integer times 2^e0 to the nearest fp64 (ties to even).
__device__ inline double limbs_to_double(uint64_t* L, int e0) {
  bool neg = (L[kLimbs - 1] >> 63) != 0;
  if (neg) {
    uint64_t c = 1;
    for (int k = 0; k < kLimbs; ++k) {
      uint64_t v = ~L[k] + c;
      c = (c && v == 0) ? 1 : 0;
      L[k] = v;
    }
  }
  int top = -1;
  for (int k = kLimbs - 1; k >= 0; --k)
    if (L[k]) { top = k; break; }
  if (top < 0) return 0.0;
  int bitpos = 63 - __clzll((long long)L[top]);
  int p = 64 * top + bitpos;                    // index of the leading bit
  double r;
  if (p < 64) {
    r = scalbn(__ull2double_rn(L[0]), e0);
  } else {
    // top 64 bits [p-63, p] with a sticky bit for everything below
    int lo_bit = p - 63;
    int lw = lo_bit >> 6, lb = lo_bit & 63;
    uint64_t top64 = lb ? ((L[lw] >> lb) | (L[lw + 1] << (64 - lb))) : L[lw];
    bool sticky = lb ? ((L[lw] & ((uint64_t(1) << lb) - 1)) != 0) : false;
    for (int k = 0; k < lw; ++k) sticky |= (L[k] != 0);
    top64 |= uint64_t(sticky);
    r = scalbn(__ull2double_rn(top64), e0 + lo_bit);
  }
  return neg ? -r : r;
}

// Round the signed 128-bit integer v times 2^e0 to the nearest fp64 (ties
// to even): the top 64 significant bits with a sticky bit for the rest go
// through one correctly rounded 64-bit conversion (the sticky bit sits below
// the rounding position, so it only breaks ties).
__device__ inline double i128_to_double(__int128 v, int e0) {
  const bool neg = v < 0;
  const unsigned __int128 m = neg ? (unsigned __int128)0 - (unsigned __int128)v : (unsigned __int128)v;
  const uint64_t hi = uint64_t(m >> 64), lo = uint64_t(m);
  double r;
  if (hi == 0) {
    r = scalbn(__ull2double_rn(lo), e0);
  } else {
    const int s = 64 - __clzll((long long)hi);             // bits of hi, 1..64
    const uint64_t mask = s == 64 ? ~uint64_t(0) : ((uint64_t(1) << s) - 1);
    const uint64_t top64 = uint64_t(m >> s) | uint64_t((lo & mask) != 0);
    r = scalbn(__ull2double_rn(top64), e0 + s);
  }
  return neg ? -r : r;
}

// Correctly rounded fp64 value of sum_c q(c) * k(c), the factors given as
// Factors by `qf(c)` and `kf(c)`.
template <class QF, class KF>
__device__ double exact_head_dot(QF qf, int n, KF kf) {
  int elo = INT_MAX, ehi = INT_MIN;
  for (int c = 0; c < n; ++c) {
    Factor a = qf(c), b = kf(c);
    if (a.sig == 0 || b.sig == 0) continue;
    uint64_t P = uint64_t(llabs((long long)a.sig)) * uint64_t(llabs((long long)b.sig));
    int E = a.exp + b.exp;
    elo = min(elo, E);
    ehi = max(ehi, E + 64 - __clzll((long long)P));
  }
  if (elo == INT_MAX) return 0.0;
  int width = ehi - elo + 8;                    // 128 terms add <= 7 bits, +sign
  if (width <= 62) {
    long long acc = 0;
    for (int c = 0; c < n; ++c) {
      Factor a = qf(c), b = kf(c);
      if (a.sig == 0 || b.sig == 0) continue;
      unsigned long long P = uint64_t(llabs((long long)a.sig)) * uint64_t(llabs((long long)b.sig));
      long long term = (long long)(P << (a.exp + b.exp - elo));
      acc += ((a.sig < 0) != (b.sig < 0)) ? -term : term;
    }
    return scalbn(__ll2double_rn(acc), elo);
  }
  if (width <= 126) {
    // every term is below 2^(width - 8) and the sum of <= 128 terms below 2^(width - 1)
    __int128 acc = 0;
    for (int c = 0; c < n; ++c) {
      Factor a = qf(c), b = kf(c);
      if (a.sig == 0 || b.sig == 0) continue;
      const uint64_t P = uint64_t(llabs((long long)a.sig)) * uint64_t(llabs((long long)b.sig));
      const __int128 term = (__int128)((unsigned __int128)P << (a.exp + b.exp - elo));
      acc += ((a.sig < 0) != (b.sig < 0)) ? -term : term;
    }
    return i128_to_double(acc, elo);
  }
  uint64_t L[kLimbs];
  for (int k = 0; k < kLimbs; ++k) L[k] = 0;
  for (int c = 0; c < n; ++c) {
    Factor a = qf(c), b = kf(c);
    if (a.sig == 0 || b.sig == 0) continue;
    uint64_t P = uint64_t(llabs((long long)a.sig)) * uint64_t(llabs((long long)b.sig));
    bool neg = (a.sig < 0) != (b.sig < 0);
    limb_add(L, P, a.exp + b.exp - elo, neg);
  }
  return limbs_to_double(L, elo);
}

// s = sum_h w_h * ReLU(d_h) in fp64, heads in order, no fused multiply-add.
__device__ inline double combine_heads(const double* d, const float* w, int hi) {
  double s = 0.0;
  for (int h = 0; h < hi; ++h) {
    double r = d[h] > 0.0 ? d[h] : 0.0;
    s = __dadd_rn(s, __dmul_rn(double(w[h]), r));
  }
  return s;
}

}  // namespace csa2
