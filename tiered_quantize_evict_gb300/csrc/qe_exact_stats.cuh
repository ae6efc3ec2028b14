// qe_exact_stats.cuh -- mean and population standard deviation of a row of float32 values,
// each the exact value rounded once to the nearest float32 (ties to even).
//
// HqeKV reading notes, §2.3 eq. (3): the normalized (1-bit) quantizer subtracts a token's mean
// and divides by its standard deviation.  The pages fix neither a precision nor an order of
// summation, so this library computes both statistics exactly and rounds each once: no
// summation order can change a code or a parameter.
//
// Every float32 x is mant * 2^(ee - 150) with a 24-bit integer mant and ee >= 1 (the biased
// exponent, 1 for subnormals).  Both paths below turn the row into integers X_i = x_i 2^-sigma,
// sum S = sum X_i and Q = sum X_i^2 exactly, and round
//   mean = S 2^sigma / D,   std = sqrt(D Q - S^2) 2^sigma / D   (D = 64 or 128, a power of 2).
//  * Fast path: sigma = E - 182 with E the row's largest ee.  A nonzero value whose ee is below
//    E - 32 would need bits under 2^sigma; otherwise X_i < 2^56, |S| < 2^63 and D Q < 2^126, so
//    64- and 128-bit integers hold everything.  Each lane sums its own values; the partial sums
//    are integers, so adding them in any order gives the same S and Q.
//  * Wide path (rows with a larger dynamic range): sigma = -149, every value an integer below
//    2^277, S in 10 and Q, S^2 and D Q - S^2 in 18 32-bit limbs.
// The helpers are __host__ __device__ so that the host can check them too.
#pragma once
#include <cmath>
#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define QX_HD __host__ __device__ __forceinline__
#else
#define QX_HD inline
#endif

namespace qe {
namespace xs {

typedef unsigned __int128 u128;
typedef unsigned long long u64;

constexpr int FAST_WINDOW = 32;   // binades below the row's largest value the fast path holds
constexpr int WS = 10;            // limbs of the wide sum (signed, two's complement)
constexpr int WQ = 18;            // limbs of the wide sum of squares and of D Q - S^2

QX_HD unsigned f2u(float x) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(x);
#else
  unsigned u;
  memcpy(&u, &x, 4);
  return u;
#endif
}
QX_HD float u2f(unsigned u) {
#if defined(__CUDA_ARCH__)
  return __uint_as_float(u);
#else
  float x;
  memcpy(&x, &u, 4);
  return x;
#endif
}
QX_HD int clz64(u64 a) {
#if defined(__CUDA_ARCH__)
  return __clzll((long long)a);
#else
  return a ? __builtin_clzll(a) : 64;
#endif
}

// x = (neg ? -1 : 1) mant 2^(ee - 150); mant = 0 for zeros
struct Parts {
  unsigned mant;
  int ee;
  bool neg;
};
QX_HD Parts parts(float x) {
  const unsigned b = f2u(x);
  const unsigned be = (b >> 23) & 0xFFu;
  Parts p;
  p.mant = (b & 0x7FFFFFu) | (be ? 0x800000u : 0u);
  p.ee = be ? (int)be : 1;
  p.neg = (b >> 31) != 0;
  return p;
}

QX_HD int bitlen128(u128 a) {
  const u64 hi = (u64)(a >> 64), lo = (u64)a;
  return hi ? 128 - clz64(hi) : (lo ? 64 - clz64(lo) : 0);
}

// n 2^q as a float32, exact: n <= 2^24, q >= -149, and n < 2^23 only when q = -149
QX_HD float compose(u64 n, int q) {
  if (n == 0) return 0.f;
  if (n == (1ull << 24)) {
    n >>= 1;
    ++q;
  }
  if (n >= (1ull << 23)) return u2f(((unsigned)(q + 150) << 23) | ((unsigned)n & 0x7FFFFFu));
  return u2f((unsigned)n);   // subnormal
}

// nearest float32 to A 2^E0 (A >= 0), ties to even
QX_HD float round_u128(u128 A, int E0) {
  if (A == 0) return 0.f;
  const int p = bitlen128(A) - 1;
  const int q = (p + E0 - 23) > -149 ? p + E0 - 23 : -149;   // exponent of the last kept place
  const int sh = q - E0;                                     // bits of A below that place
  u64 n;
  if (sh <= 0) {
    n = (u64)(A << -sh);   // A < 2^24 here
  } else {
    if (sh > 129) return 0.f;   // below a quarter of the smallest subnormal
    n = sh >= 128 ? 0ull : (u64)(A >> sh);
    const int rp = sh - 1;
    const bool rb = rp < 128 && ((A >> rp) & 1) != 0;
    const bool sticky = rp >= 128 ? A != 0 : (rp > 0 && (A & (((u128)1 << rp) - 1)) != 0);
    if (rb && (sticky || (n & 1))) ++n;
  }
  return compose(n, q);
}

// floor(sqrt(y)), y < 2^62
QX_HD u64 isqrt64(u64 y) {
  u64 r = (u64)sqrt((double)y);
  while (r * r > y) --r;
  while ((r + 1) * (r + 1) <= y) ++r;
  return r;
}

// nearest float32 to sqrt(N) 2^F (N >= 0), ties to even.  With q the exponent of the result's
// last place, n = floor(sqrt(N) 2^(F - q)) comes from an integer square root and one exact
// comparison of N with (n + 1/2)^2 4^(q - F) decides the rounding.
QX_HD float sqrt_round_u128(u128 N, int F) {
  if (N == 0) return 0.f;
  const int e = ((bitlen128(N) - 1) >> 1) + F;   // floor(log2 sqrt(N)) + F
  const int q = e - 23 > -149 ? e - 23 : -149;
  const int k = F - q;
  u64 n;
  if (k >= 0) {   // N 4^k < 2^48: an integer
    const u64 y = (u64)(N << (2 * k));
    n = isqrt64(y);
    if (y > n * n + n) ++n;   // y >= (n + 1/2)^2 for an integer y; no ties
  } else {
    const int s2 = -2 * k;    // 2 <= s2 < 128
    const u64 y = (u64)(N >> s2);
    n = isqrt64(y);
    const u128 R = ((u128)(n * n + n) << s2) + ((u128)1 << (s2 - 2));   // (n + 1/2)^2 4^|k|
    if (N > R || (N == R && (n & 1))) ++n;
  }
  return compose(n, q);
}

// ---------------------------------------------------------------------------- fast path
struct FastAcc {
  long long s;   // sum of +-X_i
  u128 q;        // sum of X_i^2
  int bad;       // a nonzero value below the window
};
QX_HD void fast_add(FastAcc& a, float x, int E) {
  const Parts p = parts(x);
  if (p.mant == 0) return;
  const int sh = p.ee - E + FAST_WINDOW;
  if (sh < 0) {
    a.bad = 1;
    return;
  }
  const u64 X = (u64)p.mant << sh;   // < 2^56
  a.s += p.neg ? -(long long)X : (long long)X;
  a.q += (u128)((u64)p.mant * p.mant) << (2 * sh);   // < 2^112
}
// S, Q of the whole row; E its largest ee; lgD = log2(D)
QX_HD void fast_finish(long long S, u128 Q, int E, int lgD, float& m, float& sd) {
  const int sigma = E - FAST_WINDOW - 150;
  const u64 a = S < 0 ? (u64)(-S) : (u64)S;
  const float mm = round_u128((u128)a, sigma - lgD);
  m = S < 0 ? -mm : mm;
  const u128 N = (Q << lgD) - (u128)a * a;   // D^2 * population variance, >= 0
  sd = sqrt_round_u128(N, sigma - lgD);
}

// ---------------------------------------------------------------------------- wide path
struct WideAcc {
  unsigned s[WS];
  unsigned q[WQ];
};
QX_HD void wide_zero(WideAcc& w) {
  for (int i = 0; i < WS; ++i) w.s[i] = 0u;
  for (int i = 0; i < WQ; ++i) w.q[i] = 0u;
}
// a += v 2^(32 w0) (or -=), v < 2^96, two's complement over NL limbs
QX_HD void wide_add(unsigned* a, int NL, u128 v, int w0, bool sub) {
  u64 c = 0;
  for (int i = w0; i < NL; ++i) {
    const int j = i - w0;
    const unsigned t = j < 3 ? (unsigned)(v >> (32 * j)) : 0u;
    if (!sub) {
      const u64 r = (u64)a[i] + t + c;
      a[i] = (unsigned)r;
      c = r >> 32;
    } else {
      const u64 r = (u64)a[i] - t - c;
      a[i] = (unsigned)r;
      c = (r >> 63) & 1ull;
    }
    if (j >= 2 && c == 0) break;
  }
}
QX_HD void wide_acc(WideAcc& w, float x) {
  const Parts p = parts(x);
  if (p.mant == 0) return;
  const int sh = p.ee - 1;   // x = mant 2^sh 2^-149
  wide_add(w.s, WS, (u128)p.mant << (sh & 31), sh >> 5, p.neg);
  const int s2 = 2 * sh;
  wide_add(w.q, WQ, (u128)((u64)p.mant * p.mant) << (s2 & 31), s2 >> 5, false);
}
QX_HD int wide_bitlen(const unsigned* a, int NL) {
  for (int i = NL - 1; i >= 0; --i)
    if (a[i]) return 32 * i + (64 - clz64((u64)a[i]));
  return 0;
}
// bits [pos, pos + 64) of a (pos >= 0)
QX_HD u64 wide_bits(const unsigned* a, int NL, int pos) {
  const int w = pos >> 5, b = pos & 31;
  u128 v = 0;
  for (int j = 2; j >= 0; --j) v = (v << 32) | (u128)(w + j < NL ? a[w + j] : 0u);
  return (u64)(v >> b);
}
QX_HD bool wide_any_below(const unsigned* a, int pos) {   // a bit below pos is set
  const int w = pos >> 5, b = pos & 31;
  for (int i = 0; i < w; ++i)
    if (a[i]) return true;
  return b > 0 && (a[w] & ((1u << b) - 1u)) != 0;
}
// nearest float32 to A 2^E0 (A >= 0 over NL limbs)
QX_HD float wide_round(const unsigned* a, int NL, int E0) {
  const int bl = wide_bitlen(a, NL);
  if (bl == 0) return 0.f;
  const int p = bl - 1;
  const int q = (p + E0 - 23) > -149 ? p + E0 - 23 : -149;
  const int sh = q - E0;
  u64 n;
  if (sh <= 0) {
    n = (u64)a[0] << -sh;   // A < 2^24
  } else {
    n = wide_bits(a, NL, sh) & 0xFFFFFFFFull;   // A >> sh < 2^25
    const bool rb = (wide_bits(a, NL, sh - 1) & 1ull) != 0;
    const bool sticky = sh - 1 > 0 && wide_any_below(a, sh - 1);
    if (rb && (sticky || (n & 1))) ++n;
  }
  return compose(n, q);
}
// compare two NL-limb magnitudes: -1, 0, 1
QX_HD int wide_cmp(const unsigned* a, const unsigned* b, int NL) {
  for (int i = NL - 1; i >= 0; --i)
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  return 0;
}
// nearest float32 to sqrt(N) 2^F (N over WQ limbs)
QX_HD float wide_sqrt_round(const unsigned* N, int F) {
  const int bl = wide_bitlen(N, WQ);
  if (bl == 0) return 0.f;
  const int e = ((bl - 1) >> 1) + F;
  const int q = e - 23 > -149 ? e - 23 : -149;
  const int k = F - q;
  u64 n;
  if (k >= 0) {   // N 4^k < 2^48, so N itself fits two limbs
    const u64 y = (((u64)N[1] << 32) | N[0]) << (2 * k);
    n = isqrt64(y);
    if (y > n * n + n) ++n;
  } else {
    const int s2 = -2 * k;
    const u64 y = wide_bits(N, WQ, s2);   // floor(N / 4^|k|) < 2^50
    n = isqrt64(y);
    unsigned R[WQ];
    for (int i = 0; i < WQ; ++i) R[i] = 0u;
    wide_add(R, WQ, (u128)(n * n + n) << (s2 & 31), s2 >> 5, false);
    wide_add(R, WQ, (u128)1 << ((s2 - 2) & 31), (s2 - 2) >> 5, false);
    const int c = wide_cmp(N, R, WQ);
    if (c > 0 || (c == 0 && (n & 1))) ++n;
  }
  return compose(n, q);
}
QX_HD void wide_finish(const WideAcc& w, int lgD, float& m, float& sd) {
  // |S| (the sum is below 2^285, so it fits 9 limbs once its sign is taken off)
  unsigned a[WS];
  const bool neg = (w.s[WS - 1] >> 31) != 0;
  u64 c = 1;
  for (int i = 0; i < WS; ++i) {
    if (neg) {
      const u64 r = (u64)(~w.s[i]) + c;
      a[i] = (unsigned)r;
      c = r >> 32;
    } else {
      a[i] = w.s[i];
    }
  }
  const float mm = wide_round(a, WS, -149 - lgD);
  m = neg ? -mm : mm;
  // N = D Q - S^2
  unsigned N[WQ];
  for (int i = 0; i < WQ; ++i) N[i] = (w.q[i] << lgD) | (i > 0 ? w.q[i - 1] >> (32 - lgD) : 0u);
  for (int i = 0; i < WS - 1; ++i) {
    if (!a[i]) continue;
    u64 carry = 0;
    unsigned row[WQ];
    for (int j = 0; j < WQ; ++j) row[j] = 0u;
    for (int j = 0; j < WS - 1 && i + j < WQ; ++j) {
      const u64 t = (u64)a[i] * a[j] + carry;
      row[i + j] = (unsigned)t;
      carry = t >> 32;
    }
    if (i + WS - 1 < WQ) row[i + WS - 1] = (unsigned)carry;
    u64 br = 0;
    for (int j = 0; j < WQ; ++j) {
      const u64 r = (u64)N[j] - row[j] - br;
      N[j] = (unsigned)r;
      br = (r >> 63) & 1ull;
    }
  }
  sd = wide_sqrt_round(N, -149 - lgD);
}

}  // namespace xs
}  // namespace qe
