// tw_common.cuh -- small device helpers shared by the libtw kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/ternary_w158a8.h"

namespace tw {

constexpr int kWarp = 32;

// L2 policy for data read exactly once (the packed weights): evict first, so the
// stream does not push the activations and outputs out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Streaming 32-bit load: read-only path, no L1 allocation, L2 evict-first hint.
__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p, uint64_t pol) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

// Bucket decomposition of a finite fp32 magnitude: |v| = m * 2^(b-1) * 2^-149 with
// m < 2^24 an integer and b = max(biased exponent, 1) in [1, 255].
__device__ __forceinline__ void f32_bucket(float v, uint32_t& m, int& b) {
  uint32_t bits = __float_as_uint(v) & 0x7fffffffu;
  uint32_t e8 = bits >> 23;
  uint32_t frac = bits & 0x7fffffu;
  m = e8 ? (frac | 0x800000u) : frac;
  b = e8 ? (int)e8 : 1;
}

// Exact value of  sum_b hist[b] * 2^(step*(b-1))  (hist[0] must be 0), rounded
// once to the nearest double with ties to even, times 2^lsb_exp.  Called by one
// full warp; every lane returns the result.  The integer is held as 32 base-2^32
// digits, one per lane (1024 bits: enough for step <= 2 and 64-bit buckets).
__device__ __forceinline__ double warp_exact_hist_to_double(const unsigned long long* hist,
                                                            int nbuckets, int step, int lsb_exp) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  unsigned long long dig = 0;
  for (int b0 = 0; b0 < nbuckets; b0 += 32) {
    const unsigned long long hv = (b0 + lane < nbuckets) ? hist[b0 + lane] : 0ull;
    unsigned nz = __ballot_sync(full, hv != 0ull);
    while (nz) {
      const int src = __ffs(nz) - 1;
      nz &= nz - 1;
      const unsigned long long v = __shfl_sync(full, hv, src);
      const int pos = step * (b0 + src - 1);
      const int d = pos >> 5, o = pos & 31;
      const unsigned long long lo = v << o;
      const unsigned long long hi = o ? (v >> (64 - o)) : 0ull;
      const int r = lane - d;
      const unsigned piece = r == 0 ? (unsigned)lo : r == 1 ? (unsigned)(lo >> 32) : r == 2 ? (unsigned)hi : 0u;
      dig += piece;
    }
  }
  // Carry propagation (each pass moves carries up one digit; a ripple across all
  // 32 digits needs at most 33 passes).
  for (int it = 0; it < 40; ++it) {
    if (!__any_sync(full, (dig >> 32) != 0ull)) break;
    const unsigned long long c = dig >> 32;
    dig &= 0xffffffffull;
    const unsigned long long cin = __shfl_up_sync(full, c, 1);
    if (lane > 0) dig += cin;
  }
  const unsigned nzmask = __ballot_sync(full, dig != 0ull);
  if (nzmask == 0u) return 0.0;
  const int top = 31 - __clz(nzmask);
  unsigned d2 = __shfl_sync(full, (unsigned)dig, top);
  unsigned d1 = __shfl_sync(full, (unsigned)dig, top >= 1 ? top - 1 : 0);
  unsigned d0 = __shfl_sync(full, (unsigned)dig, top >= 2 ? top - 2 : 0);
  if (top < 1) d1 = 0u;
  if (top < 2) d0 = 0u;
  const bool sticky_low = top >= 3 && (nzmask & ((1u << (top - 2)) - 1u)) != 0u;
  const int lz = __clz(d2);
  unsigned __int128 w = ((unsigned __int128)d2 << 64) | ((unsigned __int128)d1 << 32) | d0;
  w <<= (lz + 32);  // most significant set bit now at bit 127
  unsigned long long m = (unsigned long long)(w >> 75);  // 53 bits
  const bool round_bit = ((unsigned)(w >> 74) & 1u) != 0u;
  const bool sticky = sticky_low || (w & (((unsigned __int128)1 << 74) - 1)) != 0;
  if (round_bit && (sticky || (m & 1ull))) m += 1ull;
  const int msb = 32 * top + 31 - lz;
  return ldexp((double)m, msb - 52 + lsb_exp);
}

// Dequantisation scale fl(fl(gamma * s_x) / 127) of one token.
__device__ __forceinline__ float dequant_scale(float gamma, float s_x) {
  return __fdiv_rn(__fmul_rn(gamma, s_x), 127.0f);
}

// y = acc * gamma * s_x / 127 as fp32.  With a normal scale c = dequant_scale(): one
// more rounding, fl(acc * c), within 3 roundings (< 2e-7 relative) of the exact value.
// When c is subnormal or zero the fp32 chain would lose precision, so the product is
// formed in double as ((acc * gamma) * s_x) / 127 and rounded once to fp32 (a zero
// gamma or s_x gives the signed zero directly).
// Out of line, so that the double arithmetic never appears (not even predicated off)
// in the callers' hot loops: this part's double-precision pipe is narrow.
static __device__ __noinline__ float dequant_tiny(int acc, float gamma, float s_x) {
  if (gamma == 0.0f || s_x == 0.0f) return __fmul_rn((float)acc, 0.0f);  // the exact product, signed zero
  return (float)((((double)acc * (double)gamma) * (double)s_x) / 127.0);
}

__device__ __forceinline__ float dequant(int acc, float c, float gamma, float s_x) {
  if (__builtin_expect(c >= 1.17549435e-38f, 1)) return __fmul_rn((float)acc, c);
  return dequant_tiny(acc, gamma, s_x);
}

// The same for an accumulator already held exactly in fp32 (|acc| < 2^24).
__device__ __forceinline__ float dequant_f(float acc, float c, float gamma, float s_x) {
  if (__builtin_expect(c >= 1.17549435e-38f, 1)) return __fmul_rn(acc, c);
  return dequant_tiny(__float2int_rn(acc), gamma, s_x);
}

// ---------------------------------------------------------------------------
// Exact sum of squares of an fp32 row, fast path.
//
// |x| = m * 2^(b - 150) with m < 2^24 an integer and b = max(biased exponent, 1).
// With E the largest b of the row, x^2 = m^2 * 2^(64 - 2(E - b)) units of
// 2^(2E - 364).  When every nonzero element has E - b <= 32, each term is an
// integer below 2^112 in those units and K < 2^16 terms fit in 128 bits, so the
// sum is exact; sq_round() then rounds it once to double.  Rows with a wider
// exponent spread set `wide` and must take an exact slow path instead.
struct Sum128 {
  unsigned long long lo, hi;
};

__host__ __device__ __forceinline__ void sum128_add(Sum128& s, unsigned long long lo, unsigned long long hi) {
  const unsigned long long t = s.lo + lo;
  s.hi += hi + (t < s.lo ? 1ull : 0ull);
  s.lo = t;
}

// Adds v^2 to s, with E the row's largest biased exponent (max(e, 1)).
__device__ __forceinline__ void sum128_add_square(Sum128& s, float v, int E, bool& wide) {
  const uint32_t bits = __float_as_uint(v) & 0x7fffffffu;
  const uint32_t e8 = bits >> 23;
  const uint32_t m = e8 ? ((bits & 0x7fffffu) | 0x800000u) : (bits & 0x7fffffu);
  const int d = E - (e8 ? (int)e8 : 1);
  wide |= (m != 0u) & (d > 32);
  const unsigned long long m2 = (d > 32) ? 0ull : (unsigned long long)m * m;  // < 2^48
  const unsigned __int128 t = (unsigned __int128)m2 << (64 - 2 * min(d, 32));  // shift 0..64
  sum128_add(s, (unsigned long long)t, (unsigned long long)(t >> 64));
}

__device__ __forceinline__ Sum128 sum128_shfl_xor(const Sum128& s, int o) {
  Sum128 r;
  r.lo = __shfl_xor_sync(0xffffffffu, s.lo, o);
  r.hi = __shfl_xor_sync(0xffffffffu, s.hi, o);
  return r;
}

// Shift of a Sum128 right by sh bits (0 <= sh), reporting whether a nonzero bit
// fell off: used to bring a sum taken relative to a smaller exponent E' into the
// units 2^(2E - 364) of a larger one (sh = 2 (E - E')).
__host__ __device__ __forceinline__ bool sum128_shr_exact(Sum128& s, int sh) {
  if (sh == 0) return true;
  if (sh >= 128) {
    const bool ok = (s.lo | s.hi) == 0ull;
    s.lo = s.hi = 0ull;
    return ok;
  }
  const unsigned __int128 v = ((unsigned __int128)s.hi << 64) | s.lo;
  const unsigned __int128 r = v >> sh;
  s.lo = (unsigned long long)r;
  s.hi = (unsigned long long)(r >> 64);
  return (r << sh) == v;
}

__host__ __device__ __forceinline__ int clz64(unsigned long long v) {
#ifdef __CUDA_ARCH__
  return __clzll((long long)v);
#else
  return v ? __builtin_clzll(v) : 64;
#endif
}

// (hi * 2^64 + lo) * 2^(2E - 364) > 0 rounded once to double precision (nearest,
// ties to even), returned as m * 2^e with 2^52 <= m <= 2^53 (m = 2^53 when the
// rounding carries).
__host__ __device__ __forceinline__ void sum128_round53(const Sum128& s, int E, unsigned long long& m, int& e) {
  const unsigned __int128 v = ((unsigned __int128)s.hi << 64) | s.lo;
  const int n = s.hi ? 128 - clz64(s.hi) : 64 - clz64(s.lo);  // bit length
  if (n <= 53) {
    m = (unsigned long long)v << (53 - n);
    e = 2 * E - 364 - (53 - n);
    return;
  }
  const int drop = n - 53;
  m = (unsigned long long)(v >> drop);
  const unsigned __int128 rem = v & (((unsigned __int128)1 << drop) - 1);
  const unsigned __int128 half = (unsigned __int128)1 << (drop - 1);
  if (rem > half || (rem == half && (m & 1ull))) m += 1ull;
  e = 2 * E - 364 + drop;
}

// The same value as a double.  It is always normal (its exponent is at least -362),
// so it is assembled from its bits: m in [2^52, 2^53] added to the biased exponent
// field minus one also carries m = 2^53 into the exponent.
__device__ __forceinline__ double sum128_to_double(const Sum128& s, int E) {
  if (s.hi == 0ull && s.lo == 0ull) return 0.0;
  unsigned long long m;
  int e;
  sum128_round53(s, E, m, e);
  return __longlong_as_double((long long)(((unsigned long long)(e + 52 + 1023 - 1) << 52) + m));
}

// Division by the row length K (1 <= K <= 2^16) by multiplication with an
// invariant-integer reciprocal (Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994, Theorem 4.2): with l = ceil(log2 K) and
// mk = ceil(2^(54 + l) / K), floor(n / K) = floor(n * mk / 2^(54 + l)) for every
// 0 <= n < 2^54, since 2^(54 + l) <= mk K <= 2^(54 + l) + K - 1 < 2^(54 + l) + 2^l.
struct KDiv {
  unsigned long long mk;
  int sh;  // 54 + l
  int K;
};

__host__ inline KDiv make_kdiv(int K) {
  int l = 0;
  while ((1 << l) < K) ++l;
  const unsigned __int128 num = (unsigned __int128)1 << (54 + l);
  KDiv d;
  d.mk = (unsigned long long)((num + (unsigned __int128)(K - 1)) / (unsigned __int128)K);
  d.sh = 54 + l;
  d.K = K;
  return d;
}

__host__ __device__ __forceinline__ unsigned long long kdiv_floor(unsigned long long n, const KDiv& d) {
  return (unsigned long long)(((unsigned __int128)n * d.mk) >> d.sh);
}

// fl32(fl64(R / K)) for R = m * 2^e (2^52 <= m <= 2^53, R a normal double) with
// integer arithmetic only: the quotient is formed to 32 more bits by two
// invariant-integer divisions (the final remainder is the sticky bit), rounded to
// nearest even at 53 bits, then rounded again at fp32 precision (normal or
// subnormal), exactly as the two conversions of the double-precision formula.
__host__ __device__ __forceinline__ float div_k_round_f32(unsigned long long m, int e, const KDiv& d) {
  const unsigned long long K = (unsigned long long)d.K;
  const unsigned long long q1 = kdiv_floor(m, d), r1 = m - q1 * K;
  const unsigned long long t = r1 << 32;  // < 2^48
  const unsigned long long q0 = kdiv_floor(t, d), r0 = t - q0 * K;
  const unsigned __int128 q = ((unsigned __int128)q1 << 32) + q0;  // R / K = (q + r0 / K) 2^(e - 32)
  const unsigned long long qh = (unsigned long long)(q >> 64), ql = (unsigned long long)q;
  const int n = qh ? 128 - clz64(qh) : 64 - clz64(ql);  // >= 68
  const int drop = n - 53;
  unsigned long long mq = (unsigned long long)(q >> drop);
  const unsigned __int128 rem = q & (((unsigned __int128)1 << drop) - 1);
  const unsigned __int128 half = (unsigned __int128)1 << (drop - 1);
  if (rem > half || (rem == half && (r0 != 0ull || (mq & 1ull)))) mq += 1ull;
  const int eq = e - 32 + drop;  // fl64(R / K) = mq 2^eq, 2^52 <= mq <= 2^53
  const int lead = 52 + eq + (int)(mq >> 53);  // exponent of its leading bit
  uint32_t bits;
  if (lead > 127) {
    bits = 0x7f800000u;
  } else if (lead >= -126) {
    const int dr = (mq >> 53) ? 30 : 29;  // keep 24 bits
    unsigned long long f = mq >> dr;
    const unsigned long long rm = mq & ((1ull << dr) - 1), hf = 1ull << (dr - 1);
    if (rm > hf || (rm == hf && (f & 1ull))) f += 1ull;  // f in [2^23, 2^24]
    bits = ((uint32_t)(lead + 127 - 1) << 23) + (uint32_t)f;
    if (bits > 0x7f800000u) bits = 0x7f800000u;
  } else {
    const int sh = -149 - eq;  // bits of mq below 2^-149, >= 30 here
    if (sh >= 64) {
      bits = 0u;
    } else {
      unsigned long long f = mq >> sh;
      const unsigned long long rm = mq & ((1ull << sh) - 1), hf = 1ull << (sh - 1);
      if (rm > hf || (rm == hf && (f & 1ull))) f += 1ull;
      bits = (uint32_t)f;  // f = 2^23 is the smallest normal
    }
  }
#ifdef __CUDA_ARCH__
  return __uint_as_float(bits);
#else
  float out;
  __builtin_memcpy(&out, &bits, 4);
  return out;
#endif
}

// ---------------------------------------------------------------------------
// Sum of squares, fast path: float-float (unevaluated sum hi + lo of two fp32)
// accumulation with error-free transformations (Knuth's TwoSum, the exact square
// error v*v - fl(v*v) from one fused multiply-add, Dekker's Fast2Sum to
// renormalise).  Every step keeps |lo| <= ulp(hi)/2 and loses at most about
// 2^-45.5 of the running sum, so a row of up to 65532 elements summed by at most
// 171 steps per thread and 9 tree levels is within 2^-37.5 of the exact sum S
// (squares below 2^-126 add at most K 2^-149, negligible for the range admitted).
// ff_mean_f32 then decides fl32(fl64(fl64(S) / K)) when that accuracy suffices
// and reports failure otherwise (the caller takes the exact path).
struct FF {
  float hi, lo;
};

__host__ __device__ __forceinline__ float f_add(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  return a + b;
#endif
}
__host__ __device__ __forceinline__ float f_sub(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fsub_rn(a, b);
#else
  return a - b;
#endif
}
__host__ __device__ __forceinline__ float f_mul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}
__host__ __device__ __forceinline__ float f_fma(float a, float b, float c) {
#ifdef __CUDA_ARCH__
  return __fmaf_rn(a, b, c);
#else
  return fmaf(a, b, c);
#endif
}
__host__ __device__ __forceinline__ float f_div(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fdiv_rn(a, b);
#else
  return a / b;
#endif
}
__host__ __device__ __forceinline__ uint32_t f_bits(float v) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(v);
#else
  uint32_t b;
  __builtin_memcpy(&b, &v, 4);
  return b;
#endif
}
__host__ __device__ __forceinline__ float f_from_bits(uint32_t b) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(b);
#else
  float v;
  __builtin_memcpy(&v, &b, 4);
  return v;
#endif
}

// hi + lo = a + b exactly (TwoSum, any order of magnitudes)
__host__ __device__ __forceinline__ void ff_two_sum(float a, float b, float& hi, float& err) {
  hi = f_add(a, b);
  const float z = f_sub(hi, a);
  err = f_add(f_sub(a, f_sub(hi, z)), f_sub(b, z));
}

__host__ __device__ __forceinline__ void ff_add_square(FF& s, float v) {
  const float p = f_mul(v, v);
  const float e = f_fma(v, v, -p);  // v*v - p exactly
  float t, err;
  ff_two_sum(s.hi, p, t, err);
  const float lo = f_add(s.lo, f_add(err, e));
  s.hi = f_add(t, lo);  // Fast2Sum: |t| >= |lo|
  s.lo = f_sub(lo, f_sub(s.hi, t));
}

// Symmetric in its operands, so a butterfly leaves the same value in every lane.
__host__ __device__ __forceinline__ void ff_add(FF& a, const FF& b) {
  float t, err;
  ff_two_sum(a.hi, b.hi, t, err);
  const float lo = f_add(f_add(a.lo, b.lo), err);
  a.hi = f_add(t, lo);
  a.lo = f_sub(lo, f_sub(a.hi, t));
}

// ms = fl32(fl64(fl64(S) / K)) from s = hi + lo within 2^-37.5 S of S, with
// ik = fl32(1 / K).  The quotient is formed as qh + ql: qh = fl(hi ik) (within
// 2^-22.9 of hi / K), the remainder hi - qh K by one fused multiply-add (off by at
// most 2^-47 hi), ql = fl(fl(r + lo) ik); qh + ql is within 2^-45 of S / K beyond the
// error of s.  c = fl32(qh + ql) is the candidate, accepted when qh + ql lies farther
// than 2^-35 c from both midpoints next to c: the exact quotient, and its two double
// roundings, are then on the same side of them.  Sums outside [2^-80, 2^96] are
// left to the exact path.
__host__ __device__ __forceinline__ bool ff_mean_f32(const FF& s, int K, float ik, float& ms) {
  if (!(s.hi >= 0x1p-80f && s.hi <= 0x1p96f)) return false;
  const float kf = (float)K;
  const float qh = f_mul(s.hi, ik);
  const float r = f_fma(-qh, kf, s.hi);
  const float ql = f_mul(f_add(r, s.lo), ik);
  const float c = f_add(qh, ql);
  const float d = f_add(f_sub(qh, c), ql);  // (qh + ql) - c
  const uint32_t cb = f_bits(c);
  const float up = f_sub(f_from_bits(cb + 1u), c), down = f_sub(c, f_from_bits(cb - 1u));
  const float margin = f_mul(c, 0x1p-35f);
  ms = c;
  return f_add(d, margin) < f_mul(0.5f, up) && f_sub(d, margin) > f_mul(-0.5f, down);
}

// 1 / sqrt(ms + eps) with IEEE fp32 add, square root and divide.
__host__ __device__ __forceinline__ float inv_rms_f32(float ms, float eps) {
#ifdef __CUDA_ARCH__
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#else
  volatile float t = ms + eps;
  return 1.0f / sqrtf(t);
#endif
}

// RMSNorm scale from the exact sum of squares S = (hi:lo) 2^(2E - 364):
// 1 / sqrt(fl32(fl64(S) / K) + eps), the division in double precision emulated
// with integers (no double arithmetic).
__host__ __device__ __forceinline__ float rms_inv_sum128(const Sum128& s, int E, const KDiv& d, float eps) {
  float ms = 0.0f;
  if (s.hi | s.lo) {
    unsigned long long m;
    int e;
    sum128_round53(s, E, m, e);
    ms = div_k_round_f32(m, e, d);
  }
  return inv_rms_f32(ms, eps);
}

// The same from a sum already rounded to double (the exact histogram path).
__device__ __forceinline__ float rms_inv(double r, const KDiv& d, float eps) {
  float ms = 0.0f;
  if (r > 0.0) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(r);
    const int be = (int)(b >> 52);  // r >= 2^-298: normal
    ms = div_k_round_f32((b & ((1ull << 52) - 1)) | (1ull << 52), be - 1075, d);
  }
  return inv_rms_f32(ms, eps);
}

// round_half_even(fl32(p / a)) for a > 0 and |p| <= fl32(127 a), the same integer as
// __float2int_rn(__fdiv_rn(p, a)), with ra = fl32(1 / a).  d = fl(p * ra) is within
// |p/a| * 2^-22.9 < 1.6e-5 of the exact quotient and fl32(p/a) within 2^-18 of it, so
// when d is more than 1e-4 away from a half-integer both round to the same integer
// (rintf(d)); only nearer than that is the exact IEEE divide taken.
__device__ __forceinline__ int quant_div(float p, float a, float ra) {
  const float d = __fmul_rn(p, ra);
  const float r = rintf(d);
  if (fabsf(d - r) < 0.4999f) return (int)r;
  return __float2int_rn(__fdiv_rn(p, a));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum(int v) { return __reduce_add_sync(0xffffffffu, v); }

// Transpose the 4x4 bytes of a 16-byte activation group so that word s holds
// x[4j + s] in byte j (j = 0..3): the order in which (packed_word >> 2s) &
// 0x03030303 presents the weights of that group.
__device__ __forceinline__ uint4 permute_group(uint4 a) {
  const uint32_t t0 = __byte_perm(a.x, a.y, 0x5140);
  const uint32_t t1 = __byte_perm(a.x, a.y, 0x7362);
  const uint32_t t2 = __byte_perm(a.z, a.w, 0x5140);
  const uint32_t t3 = __byte_perm(a.z, a.w, 0x7362);
  uint4 o;
  o.x = __byte_perm(t0, t2, 0x5410);
  o.y = __byte_perm(t0, t2, 0x7632);
  o.z = __byte_perm(t1, t3, 0x5410);
  o.w = __byte_perm(t1, t3, 0x7632);
  return o;
}

// Thread-block clusters: this CTA's rank and the cluster's size, the split cluster barrier
// (every thread of every CTA arrives, then waits; release/acquire orders the shared-memory
// stores made through distributed shared memory before it), and a peer CTA's copy of a
// shared variable.
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <typename T>
__device__ __forceinline__ T* peer(T* p, uint32_t rank) {
  return static_cast<T*>(__cluster_map_shared_rank(static_cast<void*>(p), rank));
}

__device__ __forceinline__ int byte_sum16(uint4 a) {
  int s = __dp4a((int)a.x, 0x01010101, 0);
  s = __dp4a((int)a.y, 0x01010101, s);
  s = __dp4a((int)a.z, 0x01010101, s);
  return __dp4a((int)a.w, 0x01010101, s);
}

}  // namespace tw
