// tw_gemv_stream.cu -- batch 1..4 ternary GEMV that streams the packed weights
// straight into registers, optionally with the activation quantisation (and
// RMSNorm) fused in front.
//
// The GEMV is bound by reading the packed weights once ("1bit-systems" page,
// 性能实测: the ternary GEMV saturates the memory system; only fewer bytes make
// it faster).  At decode sizes (1.6 - 9 MB per matrix on a 148-SM part) the cost
// of a launch is mostly latency, so the kernel is built around hiding it:
//   * one CTA of 12 warps per SM, small enough (<= 85 registers per thread, little
//     shared memory) that the next launch's CTA fits beside it;
//   * CTA c owns a contiguous block of rows; warp group g (of G = 12/S warps) takes
//     rows g, g + G, ...; the S warps of a group split K;
//   * every warp loads the packed words of its first PRE rows (one 32-bit word =
//     16 weights per lane and step, 128 contiguous bytes per warp load, L2
//     evict-first, no L1 allocation) BEFORE griddepcontrol.wait: under
//     programmatic dependent launch the weight stream of this GEMV runs while the
//     kernel before it is still finishing; only then are the activations read;
//   * the activations (fused quantisation, or int8 x_q) go to shared memory with
//     each 16-element group byte-transposed, and each warp keeps the groups of
//     its K slice in registers;
//   * decode without shifts: for a word w of codes c = t + 1, (w & (3 << 2s) in
//     every byte) holds c(4j+s) * 4^s in byte j, so one AND and one dp4a
//     (unsigned codes x signed activations) per s and token give 4^s * sum c*x;
//     the four sums are scaled back exactly by arithmetic shifts, and
//     sum c*x - sum x = sum t*x exactly;
//   * row totals (redux.sync per warp, summed over K slices with shared atomics)
//     stay in shared memory; one coalesced epilogue writes y.
// The fused prologue's RMSNorm sum of squares is exact (128-bit fixed point
// relative to the row's largest exponent; rows whose exponents spread further fall
// back to the exponent-bucket histogram), so x_q is independent of launch shape.
#include "tw_common.cuh"

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

namespace tw {

__device__ int g_stream_status;  // 0 or a tw_status recorded by a kernel (sticky until read)

constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// sum of (unsigned bytes of a) * (signed bytes of b) + c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The packed word at byte offset OFF from p when bit BIT of ok is set: one predicated load,
// its predicate formed inside, no branch.  Otherwise v is left undefined; the callers
// multiply such words by x = 0, so any value gives the same result.
template <int OFF, uint32_t BIT>
__device__ __forceinline__ void ld_stream_if(uint32_t& v, const uint32_t* p, uint32_t ok, uint64_t pol) {
  asm volatile(
      "{\n .reg .pred q;\n .reg .b32 t;\n and.b32 t, %1, %3;\n setp.ne.b32 q, t, 0;\n"
      " @q ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%2+%4], %5;\n}\n"
      : "=r"(v)
      : "r"(ok), "l"(p), "n"(BIT), "n"(OFF), "l"(pol));
}
// Words j = 0 .. JMAX-1 of one row: word j at 128 j bytes from p (a lane's word of each
// 32-word step), loaded where bit j of ok is set.
template <int... J>
__device__ __forceinline__ void ld_row_words(uint32_t* w, const uint32_t* p, uint32_t ok, uint64_t pol,
                                             std::integer_sequence<int, J...>) {
  (ld_stream_if<128 * J, 1u << J>(w[J], p, ok, pol), ...);
}

struct StreamArgs {
  const uint8_t* packed;
  const float* w_scale;
  const float* x;         // fused: fp32 activations [M][K] (NULL -> use x_q_in)
  const float* g;         // fused RMSNorm gain [K] or NULL
  float eps;
  KDiv kd;                // invariant-integer division by K (RMSNorm mean, exact path)
  float inv_k;            // fl32(1 / K) (RMSNorm mean, fast path)
  const int8_t* x_q_in;   // pre-quantised activations [M][K]
  const float* s_x_in;    // their scales [M]
  int M, N, K;
  int rows_base, rows_rem;  // CTA c owns rows_base (+1 if c < rows_rem) rows
  int S;                    // warps per row (K slices)
  int xs_off, acc_off;      // byte offsets in dynamic shared memory
  int xf_off;               // staged fp32 activations (+ gain), or -1: read x from global
  float* y;
  int32_t* acc_out;
  int8_t* x_q_out;        // fused: written by CTA 0 when non-NULL
  float* s_x_out;
  int32_t* x_sum_out;
  // one token, residual epilogue: res_out = fl(res + y) (y as the definition states, in
  // double); each CTA stores the partial statistics of its rows of res_out for the next
  // RMSNorm (gain g_next) as parts[CTA] = {float-float sum of squares (hi, lo), and the
  // element h with its gain g of the largest fl(|h g|)}
  const float* res;
  float* res_out;
  const float* g_next;
  KDiv kd127;             // division by 127 (the exact y)
  float4* parts_out;
  int h_off;              // byte offset of the CTA's res_out values and g_next values in shared memory
  // one token, finished statistics: the nparts partials a residual epilogue left for x
  const float4* parts_in;
  int nparts;
};

// Partials of the residual epilogue: one float4 per CTA of the writing launch (its grid is
// min(N, SMs) <= kDecThreads).
constexpr int kMaxEpiParts = 512;

// Block-wide sum of MT values (every thread gets the results).
template <int MT>
__device__ __forceinline__ void breduce_sum_i32(int (&v)[MT], int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    v[m] = __reduce_add_sync(0xffffffffu, v[m]);
    if (lane == 0) red[warp * MT + m] = v[m];
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += red[w * MT + m];
    v[m] = t;
  }
  __syncthreads();
}

// Exact sum of squares of one row by the whole block through the exponent-bucket
// histogram (slow path for rows with a wide exponent spread).
template <int NW>
__device__ double row_sumsq_hist(const float4* xr, int K4, uint32_t (*limb)[256], unsigned long long* hist,
                                 double* out) {
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256; i += NT) limb[0][i] = limb[1][i] = limb[2][i] = 0u;
  __syncthreads();
  for (int i = tid; i < K4; i += NT) {
    const float4 v = xr[i];
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t mm;
      int b;
      f32_bucket(e[j], mm, b);
      if (mm) {
        const unsigned long long sq = (unsigned long long)mm * mm;
        atomicAdd(&limb[0][b], (uint32_t)(sq & 0xffffu));
        atomicAdd(&limb[1][b], (uint32_t)((sq >> 16) & 0xffffu));
        atomicAdd(&limb[2][b], (uint32_t)(sq >> 32));
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < 256; i += NT)
    hist[i] = (unsigned long long)limb[0][i] + ((unsigned long long)limb[1][i] << 16) +
              ((unsigned long long)limb[2][i] << 32);
  __syncthreads();
  if (warp == 0) {
    const double r = warp_exact_hist_to_double(hist, 256, 2, -298);
    if (lane == 0) *out = r;
  }
  __syncthreads();
  return *out;
}

// Quantisation of MT tokens into xs (byte-transposed 16-element groups): element k
// of group k/16 goes to byte (k/4) % 4 of word k % 4 of that group.  u4 holds u
// itself ([MT][K4]); with u4 == NULL, u = fl(fl(x * inv) * g) is recomputed from x
// and g4.  CTA 0 also stores x_q, s_x and x_sum when asked.
template <int MT>
__device__ __forceinline__ void quantise_tokens(const StreamArgs& a, uint4* xs, const float4* u4, const float4* g4,
                                                const float (&inv)[MT], const uint32_t (&am)[MT], int* red_i,
                                                float* s_scale) {
  const int tid = threadIdx.x;
  const int K = a.K, Kw = K >> 4, K4 = K >> 2;
  unsigned char* xsb = reinterpret_cast<unsigned char*>(xs);
  int qsum[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    qsum[m] = 0;
    const float amax = __uint_as_float(am[m]);
    // d = fl(p ra) with ra within one ulp of 1 / a (rcp.approx, documented to 1 ulp)
    // is within |p/a| 2^-22 < 3.1e-5 of p / a (|p/a| <= 127), and fl32(p/a) within
    // 2^-18 of it: when d is at least 5e-5 from a half-integer, rint(d) is
    // round_half_even(fl32(p / a)).  Units with an element nearer than that, or with
    // a non-finite d (ra is NaN when a lies outside [2^-120, 2^120]), are redone with
    // the IEEE divide.
    float ra = amax == 0.0f ? 0.0f : __int_as_float(0x7fffffff);
    if (amax >= 0x1p-120f && amax <= 0x1p120f) asm("rcp.approx.f32 %0, %1;" : "=f"(ra) : "f"(amax));
    const float4* ur = u4 ? u4 + (size_t)m * K4 : reinterpret_cast<const float4*>(a.x + (size_t)m * K);
    auto load_u = [&](int u) -> float4 {
      float4 v = ur[u];
      if (!u4) {
        const float4 gg = g4[u];
        v = make_float4(__fmul_rn(__fmul_rn(v.x, inv[m]), gg.x), __fmul_rn(__fmul_rn(v.y, inv[m]), gg.y),
                        __fmul_rn(__fmul_rn(v.z, inv[m]), gg.z), __fmul_rn(__fmul_rn(v.w, inv[m]), gg.w));
      }
      return v;
    };
    // round to nearest even without conversion instructions: for |d| < 2^22,
    // d + 1.5 2^23 rounds d to an integer held in the low mantissa bits
    auto q_fast = [&](float uv, bool& near) -> uint32_t {
      const float d = __fmul_rn(__fmul_rn(uv, 127.0f), ra);
      const float sb = __fadd_rn(d, 12582912.0f);
      const float r = __fsub_rn(sb, 12582912.0f);
      near |= !(fabsf(__fsub_rn(d, r)) < 0.49995f);  // also when d is not finite
      const int t = (int)(__float_as_uint(sb) & 0x7fffffu) - 0x400000;
      return (uint32_t)max(-128, min(127, t)) & 0xffu;
    };
    auto q_exact = [&](float uv) -> uint32_t {
      const int t = amax > 0.0f ? __float2int_rn(__fdiv_rn(__fmul_rn(uv, 127.0f), amax)) : 0;
      return (uint32_t)max(-128, min(127, t)) & 0xffu;
    };
    if (m < a.M) {
      // warp-uniform trip count (lane l takes unit base + l), so the vote below is safe
#pragma unroll 2
      for (int base = (tid & ~31); base < K4; base += kThreads) {
        const int u = base + (tid & 31);
        uint32_t pq = 0u;
        bool near = false;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (u < K4) {
          v = load_u(u);
          pq = q_fast(v.x, near) | (q_fast(v.y, near) << 8) | (q_fast(v.z, near) << 16) | (q_fast(v.w, near) << 24);
        }
        if (__any_sync(0xffffffffu, near) && near)  // rare
          pq = q_exact(v.x) | (q_exact(v.y) << 8) | (q_exact(v.z) << 16) | (q_exact(v.w) << 24);
        if (u < K4) {
          qsum[m] += (int)(int8_t)(pq & 0xffu) + (int)(int8_t)((pq >> 8) & 0xffu) +
                     (int)(int8_t)((pq >> 16) & 0xffu) + (int)(int8_t)(pq >> 24);
          if (blockIdx.x == 0 && a.x_q_out) reinterpret_cast<uint32_t*>(a.x_q_out + (size_t)m * K)[u] = pq;
          unsigned char* gb = xsb + (size_t)m * Kw * 16 + (u >> 2) * 16 + (u & 3);
#pragma unroll
          for (int e = 0; e < 4; ++e) gb[4 * e] = (unsigned char)(pq >> (8 * e));
        }
      }
    } else {  // padding token: zeros in xs only
      for (int u = tid; u < K4; u += kThreads) {
        unsigned char* gb = xsb + (size_t)m * Kw * 16 + (u >> 2) * 16 + (u & 3);
#pragma unroll
        for (int e = 0; e < 4; ++e) gb[4 * e] = 0;
      }
    }
  }
  if (blockIdx.x == 0 && a.x_sum_out) {
    breduce_sum_i32<MT>(qsum, red_i);
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (tid == m && m < a.M) a.x_sum_out[m] = qsum[m];
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (tid == m) {
      s_scale[m] = __uint_as_float(am[m]);
      if (blockIdx.x == 0 && a.s_x_out && m < a.M) a.s_x_out[m] = __uint_as_float(am[m]);
    }
  }
}

// Exact RMSNorm scale of one row by the whole block (taken only when the fast
// path below cannot decide the rounding of the mean square): each warp sums its
// squares in 128-bit fixed point relative to its own largest exponent, warp 0 brings
// the per-warp sums to the row's largest exponent (exact unless a nonzero bit would
// fall off, which sends the row to the exponent-bucket histogram) and forms the scale
// with integer arithmetic only.
template <int NW>
__device__ __noinline__ float rms_inv_exact(const float4* xr, int K4, KDiv kd, float eps, uint32_t* red_u,
                                            unsigned long long* red_lo, unsigned long long* red_hi,
                                            uint32_t (*limb)[256], unsigned long long* hist, double* s_dbl,
                                            float* s_out, int* s_flag) {
  static_assert(NW <= 16, "the cross-warp combine below covers at most 16 warps");
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t mx = 0u;
  for (int i = tid; i < K4; i += NT) {
    const float4 v = xr[i];
    mx = max(mx, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                     max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
  }
  const uint32_t mw = __reduce_max_sync(0xffffffffu, mx);
  const int Ew = max((int)(mw >> 23), 1);
  Sum128 sq;
  sq.lo = sq.hi = 0ull;
  bool wd = false;
  for (int i = tid; i < K4; i += NT) {
    const float4 v = xr[i];
    sum128_add_square(sq, v.x, Ew, wd);
    sum128_add_square(sq, v.y, Ew, wd);
    sum128_add_square(sq, v.z, Ew, wd);
    sum128_add_square(sq, v.w, Ew, wd);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Sum128 t = sum128_shfl_xor(sq, o);
    sum128_add(sq, t.lo, t.hi);
  }
  wd = __any_sync(0xffffffffu, wd);
  if (lane == 0) {
    red_lo[warp] = sq.lo;
    red_hi[warp] = sq.hi;
    red_u[warp] = mw | (wd ? 0x80000000u : 0u);  // bit 31: this warp's spread exceeded the window
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = lane < NW ? red_u[lane] : 0u;
    const uint32_t w = t & 0x7fffffffu;
    const uint32_t mb = __reduce_max_sync(0xffffffffu, w);
    const int Eb = max((int)(mb >> 23), 1), Ewl = max((int)(w >> 23), 1);
    Sum128 tot;
    tot.lo = lane < NW ? red_lo[lane] : 0ull;
    tot.hi = lane < NW ? red_hi[lane] : 0ull;
    bool slow = (t >> 31) != 0u;
    if (!sum128_shr_exact(tot, 2 * (Eb - Ewl))) slow = true;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // NW <= 16
      const Sum128 u = sum128_shfl_xor(tot, o);
      sum128_add(tot, u.lo, u.hi);
    }
    slow = __any_sync(0xffffffffu, slow);
    if (lane == 0) {
      *s_flag = slow ? 1 : 0;
      *s_out = slow ? 0.0f : rms_inv_sum128(tot, Eb, kd, eps);
    }
  }
  __syncthreads();
  if (*s_flag) {
    const double r = row_sumsq_hist<NW>(xr, K4, limb, hist, s_dbl);
    if (tid == 0) *s_out = rms_inv(r, kd, eps);
    __syncthreads();
  }
  const float inv = *s_out;
  __syncthreads();  // s_out and the reduction slots may be reused by the caller
  return inv;
}

// Quantise the activations of MT tokens (after RMSNorm when RMS) into xs
// (byte-transposed 16-element groups); scales to s_scale.  CTA 0 also stores
// x_q, s_x and x_sum when asked.  When xf is not NULL the first pass copies x into
// shared memory (the gain is already there), and later passes read it (with RMSNorm, the
// normalised u replaces x there).  Barriers: one without RMSNorm; two with it in
// the common case: the first pass also sums the squares in float-float, every warp
// then combines the per-warp sums itself and decides the mean square when the
// float-float accuracy suffices (else the block takes the exact path).
template <int MT, bool RMS>
__device__ __forceinline__ void fused_prologue(const StreamArgs& a, uint4* xs, float* xf, float* s_scale,
                                               uint32_t* red_u, uint32_t* red_a, float2* red_ff, int* red_i,
                                               unsigned long long* red_lo, unsigned long long* red_hi,
                                               uint32_t (*limb)[256], unsigned long long* hist, double* s_dbl,
                                               float* s_inv, int* s_slow) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4, K4 = K >> 2;
  const bool staged = xf != nullptr;
  float4* xf4 = reinterpret_cast<float4*>(xf);  // [MT][K4] then the gain [K4]
  const float4* g4 = staged && RMS ? xf4 + (size_t)MT * K4 : reinterpret_cast<const float4*>(a.g);
  auto xsrc = [&](int m) -> const float4* {
    return staged ? xf4 + (size_t)m * K4 : reinterpret_cast<const float4*>(a.x + (size_t)m * K);
  };
  // first pass: from global memory (staging copy), largest magnitude per token as bits
  // and, with RMSNorm, the float-float sum of squares
  uint32_t mx[MT];
  FF sq[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    mx[m] = 0u;
    // one accumulator per vector component: four independent dependency chains
    FF s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f}, s2 = {0.0f, 0.0f}, s3 = {0.0f, 0.0f};
    if (m < a.M) {
      const float4* xg = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
#pragma unroll 2
      for (int i = tid; i < K4; i += kThreads) {
        const float4 v = xg[i];
        if (staged) xf4[(size_t)m * K4 + i] = v;
        mx[m] = max(mx[m], max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                               max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
        if (RMS) {
          ff_add_square(s0, v.x);
          ff_add_square(s1, v.y);
          ff_add_square(s2, v.z);
          ff_add_square(s3, v.w);
        }
      }
    }
    if (RMS) {
      ff_add(s0, s1);
      ff_add(s2, s3);
      ff_add(s0, s2);
    }
    sq[m] = s0;
  }
  // (with RMSNorm and staging, the gain was staged before the dependency wait)
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const uint32_t mw = __reduce_max_sync(0xffffffffu, mx[m]);
    if (RMS) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        FF t;
        t.hi = __shfl_xor_sync(0xffffffffu, sq[m].hi, o);
        t.lo = __shfl_xor_sync(0xffffffffu, sq[m].lo, o);
        ff_add(sq[m], t);
      }
    }
    if (lane == 0) {
      red_u[warp * MT + m] = mw;
      if (RMS) red_ff[warp * MT + m] = make_float2(sq[m].hi, sq[m].lo);
    }
  }
  __syncthreads();  // (1) per-warp maxima and sums; also publishes the staged copy
  uint32_t am[MT];  // a = max |u| per token (u >= 0 compares as its bits)
  if constexpr (RMS) {
    // every warp combines the per-warp sums of each token (same values, same order:
    // the same result in every lane of every warp) and decides the mean square
    float inv[MT];
    bool okm[MT];
    bool slow = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      FF t;
      t.hi = t.lo = 0.0f;
      if (lane < kWarps) {
        const float2 f = red_ff[lane * MT + m];
        t.hi = f.x;
        t.lo = f.y;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {  // kWarps <= 16
        FF u;
        u.hi = __shfl_xor_sync(0xffffffffu, t.hi, o);
        u.lo = __shfl_xor_sync(0xffffffffu, t.lo, o);
        ff_add(t, u);
      }
      // lane 0's sum to every lane: the decision below (and the barriers of the exact
      // path it may select) is then the same in every thread of the block
      t.hi = __shfl_sync(0xffffffffu, t.hi, 0);
      t.lo = __shfl_sync(0xffffffffu, t.lo, 0);
      float ms = 0.0f;
      okm[m] = m >= a.M || ff_mean_f32(t, K, a.inv_k, ms);
      inv[m] = okm[m] ? inv_rms_f32(ms, a.eps) : 0.0f;
      slow |= !okm[m];
    }
    if (slow) {  // block-uniform: every warp took the same decisions
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (!okm[m])
          inv[m] = rms_inv_exact<kWarps>(xsrc(m), K4, a.kd, a.eps, red_u + kWarps * MT, red_lo, red_hi, limb, hist, s_dbl,
                                 s_inv, s_slow);
    }
    // second pass: u = fl(fl(x * inv) * g) (kept in the staging copy) and a = max |u|
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      am[m] = 0u;
      if (m < a.M) {
        const float4* xr = xsrc(m);
#pragma unroll 2
        for (int i = tid; i < K4; i += kThreads) {
          const float4 v = xr[i];
          const float4 gg = g4[i];
          const float4 u = make_float4(__fmul_rn(__fmul_rn(v.x, inv[m]), gg.x), __fmul_rn(__fmul_rn(v.y, inv[m]), gg.y),
                                       __fmul_rn(__fmul_rn(v.z, inv[m]), gg.z), __fmul_rn(__fmul_rn(v.w, inv[m]), gg.w));
          if (staged) xf4[(size_t)m * K4 + i] = u;  // this thread's own slots
          const float t = fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w)));
          am[m] = max(am[m], __float_as_uint(t));
        }
      }
      am[m] = __reduce_max_sync(0xffffffffu, am[m]);
      if (lane == 0) red_a[warp * MT + m] = am[m];
    }
    __syncthreads();  // (2)
#pragma unroll
    for (int m = 0; m < MT; ++m) am[m] = __reduce_max_sync(0xffffffffu, lane < kWarps ? red_a[lane * MT + m] : 0u);
    // quantise u (from the staging copy, or recomputed from x)
    quantise_tokens<MT>(a, xs, staged ? xf4 : nullptr, g4, inv, am, red_i, s_scale);
  } else {
    // without RMSNorm u = x: a is the largest |x| of the first pass
#pragma unroll
    for (int m = 0; m < MT; ++m) am[m] = __reduce_max_sync(0xffffffffu, lane < kWarps ? red_u[lane * MT + m] : 0u);
    float inv[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) inv[m] = 1.0f;
    quantise_tokens<MT>(a, xs, staged ? xf4 : reinterpret_cast<const float4*>(a.x), nullptr, inv, am, red_i,
                        s_scale);
  }
}

// ---------------------------------------------------------------------------
// Fused prologue shared by a thread-block cluster.  Every CTA needs all of x_q, and with
// the whole row quantised in each of up to 296 CTAs a long row costs several us after the
// dependency wait, while the weight stream stands (each CTA reads the fp32 row from L2 two
// or three times and spends some 30 instructions per element on it: 10 us of a 26 us
// launch at K = 28672).  With C CTAs in a cluster, CTA rank r handles only the
// 16-element groups [r gw, (r + 1) gw) (gw = ceil(K / 16 / C)) and the ranks exchange
// through distributed shared memory, always by pushing into the peers' own slots so
// that no CTA reads another's shared memory:
//   (0) an arrive at kernel start, waited for before the first remote store (every CTA
//       of the cluster has then started);
//   (1) per token the largest |x| and, with RMSNorm, the float-float sum of squares of
//       the chunk, pushed to every rank; each rank combines the C values in rank order,
//       so every CTA of the cluster takes the same mean-square decision (the exact path,
//       when taken, runs over the whole row in every CTA);
//   (2) with RMSNorm, the largest |u| of the chunk the same way;
//   (3) the quantised groups, byte-transposed, stored into the xs of every rank, and the
//       chunk's sum of x_q into rank 0.
// The float-float sum has at most ceil(K / 4 / C / threads) steps per accumulator, two
// levels per thread, five per warp, a sequence of 12 over the warps and one of C over
// the ranks: well inside the error bound that the mean-square decision assumes, so a
// decided mean square is the exact one, as in one CTA.  x_q, s_x and x_sum are written by
// cluster 0.
constexpr int kMaxCluster = 4;  // clusters of 2 or 4 CTAs


template <int MT>
struct ClusterSlots {
  uint32_t mx[kMaxCluster][MT];  // [source rank][token] largest |x| bits of the chunk
  float2 ff[kMaxCluster][MT];    // float-float sum of squares of the chunk
  uint32_t am[kMaxCluster][MT];  // largest |u| bits of the chunk
  int qs[kMaxCluster][MT];       // sum of x_q over the chunk (rank 0's copy is read)
};

template <int MT, bool RMS>
__device__ __forceinline__ void cluster_prologue(const StreamArgs& a, uint4* xs, float* s_scale, ClusterSlots<MT>& cs,
                                                 uint32_t* red_u, uint32_t* red_a, float2* red_ff, int* red_i,
                                                 unsigned long long* red_lo, unsigned long long* red_hi,
                                                 uint32_t (*limb)[256], unsigned long long* hist, double* s_dbl,
                                                 float* s_inv, int* s_slow) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4, K4 = K >> 2;
  const uint32_t rank = cl_rank(), C = cl_size();
  const bool first = blockIdx.x < C;  // cluster 0 writes the optional outputs
  const int gw = (Kw + (int)C - 1) / (int)C;
  const int u0 = 4 * min(Kw, (int)rank * gw), u1 = 4 * min(Kw, ((int)rank + 1) * gw);  // float4 range
  const float4* g4 = reinterpret_cast<const float4*>(a.g);
  // padding tokens: zeros in this CTA's own xs (no rank writes them)
#pragma unroll
  for (int m = 0; m < MT; ++m)
    if (m >= a.M)
      for (int i = tid; i < Kw; i += kThreads) xs[m * Kw + i] = make_uint4(0u, 0u, 0u, 0u);

  // (1) chunk statistics
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    uint32_t mx = 0u;
    FF s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f}, s2 = {0.0f, 0.0f}, s3 = {0.0f, 0.0f};
    if (m < a.M) {
      const float4* xg = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
      for (int u = u0 + tid; u < u1; u += kThreads) {
        const float4 v = xg[u];
        mx = max(mx, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                         max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
        if (RMS) {
          ff_add_square(s0, v.x);
          ff_add_square(s1, v.y);
          ff_add_square(s2, v.z);
          ff_add_square(s3, v.w);
        }
      }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (RMS) {
      ff_add(s0, s1);
      ff_add(s2, s3);
      ff_add(s0, s2);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        FF t;
        t.hi = __shfl_xor_sync(0xffffffffu, s0.hi, o);
        t.lo = __shfl_xor_sync(0xffffffffu, s0.lo, o);
        ff_add(s0, t);
      }
    }
    if (lane == 0) {
      red_u[warp * MT + m] = mx;
      if (RMS) red_ff[warp * MT + m] = make_float2(s0.hi, s0.lo);
    }
  }
  __syncthreads();
  cl_wait();  // (0): every CTA of the cluster runs; remote stores are allowed from here
  if (tid < (int)C * MT) {  // the CTA's totals (fixed order) to rank tid / MT
    const int m = tid % MT;
    uint32_t mx = 0u;
    FF t = {0.0f, 0.0f};
    for (int w = 0; w < kWarps; ++w) {
      mx = max(mx, red_u[w * MT + m]);
      if (RMS) {
        const float2 f = red_ff[w * MT + m];
        ff_add(t, FF{f.x, f.y});
      }
    }
    const uint32_t dst = (uint32_t)(tid / MT);
    *peer(&cs.mx[rank][m], dst) = mx;
    if (RMS) *peer(&cs.ff[rank][m], dst) = make_float2(t.hi, t.lo);
  }
  cl_arrive();
  cl_wait();  // (1)
  uint32_t am[MT];
  float inv[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    am[m] = 0u;
    inv[m] = 1.0f;
  }
  if constexpr (RMS) {
    bool okm[MT];
    bool slow = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      FF t = {0.0f, 0.0f};
      for (uint32_t r = 0; r < C; ++r) {
        const float2 f = cs.ff[r][m];
        ff_add(t, FF{f.x, f.y});
      }
      float ms = 0.0f;
      okm[m] = m >= a.M || ff_mean_f32(t, K, a.inv_k, ms);
      inv[m] = okm[m] ? inv_rms_f32(ms, a.eps) : 0.0f;
      slow |= !okm[m];
    }
    if (slow) {  // cluster-uniform: every CTA combined the same values in the same order
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (!okm[m])
          inv[m] = rms_inv_exact<kWarps>(reinterpret_cast<const float4*>(a.x + (size_t)m * K), K4, a.kd, a.eps,
                                         red_u + kWarps * MT, red_lo, red_hi, limb, hist, s_dbl, s_inv, s_slow);
    }
    // (2) largest |u| of the chunk, u = fl(fl(x inv) g)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      uint32_t t = 0u;
      if (m < a.M) {
        const float4* xg = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
        for (int u = u0 + tid; u < u1; u += kThreads) {
          const float4 v = xg[u];
          const float4 gg = g4[u];
          const float4 w = make_float4(__fmul_rn(__fmul_rn(v.x, inv[m]), gg.x), __fmul_rn(__fmul_rn(v.y, inv[m]), gg.y),
                                       __fmul_rn(__fmul_rn(v.z, inv[m]), gg.z), __fmul_rn(__fmul_rn(v.w, inv[m]), gg.w));
          t = max(t, __float_as_uint(fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w)))));
        }
      }
      t = __reduce_max_sync(0xffffffffu, t);
      if (lane == 0) red_a[warp * MT + m] = t;
    }
    __syncthreads();
    if (tid < (int)C * MT) {
      const int m = tid % MT;
      uint32_t t = 0u;
      for (int w = 0; w < kWarps; ++w) t = max(t, red_a[w * MT + m]);
      *peer(&cs.am[rank][m], (uint32_t)(tid / MT)) = t;
    }
    cl_arrive();
    cl_wait();  // (2)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      for (uint32_t r = 0; r < C; ++r) am[m] = max(am[m], cs.am[r][m]);
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m)
      for (uint32_t r = 0; r < C; ++r) am[m] = max(am[m], cs.mx[r][m]);
  }

  // (3) quantise the chunk: lane l takes float4 u = base + l (base a multiple of 32, so the
  // four float4s of a group sit in lanes 4q..4q+3 and the chunk ends on a group boundary)
  int qsum[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    qsum[m] = 0;
    if (m >= a.M) continue;
    const float amax = __uint_as_float(am[m]);
    // the conversion-free rounding of the single-CTA quantisation, with the same checks
    float ra = amax == 0.0f ? 0.0f : __int_as_float(0x7fffffff);
    if (amax >= 0x1p-120f && amax <= 0x1p120f) asm("rcp.approx.f32 %0, %1;" : "=f"(ra) : "f"(amax));
    const float4* xg = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
    uint32_t* qout = a.x_q_out ? reinterpret_cast<uint32_t*>(a.x_q_out + (size_t)m * K) : nullptr;
    for (int base = u0 + warp * 32; base < u1; base += kThreads) {  // warp-uniform trip count
      const int u = base + lane;
      const bool act = u < u1;
      float e[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      uint32_t pq = 0u;
      bool near = false;
      if (act) {
        const float4 v = xg[u];
        if (RMS) {
          const float4 gg = g4[u];
          e[0] = __fmul_rn(__fmul_rn(v.x, inv[m]), gg.x);
          e[1] = __fmul_rn(__fmul_rn(v.y, inv[m]), gg.y);
          e[2] = __fmul_rn(__fmul_rn(v.z, inv[m]), gg.z);
          e[3] = __fmul_rn(__fmul_rn(v.w, inv[m]), gg.w);
        } else {
          e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float d = __fmul_rn(__fmul_rn(e[j], 127.0f), ra);
          const float sb = __fadd_rn(d, 12582912.0f);  // d + 1.5 2^23: rounds d to an integer
          near |= !(fabsf(__fsub_rn(d, __fsub_rn(sb, 12582912.0f))) < 0.49995f);  // also non-finite d
          const int t = (int)(__float_as_uint(sb) & 0x7fffffu) - 0x400000;
          pq |= ((uint32_t)max(-128, min(127, t)) & 0xffu) << (8 * j);
        }
      }
      if (__any_sync(0xffffffffu, near) && near) {  // rare: the IEEE divide
        pq = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = amax > 0.0f ? __float2int_rn(__fdiv_rn(__fmul_rn(e[j], 127.0f), amax)) : 0;
          pq |= ((uint32_t)max(-128, min(127, t)) & 0xffu) << (8 * j);
        }
      }
      const uint32_t p1 = __shfl_down_sync(0xffffffffu, pq, 1);
      const uint32_t p2 = __shfl_down_sync(0xffffffffu, pq, 2);
      const uint32_t p3 = __shfl_down_sync(0xffffffffu, pq, 3);
      if (act) {
        qsum[m] += (int)(int8_t)(pq & 0xffu) + (int)(int8_t)((pq >> 8) & 0xffu) + (int)(int8_t)((pq >> 16) & 0xffu) +
                   (int)(int8_t)(pq >> 24);
        if (first && qout) qout[u] = pq;
        if ((lane & 3) == 0) {
          const uint4 grp = permute_group(make_uint4(pq, p1, p2, p3));
          uint4* dst = xs + m * Kw + (u >> 2);
          for (uint32_t r = 0; r < C; ++r) *peer(dst, r) = grp;
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    qsum[m] = __reduce_add_sync(0xffffffffu, qsum[m]);
    if (lane == 0) red_i[warp * MT + m] = qsum[m];
  }
  __syncthreads();
  if (tid < MT) {
    int t = 0;
    for (int w = 0; w < kWarps; ++w) t += red_i[w * MT + tid];
    *peer(&cs.qs[rank][tid], 0u) = t;
    s_scale[tid] = __uint_as_float(am[tid]);
  }
  cl_arrive();
  cl_wait();  // (3): xs complete in every CTA of the cluster
  if (blockIdx.x == 0 && tid < a.M) {
    if (a.x_sum_out) {
      int t = 0;
      for (uint32_t r = 0; r < C; ++r) t += cs.qs[r][tid];
      a.x_sum_out[tid] = t;
    }
    if (a.s_x_out) a.s_x_out[tid] = __uint_as_float(am[tid]);
  }
}

// CL: launched in clusters of 2 or 4 CTAs that share the fused prologue (cluster_prologue).
template <int MT, int JMAX, int PRE, bool FUSED, bool RMS, bool CL = false>
__global__ void __launch_bounds__(kThreads, 2) gemv_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4;
  const int c = blockIdx.x;
  const int nrows = a.rows_base + (c < a.rows_rem ? 1 : 0);
  const int row0 = c * a.rows_base + min(c, a.rows_rem);
  uint4* xs = reinterpret_cast<uint4*>(smem + a.xs_off);  // [MT][Kw] byte-transposed x_q
  int* sacc = reinterpret_cast<int*>(smem + a.acc_off);   // [nrows][MT] row totals
  __shared__ uint32_t red_u[kWarps * MT + (RMS ? kWarps : 0)];
  __shared__ uint32_t red_a[RMS ? kWarps * MT : 1];
  __shared__ float2 red_ff[RMS ? kWarps * MT : 1];
  __shared__ int red_i[kWarps * MT];
  __shared__ unsigned long long red_lo[RMS ? kWarps : 1], red_hi[RMS ? kWarps : 1];
  __shared__ float s_scale[MT];
  __shared__ float s_inv[MT];
  __shared__ int s_slow[1];
  __shared__ double s_dbl;
  __shared__ uint32_t limb[RMS ? 3 : 1][256];
  __shared__ unsigned long long hist[RMS ? 256 : 1];
  __shared__ ClusterSlots<CL ? MT : 1> cslots;

  pdl_launch_dependents();
  if constexpr (CL) cl_arrive_relaxed();  // (0) of the cluster prologue

  // ---------------------------------------------------------------- rows of this warp
  const int S = a.S, G = kWarps / S;
  const int sl = warp % S, gr = warp / S;
  const int Ws = (Kw + S - 1) / S;
  const int ws0 = sl * Ws, ws1 = min(Kw, ws0 + Ws);
  const int nr = nrows > gr ? (nrows - gr + G - 1) / G : 0;  // rows of this group
  const uint32_t* Wp = reinterpret_cast<const uint32_t*>(a.packed) + (size_t)row0 * Kw;
  const uint64_t pol = l2_evict_first_policy();

  // Word j of a row for this lane is at ws0 + lane + 32 j: one address per row, the words at
  // immediate offsets, each load predicated on bit j of wok (the word lies in the K slice).
  // Words outside the slice are not loaded and meet x = 0; rows past the group's end read
  // its first row again (their sums are never formed).
  uint32_t wv[PRE][JMAX];
  uint32_t wok = 0u;
#pragma unroll
  for (int j = 0; j < JMAX; ++j)
    if (ws0 + lane + 32 * j < ws1) wok |= 1u << j;
  const uint32_t* Wl = Wp + (size_t)gr * Kw + ws0 + lane;
  const size_t rstride = (size_t)G * Kw;
  // One token: the registers hold two halves of H = PRE / 2 rows each; half h (rows h H ..
  // h H + H - 1 of the group) goes to buffer h % 2 and is reloaded with half h + 2 as soon as it
  // has been multiplied, so that one half is in flight while the other is computed (measured:
  // the 70B gate|up product 26.8 -> 25.7 us).  Two to four tokens: one buffer of PRE rows,
  // reloaded after it has been multiplied (the halves measured slower there: 43.4 -> 49.0 us
  // at two tokens).
  constexpr bool kHalves = MT == 1;
  constexpr int H = kHalves ? PRE / 2 : PRE;
  static_assert(!kHalves || PRE % 2 == 0, "two halves");
  auto load_half = [&](int h, int buf) {
#pragma unroll
    for (int q = 0; q < H; ++q) {
      const int i = h * H + q;
      ld_row_words(wv[buf * H + q], Wl + (size_t)(i < nr ? i : 0) * rstride, wok, pol,
                   std::make_integer_sequence<int, JMAX>{});
    }
  };
  // weights (and their scale) do not depend on the previous kernel: start streaming now
  if (nr > 0) {
    load_half(0, 0);
    if (kHalves) load_half(1, 1);
  }
  const float gam = __ldg(a.w_scale);

  for (int i = tid; i < nrows * MT; i += kThreads) sacc[i] = 0;
  if constexpr (FUSED) {
    // The RMSNorm gain, like the weights, is a parameter: stage it now.  x may come from
    // the previous kernel, so it is only prefetched into L2 (coherent; no data is read
    // into the SM before the wait).
    if (RMS && a.xf_off >= 0) {
      float4* gst = reinterpret_cast<float4*>(smem + a.xf_off) + (size_t)MT * (K >> 2);
      const float4* gg = reinterpret_cast<const float4*>(a.g);
      for (int i = tid; i < (K >> 2); i += kThreads) gst[i] = __ldg(gg + i);
    }
    for (int i = tid; i < a.M * (K >> 5); i += kThreads)  // one 128-byte line per thread
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.x + (size_t)i * 32) : "memory");
    if (RMS && a.xf_off < 0) {
      for (int i = tid; i < (K >> 5); i += kThreads) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.g + (size_t)i * 32) : "memory");
    }
  }
  pdl_wait();  // activations and outputs may belong to the previous kernel

  // ---------------------------------------------------------------- activations -> xs
  if constexpr (!FUSED) {
    for (int m = 0; m < MT; ++m) {
      if (m < a.M) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x_q_in + (size_t)m * K);
        for (int i = tid; i < Kw; i += kThreads) xs[m * Kw + i] = permute_group(src[i]);
      } else {
        for (int i = tid; i < Kw; i += kThreads) xs[m * Kw + i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (tid < MT) s_scale[tid] = tid < a.M ? a.s_x_in[tid] : 0.0f;
  } else if constexpr (CL) {
    cluster_prologue<MT, RMS>(a, xs, s_scale, cslots, red_u, red_a, red_ff, red_i, red_lo, red_hi, limb, hist,
                              &s_dbl, s_inv, s_slow);
  } else {
    float* xf = a.xf_off >= 0 ? reinterpret_cast<float*>(smem + a.xf_off) : nullptr;
    fused_prologue<MT, RMS>(a, xs, xf, s_scale, red_u, red_a, red_ff, red_i, red_lo, red_hi, limb, hist, &s_dbl,
                            s_inv, s_slow);
  }
  __syncthreads();

  // ---------------------------------------------------------------- x slice -> registers
  uint4 xr[JMAX][MT];
  int lane_xsum[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) lane_xsum[m] = 0;
#pragma unroll
  for (int j = 0; j < JMAX; ++j) {
    const int wi = ws0 + lane + 32 * j;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      xr[j][m] = (wi < ws1) ? xs[m * Kw + wi] : make_uint4(0u, 0u, 0u, 0u);
      lane_xsum[m] += byte_sum16(xr[j][m]);
    }
  }

  // ---------------------------------------------------------------- dot products
  // the H rows of half h from buffer buf
  auto rows_of = [&](int h, int buf) {
#pragma unroll
    for (int q = 0; q < H; ++q) {
      const int i = h * H + q;
      if (i >= nr) break;  // warp-uniform
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0;
#pragma unroll
      for (int j = 0; j < JMAX; ++j) {
        const uint32_t w = wv[buf * H + q][j];
        const uint32_t c0 = w & 0x03030303u, c1 = w & 0x0C0C0C0Cu;
        const uint32_t c2 = w & 0x30303030u, c3 = w & 0xC0C0C0C0u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          acc[m][0] = dp4a_us(c0, xr[j][m].x, acc[m][0]);
          acc[m][1] = dp4a_us(c1, xr[j][m].y, acc[m][1]);
          acc[m][2] = dp4a_us(c2, xr[j][m].z, acc[m][2]);
          acc[m][3] = dp4a_us(c3, xr[j][m].w, acc[m][3]);
        }
      }
      // words outside the K slice meet x = 0; lane_xsum covers exactly the words this lane
      // multiplied.  acc[m][s] is 4^s times an integer: the shifts are exact.
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int t = acc[m][0] + (acc[m][1] >> 2) + (acc[m][2] >> 4) + (acc[m][3] >> 6) - lane_xsum[m];
        const int tot = __reduce_add_sync(0xffffffffu, t);
        if (lane == 0) {
          const int r = gr + i * G;
          if (S == 1) sacc[r * MT + m] = tot;
          else atomicAdd(&sacc[r * MT + m], tot);
        }
      }
    }
  };
  const int nh = (nr + H - 1) / H;
  if constexpr (kHalves) {
    for (int h = 0; h < nh; h += 2) {
      rows_of(h, 0);
      if (h + 2 < nh) load_half(h + 2, 0);
      if (h + 1 < nh) {
        rows_of(h + 1, 1);
        if (h + 3 < nh) load_half(h + 3, 1);
      }
    }
  } else {
    for (int h = 0; h < nh; ++h) {
      if (h > 0) load_half(h, 0);
      rows_of(h, 0);
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- epilogue (coalesced)
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m >= a.M) break;
    const float sm = s_scale[m];
    const float c = dequant_scale(gam, sm);  // once per token, not per output
    for (int r = tid; r < nrows; r += kThreads) {
      const int acc = sacc[r * MT + m];
      const size_t o = (size_t)m * a.N + row0 + r;
      a.y[o] = dequant(acc, c, gam, sm);
      if (a.acc_out) a.acc_out[o] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// One token (the decode step): the CTA's weight block copied into shared memory before
// the dependency wait, a lean fused prologue, and per-warp row outputs.
//
// * A CTA owns a contiguous block of rows (contiguous in the packed tensor); one thread
//   copies all of it into shared memory with cp.async.bulk (completion on an mbarrier)
//   before griddepcontrol.wait, so the weight stream of this GEMV runs while the previous
//   kernel finishes, without holding registers.  Everything else that does not depend on
//   the previous kernel (the RMSNorm gain, the row mapping) is also prepared before the
//   wait.  Used when the block fits (a 2B-shaped layer, 8B q|k|v and o); longer streams
//   take gemv_stream_kernel.  The kernel is kept small: its code is fetched afresh after
//   every dependency wait, and a larger body measurably lengthened that wait.
// * After the wait every thread loads its NV float4s of x (all loads in flight at once:
//   one L2 round trip).
// * Pass 1 (registers only): per warp either the largest |x| (no RMSNorm: that is a) or,
//   with RMSNorm, the float-float sum of squares and the float4 holding the largest
//   p = fl(|x| |g|).  After the first barrier every warp combines the per-warp results
//   itself (same values, same order: the same result in every warp).  With RMSNorm the
//   scale a = max_k |u_k|, u_k = fl(fl(x_k inv) g_k), is first taken over that float4:
//   both roundings are relative errors of at most 2^-24 for normal results, so only an
//   element whose p lies within a few units of 2^-24 of the largest one can have a
//   larger |u|.  The quantisation pass checks |u_k| <= a for every element it quantises
//   anyway; when some element exceeds it (near-ties, underflow) the block takes the
//   maximum over all elements and quantises once more.  Two block barriers in the
//   common case, whatever RMSNorm, and the result is always exact.
// * Dot products from shared memory, up to four rows at a time (independent chains,
//   no padded rows computed); a warp that owns whole rows writes their outputs itself.
constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;

struct DecodeRed {
  float2 ff[kDecWarps];   // per-warp float-float sums of squares
  uint32_t pm[kDecWarps]; // per-warp largest p (RMSNorm) or |x|, as bits
  float4 cx[kDecWarps];   // per-warp candidate float4 of x ...
  float4 cg[kDecWarps];   // ... and of the gain
  uint32_t am[kDecWarps]; // re-check: per-warp largest |u|
  int qs[kDecWarps];      // per-warp sums of x_q
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool dec_mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase (2 s of wall time).
__device__ __forceinline__ bool dec_mbar_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (dec_mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
}

// The unit (float4 index of x) of this thread's float4 q.
__device__ __forceinline__ int dec_unit(int q) { return q * kDecThreads + (int)threadIdx.x; }

// Quantises this thread's float4s of x (registers xv, and the gain gv when RMS) with scale
// amax into xs (and x_q_out when wout).  Returns the thread's sum of x_q; sets viol when
// `check` and some |u| > amax.
template <bool RMS, int NV>
__device__ __forceinline__ int decode_quantise(const StreamArgs& a, uint4* xs, const float4 (&xv)[NV],
                                               const float4 (&gv)[NV], float inv, float amax, float ra,
                                               bool check, bool& viol, bool wout) {
  const int K4 = a.K >> 2;
  unsigned char* xsb = reinterpret_cast<unsigned char*>(xs);
  // d = fl(fl(u 127) ra) is within 2^-22 |d| < 3.1e-5 of fl(u 127) / a (|d| <= 127 once
  // |u| <= a); when it is at least 5e-5 from a half-integer, rounding d gives
  // round_half_even(fl32(fl(u 127) / a)).  Rounding by adding 1.5 2^23: the integer is then
  // in the low mantissa bits, its two's-complement low byte in the low byte of the sum.
  // Units with an element nearer a half-integer (or a non-finite d) take the IEEE divide.
  uint32_t pq[NV];
  bool near[NV];
  bool any = false, bad = false;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const bool valid = dec_unit(q) < K4;
    float4 v = valid ? xv[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (RMS) {
      const float4 gg = gv[q];
      v = make_float4(__fmul_rn(__fmul_rn(v.x, inv), gg.x), __fmul_rn(__fmul_rn(v.y, inv), gg.y),
                      __fmul_rn(__fmul_rn(v.z, inv), gg.z), __fmul_rn(__fmul_rn(v.w, inv), gg.w));
      if (check && valid) bad |= fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) > amax;
    }
    const float d0 = __fmul_rn(__fmul_rn(v.x, 127.0f), ra), d1 = __fmul_rn(__fmul_rn(v.y, 127.0f), ra);
    const float d2 = __fmul_rn(__fmul_rn(v.z, 127.0f), ra), d3 = __fmul_rn(__fmul_rn(v.w, 127.0f), ra);
    const float s0 = __fadd_rn(d0, 12582912.0f), s1 = __fadd_rn(d1, 12582912.0f);
    const float s2 = __fadd_rn(d2, 12582912.0f), s3 = __fadd_rn(d3, 12582912.0f);
    const float e = fmaxf(fmaxf(fabsf(__fsub_rn(d0, __fsub_rn(s0, 12582912.0f))),
                                fabsf(__fsub_rn(d1, __fsub_rn(s1, 12582912.0f)))),
                          fmaxf(fabsf(__fsub_rn(d2, __fsub_rn(s2, 12582912.0f))),
                                fabsf(__fsub_rn(d3, __fsub_rn(s3, 12582912.0f)))));
    near[q] = valid && !(e < 0.49995f);  // also when some d is not finite
    any |= near[q];
    pq[q] = __byte_perm(__byte_perm(__float_as_uint(s0), __float_as_uint(s1), 0x0040u),
                        __byte_perm(__float_as_uint(s2), __float_as_uint(s3), 0x0040u), 0x5410u);
  }
  if (__any_sync(0xffffffffu, any) && any) {  // rare: the IEEE divide for units near a tie
    auto q_exact = [&](float uv) -> uint32_t {
      const int t = amax > 0.0f ? __float2int_rn(__fdiv_rn(__fmul_rn(uv, 127.0f), amax)) : 0;
      return (uint32_t)max(-128, min(127, t)) & 0xffu;
    };
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      if (near[q]) {
        float4 v = xv[q];
        if (RMS) {
          const float4 gg = gv[q];
          v = make_float4(__fmul_rn(__fmul_rn(v.x, inv), gg.x), __fmul_rn(__fmul_rn(v.y, inv), gg.y),
                          __fmul_rn(__fmul_rn(v.z, inv), gg.z), __fmul_rn(__fmul_rn(v.w, inv), gg.w));
        }
        pq[q] = q_exact(v.x) | (q_exact(v.y) << 8) | (q_exact(v.z) << 16) | (q_exact(v.w) << 24);
      }
    }
  }
  int qsum = 0;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const int u = dec_unit(q);
    if (u < K4) {
      qsum = __dp4a((int)pq[q], 0x01010101, qsum);
      if (wout && a.x_q_out) reinterpret_cast<uint32_t*>(a.x_q_out)[u] = pq[q];
      // element k of 16-element group k/16 goes to byte (k/4) % 4 of word k % 4
      unsigned char* gb = xsb + (u >> 2) * 16 + (u & 3);
      gb[0] = (unsigned char)pq[q];
      gb[4] = (unsigned char)(pq[q] >> 8);
      gb[8] = (unsigned char)(pq[q] >> 16);
      gb[12] = (unsigned char)(pq[q] >> 24);
    }
  }
  viol = bad;
  return qsum;
}

// The one-token prologue: x (fp32, global) -> xs (byte-transposed int8 groups).  Returns
// a = max |u|; sets *cs to the dequantisation scale fl(fl(gamma a) / 127) and *xtot to the
// sum of x_q over the whole row.  A thread's float4s are units dec_unit(q), q < NV
// (NV * kDecThreads >= K / 4); gv holds the gain's (RMS: loaded before the dependency wait).
// STATS (RMS only): the sum of squares and the scale candidate come from the partials a
// residual epilogue left (a.parts_in): no first pass over x and no block reduction.
template <bool RMS, int NV, bool STATS = false>
__device__ __forceinline__ float decode_prologue(const StreamArgs& a, uint4* xs, float4 (&gv)[NV], DecodeRed& r,
                                                 uint32_t* red_u, unsigned long long* red_lo,
                                                 unsigned long long* red_hi, uint32_t (*limb)[256],
                                                 unsigned long long* hist, double* s_dbl, float* s_inv,
                                                 int* s_slow, float gam, float* cs, int* xtot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;
  const int K = a.K, K4 = K >> 2;
  const float4* xg = reinterpret_cast<const float4*>(a.x);
  static_assert(!STATS || RMS, "finished statistics are those of an RMSNorm");
  float4 xv[NV];
#pragma unroll
  for (int q = 0; q < NV; ++q) xv[q] = dec_unit(q) < K4 ? __ldcg(xg + dec_unit(q)) : make_float4(0.f, 0.f, 0.f, 0.f);

  float amax, inv = 1.0f;
  {
  // ---- pass 1 (padding float4s are zero: they add nothing).  STATS: thread t takes the
  // residual epilogue's partial t instead (a float-float sum of squares and the element
  // with the largest fl(|h g|)), and everything below is the same.
  FF s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f}, s2 = {0.0f, 0.0f}, s3 = {0.0f, 0.0f};
  float pmf = 0.0f;
  float4 cxv = make_float4(0.f, 0.f, 0.f, 0.f), cgv = cxv;
  if constexpr (STATS) {
    if (tid < a.nparts) {
      const float4 pp = __ldcg(a.parts_in + tid);
      s0.hi = pp.x;
      s0.lo = pp.y;
      pmf = fabsf(__fmul_rn(pp.z, pp.w));
      cxv.x = pp.z;
      cgv.x = pp.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const float4 v = xv[q];
      if (RMS) {
        const float4 gg = gv[q];
        ff_add_square(s0, v.x);  // one chain per component
        ff_add_square(s1, v.y);
        ff_add_square(s2, v.z);
        ff_add_square(s3, v.w);
        const float m = fmaxf(fmaxf(fabsf(__fmul_rn(v.x, gg.x)), fabsf(__fmul_rn(v.y, gg.y))),
                              fmaxf(fabsf(__fmul_rn(v.z, gg.z)), fabsf(__fmul_rn(v.w, gg.w))));
        if (m > pmf) {
          pmf = m;
          cxv = v;
          cgv = gg;
        }
      } else {
        pmf = fmaxf(pmf, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
  }
  const uint32_t pm = __float_as_uint(pmf);  // >= 0: compares as its bits
  const uint32_t wm = __reduce_max_sync(full, pm);
  if (RMS) {
    ff_add(s0, s1);
    ff_add(s2, s3);
    ff_add(s0, s2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      FF t;
      t.hi = __shfl_xor_sync(full, s0.hi, o);
      t.lo = __shfl_xor_sync(full, s0.lo, o);
      ff_add(s0, t);
    }
    if (lane == __ffs(__ballot_sync(full, pm == wm)) - 1) {
      r.cx[warp] = cxv;
      r.cg[warp] = cgv;
    }
    if (lane == 0) r.ff[warp] = make_float2(s0.hi, s0.lo);
  }
  if (lane == 0) r.pm[warp] = wm;
  __syncthreads();  // (1) per-warp results

  // ---- every warp: combine (kDecWarps <= 16 partials, one per lane)
  const uint32_t ml = lane < kDecWarps ? r.pm[lane] : 0u;
  const uint32_t bm = __reduce_max_sync(full, ml);
  if constexpr (!RMS) {
    amax = __uint_as_float(bm);
  } else {
    FF t;
    t.hi = t.lo = 0.0f;
    if (lane < kDecWarps) {
      const float2 f = r.ff[lane];
      t.hi = f.x;
      t.lo = f.y;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      FF u;
      u.hi = __shfl_xor_sync(full, t.hi, o);
      u.lo = __shfl_xor_sync(full, t.lo, o);
      ff_add(t, u);
    }
    t.hi = __shfl_sync(full, t.hi, 0);  // the same decision in every thread of the block
    t.lo = __shfl_sync(full, t.lo, 0);
    float ms = 0.0f;
    if (ff_mean_f32(t, K, a.inv_k, ms)) {
      inv = inv_rms_f32(ms, a.eps);
    } else {  // block-uniform; reads x again (from L2)
      inv = rms_inv_exact<kDecWarps>(xg, K4, a.kd, a.eps, red_u, red_lo, red_hi, limb, hist, s_dbl, s_inv, s_slow);
    }
    const int wsel = __ffs(__ballot_sync(full, lane < kDecWarps && ml == bm)) - 1;
    const float4 v = r.cx[wsel], gg = r.cg[wsel];
    amax = fmaxf(fmaxf(fabsf(__fmul_rn(__fmul_rn(v.x, inv), gg.x)), fabsf(__fmul_rn(__fmul_rn(v.y, inv), gg.y))),
                 fmaxf(fabsf(__fmul_rn(__fmul_rn(v.z, inv), gg.z)), fabsf(__fmul_rn(__fmul_rn(v.w, inv), gg.w))));
  }
  }
  *cs = dequant_scale(gam, amax);

  // ---- quantisation.  With RMSNorm the first pass checks the candidate scale; when some
  // |u| exceeded it (block-uniform, rare) a is taken over all elements and the same code
  // quantises once more.
  for (int pass = 0;; ++pass) {
    float ra = amax == 0.0f ? 0.0f : __int_as_float(0x7fffffff);
    if (amax >= 0x1p-120f && amax <= 0x1p120f) asm("rcp.approx.f32 %0, %1;" : "=f"(ra) : "f"(amax));
    bool bad = false;
    int qs = decode_quantise<RMS, NV>(a, xs, xv, gv, inv, amax, ra, RMS && pass == 0, bad, blockIdx.x == 0);
    qs = __reduce_add_sync(full, qs);
    if (lane == 0) r.qs[warp] = qs;
    const bool viol = __syncthreads_or(bad);  // (2) xs and the per-warp sums complete
    if (!RMS || pass > 0 || !viol) break;
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const float4 v = xv[q], gg = gv[q];
      m = fmaxf(m, fmaxf(fmaxf(fabsf(__fmul_rn(__fmul_rn(v.x, inv), gg.x)), fabsf(__fmul_rn(__fmul_rn(v.y, inv), gg.y))),
                         fmaxf(fabsf(__fmul_rn(__fmul_rn(v.z, inv), gg.z)), fabsf(__fmul_rn(__fmul_rn(v.w, inv), gg.w)))));
    }
    const uint32_t am = __reduce_max_sync(full, __float_as_uint(m));
    if (lane == 0) r.am[warp] = am;
    __syncthreads();  // also: every warp has read r.qs of the first pass
    amax = __uint_as_float(__reduce_max_sync(full, lane < kDecWarps ? r.am[lane] : 0u));
    *cs = dequant_scale(gam, amax);
  }
  *xtot = __reduce_add_sync(full, lane < kDecWarps ? r.qs[lane] : 0);
  if (blockIdx.x == 0 && tid == 0) {
    if (a.s_x_out) a.s_x_out[0] = amax;
    if (a.x_sum_out) a.x_sum_out[0] = *xtot;
  }
  return amax;
}

// R rows of one warp (rows i0 .. i0+R-1 of its group, in the chunk at wsm): per-lane partial
// dot products from shared memory, then one warp sum per row.  Words of the lane's range
// past its K slice meet x = 0 there, so their (arbitrary) weights add nothing.
template <int JMAX, int R>
__device__ __forceinline__ void decode_rows(const uint32_t* wsm, int Kw, int G, int gr, int i0, int wbase,
                                            const uint4 (&xr)[JMAX], int (&tot)[4]) {
  int acc[R][4];
#pragma unroll
  for (int q = 0; q < R; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0;
#pragma unroll
  for (int j = 0; j < JMAX; ++j) {
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const uint32_t w = wsm[(size_t)(gr + (i0 + q) * G) * Kw + wbase + 32 * j];
      acc[q][0] = dp4a_us(w & 0x03030303u, xr[j].x, acc[q][0]);
      acc[q][1] = dp4a_us(w & 0x0C0C0C0Cu, xr[j].y, acc[q][1]);
      acc[q][2] = dp4a_us(w & 0x30303030u, xr[j].z, acc[q][2]);
      acc[q][3] = dp4a_us(w & 0xC0C0C0C0u, xr[j].w, acc[q][3]);
    }
  }
  // acc_s is 4^s times an integer: the shifts are exact.  tot = sum of c x over the warp's
  // K slice (c = t + 1); the caller subtracts sum x once per row.
#pragma unroll
  for (int q = 0; q < R; ++q)
    tot[q] = __reduce_add_sync(0xffffffffu, acc[q][0] + (acc[q][1] >> 2) + (acc[q][2] >> 4) + (acc[q][3] >> 6));
}

// y = acc gamma s_x / 127 as the definition states it: ((acc gamma) s_x) / 127 in double,
// then rounded to fp32 (the residual epilogue adds exactly this value).  The two products
// are double multiplies (the first is exact); the division by 127 and both roundings are
// done with integers (div_k_round_f32, d127 = make_kdiv(127)), so no double-precision
// divide runs on this part's narrow double pipe.  |p| lies in [2^-298, 2^280]: a normal double.
__device__ __forceinline__ float dequant_exact(int acc, float gamma, float s_x, const KDiv& d127) {
  const double p = __dmul_rn(__dmul_rn((double)acc, (double)gamma), (double)s_x);
  const unsigned long long b = (unsigned long long)__double_as_longlong(p);
  if (p == 0.0) return (b >> 63) ? -0.0f : 0.0f;  // the signed zero of the double expression
  const int be = (int)((b >> 52) & 0x7ffull);
  const float q = div_k_round_f32((b & ((1ull << 52) - 1)) | (1ull << 52), be - 1075, d127);
  return (b >> 63) ? -q : q;
}

// Residual epilogue, after the CTA's rows of res_out are written (hb: their values, gb: the
// next gain at those rows): warp 0 stores the CTA's partial statistics (float-float sum of
// squares, and the element with the largest fl(|h g|)).  Nothing waits: the launch that reads
// the partials does so after griddepcontrol.wait, when this whole grid has finished.
__device__ __forceinline__ void decode_epilogue(const StreamArgs& a, int nrows, const float* hb, const float* gb) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  FF t = {0.0f, 0.0f};
  float pmf = 0.0f, hc = 0.0f, gc = 0.0f;
  for (int rr = lane; rr < nrows; rr += 32) {
    const float h = hb[rr], gg = gb[rr];
    ff_add_square(t, h);
    const float pv = fabsf(__fmul_rn(h, gg));
    if (pv > pmf) {
      pmf = pv;
      hc = h;
      gc = gg;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF u;
    u.hi = __shfl_xor_sync(full, t.hi, o);
    u.lo = __shfl_xor_sync(full, t.lo, o);
    ff_add(t, u);
  }
  const uint32_t pm = __float_as_uint(pmf);
  const uint32_t wm = __reduce_max_sync(full, pm);
  const int sel = __ffs(__ballot_sync(full, pm == wm)) - 1;
  hc = __shfl_sync(full, hc, sel);
  gc = __shfl_sync(full, gc, sel);
  if (lane == 0) a.parts_out[blockIdx.x] = make_float4(t.hi, t.lo, hc, gc);
}

// The fused one-token GEMV (see above).  Dynamic shared memory: the CTA's packed rows at
// offset 0 (plus slack for the last row's reads past its slice), xs (a.xs_off), the row
// totals (a.acc_off, used when S > 1), and with the residual epilogue the CTA's res_out and
// g_next values (a.h_off).
// MODE 0: as above.  MODE 1: residual epilogue (y exact as defined; res_out = fl(res + y);
// partial statistics for the next RMSNorm).  MODE 2: RMSNorm from the partial statistics a
// residual epilogue left for x (no first pass over x, no block reduction before quantising).
template <int JMAX, int NV, bool RMS, int MODE = 0>
__global__ void __launch_bounds__(kDecThreads, 2) gemv_decode_kernel(StreamArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4;
  const int c = blockIdx.x;
  const int nrows = a.rows_base + (c < a.rows_rem ? 1 : 0);
  const int row0 = c * a.rows_base + min(c, a.rows_rem);
  const uint32_t* wsm = reinterpret_cast<const uint32_t*>(smem);  // [nrows][Kw] packed words
  uint4* xs = reinterpret_cast<uint4*>(smem + a.xs_off);         // [Kw] byte-transposed x_q
  int* sacc = reinterpret_cast<int*>(smem + a.acc_off);          // [nrows] (S > 1)
  __shared__ DecodeRed red;
  __shared__ __align__(8) unsigned long long wbar;
  constexpr bool kExact = RMS;  // the exact RMSNorm fallback may run
  __shared__ uint32_t red_u[kExact ? kDecWarps : 1];
  __shared__ unsigned long long red_lo[kExact ? kDecWarps : 1], red_hi[kExact ? kDecWarps : 1];
  __shared__ float s_inv[1];
  __shared__ int s_slow[1];
  __shared__ double s_dbl;
  __shared__ uint32_t limb[kExact ? 3 : 1][256];
  __shared__ unsigned long long hist[kExact ? 256 : 1];
  float* hb = reinterpret_cast<float*>(smem + a.h_off);  // MODE 1: [nrows] res_out values, then [nrows] g_next

  pdl_launch_dependents();

  // ---- the weights, their scale and the RMSNorm gain are parameters: fetch them now
  const uint32_t bar = smem_addr(&wbar);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t total = (uint32_t)nrows * (uint32_t)(K >> 2);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(total) : "memory");
    const unsigned char* src = a.packed + (size_t)row0 * (K >> 2);
    for (uint32_t off = 0; off < total; off += 32768u) {
      const uint32_t n = min(32768u, total - off);
      asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       smem_addr(smem + off)),
                   "l"(src + off), "r"(n), "r"(bar)
                   : "memory");
    }
  }
  const float gam = __ldg(a.w_scale);
  const int S = a.S, G = kDecWarps / S;
  if (S > 1)
    for (int i = tid; i < nrows; i += kDecThreads) sacc[i] = 0;
  if constexpr (MODE == 1) {  // the next gain at this CTA's rows is a parameter too
    for (int i = tid; i < nrows; i += kDecThreads) {
      hb[i] = 0.0f;
      hb[nrows + i] = __ldg(a.g_next + row0 + i);
    }
  }
  if (MODE == 1 && S == 1)
    for (int i = tid; i < nrows; i += kDecThreads) sacc[i] = 0;
  float4 gv[NV];  // this thread's float4s of the RMSNorm gain
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const int u = dec_unit(q);
    gv[q] = (RMS && u < (K >> 2)) ? __ldg(reinterpret_cast<const float4*>(a.g) + u) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // the rows and K slice of this warp (integer divisions are slow here: before the wait)
  const int sl = warp % S, gr = warp / S;
  const int Ws = (Kw + S - 1) / S;
  const int ws0 = sl * Ws, ws1 = min(Kw, ws0 + Ws);
  const int nr = nrows > gr ? (nrows - gr + G - 1) / G : 0;  // rows of this group
  // x may come from the previous kernel: only prefetched into the coherent L2 before the wait
  for (int i = tid; i < (K >> 5); i += kDecThreads)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.x + (size_t)i * 32) : "memory");
  pdl_wait();
  float resv = 0.0f;  // MODE 1: the residual at this thread's row (rows one per thread), in flight with x
  if (MODE == 1 && tid < nrows) resv = __ldcg(a.res + row0 + tid);

  float cs;
  int xtot;
  const float amax = decode_prologue<RMS, NV, MODE == 2>(a, xs, gv, red, red_u, red_lo, red_hi, limb, hist, &s_dbl,
                                                          s_inv, s_slow, gam, &cs, &xtot);
  // one row's outputs (MODE 1: y as defined, then the residual; rv = res at that row)
  auto store_row = [&](int rr, int acc, float rv) {
    const int n = row0 + rr;
    if constexpr (MODE == 1) {
      const float yv = dequant_exact(acc, gam, amax, a.kd127);
      const float hv = __fadd_rn(rv, yv);
      a.res_out[n] = hv;
      hb[rr] = hv;
      if (a.y) a.y[n] = yv;
    } else {
      a.y[n] = dequant(acc, cs, gam, amax);
    }
    if (a.acc_out) a.acc_out[n] = acc;
  };
  const bool cs_normal = cs >= 1.17549435e-38f;

  uint4 xr[JMAX];
#pragma unroll
  for (int j = 0; j < JMAX; ++j) {
    const int wi = ws0 + lane + 32 * j;
    xr[j] = (wi < ws1) ? xs[wi] : make_uint4(0u, 0u, 0u, 0u);
  }

  // every thread that reads the copied rows waits on the mbarrier (bounded); a warp gives
  // up only as a whole
  const bool arrived = __all_sync(0xffffffffu, dec_mbar_wait(bar, 0));
  if (!arrived && lane == 0) atomicCAS(&g_stream_status, 0, (int)TW_ERR_TIMEOUT);
  if (arrived) {
    auto emit = [&](int i0, int n, const int (&tot)[4]) {
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < n) {
            const int rr = gr + (i0 + q) * G;  // row within the CTA
            if (MODE == 1 && S == 1) {
              sacc[rr] = tot[q];  // outputs below, one row per thread
            } else if (S == 1) {
              const int acc = tot[q] - xtot;
              a.y[row0 + rr] = cs_normal ? __fmul_rn((float)acc, cs) : dequant_tiny(acc, gam, amax);
              if (a.acc_out) a.acc_out[row0 + rr] = acc;
            } else {
              atomicAdd(&sacc[rr], tot[q]);
            }
          }
        }
      }
    };
    // RB rows at a time (independent chains) while that many remain, then one by one
    constexpr int RB = JMAX <= 5 ? 4 : 2;
    const int wbase = ws0 + lane;
    int i0 = 0;
    int tot[4];
    for (; i0 + RB <= nr; i0 += RB) {
      decode_rows<JMAX, RB>(wsm, Kw, G, gr, i0, wbase, xr, tot);
      emit(i0, RB, tot);
    }
    for (; i0 < nr; ++i0) {
      decode_rows<JMAX, 1>(wsm, Kw, G, gr, i0, wbase, xr, tot);
      emit(i0, 1, tot);
    }
  }
  if (S > 1 || MODE == 1) {  // block-uniform
    if (!__syncthreads_or(!arrived)) {
      if (MODE == 1 && tid < nrows) store_row(tid, sacc[tid] - xtot, resv);  // nrows <= kDecThreads
      for (int rr = tid + (MODE == 1 ? kDecThreads : 0); rr < nrows; rr += kDecThreads)
        store_row(rr, sacc[rr] - xtot, MODE == 1 ? __ldcg(a.res + row0 + rr) : 0.0f);
    }
  }
  if constexpr (MODE == 1) {
    __syncthreads();  // hb complete
    if (warp == 0) decode_epilogue(a, nrows, hb, hb + nrows);
  }
  // a warp that gave up must not let the CTA exit while the copy may still land in shared
  // memory: one more bounded wait
  if (!arrived) dec_mbar_wait(bar, 0);
}

}  // namespace tw

namespace {

struct Plan {
  int grid, rows_base, rows_rem, S, jmax;
  int xs_off, acc_off, xf_off;
  int h_off = 0;
  int cl = 1;  // streaming kernel with the fused prologue: CTAs per cluster sharing it
  size_t smem;
};

constexpr int kMaxRowsPerCta = 8192;
// Rows of at least this many weights share the fused quantisation across a cluster.  Below
// it the per-CTA prologue is shorter than the cluster's extra barrier rounds (measured on the
// 8B and 70B shapes: K = 14336 and 28672 gain 0.4 to 8 us per launch; K = 4096 loses up to
// 1.2 us, and K = 8192 up to 1.5 us without RMSNorm; with RMSNorm K = 8192 gains up to 0.7 us
// and its single-CTA prologue would spill registers).
constexpr int kClusterMinK = 12288;
constexpr int kClusterMinKRms = 8192;
// Dynamic shared memory of the one-token decode kernel: at most this much, so that the
// next launch's CTA (programmatic dependent launch) fits on the SM beside it.
constexpr size_t kDecodeSmemMax = 110 * 1024;

// Largest number of 32-bit words of x (per token) a lane keeps in registers.
int jmax_cap(int MT) { return MT == 1 ? 6 : MT == 2 ? 3 : 2; }

// Returns false when the shape is outside what the streaming kernel handles.
bool make_plan(int M, int N, int K, int num_sms, Plan& p, bool fused, bool rms = true) {
  const int MT = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  if (M > 4 || K % 64 != 0) return false;
  const int Kw = K / 16;
  p.S = 0;
  for (int S : {1, 2, 3, 4, 6, 12}) {
    const int Ws = (Kw + S - 1) / S;
    if ((Ws + 31) / 32 <= jmax_cap(MT)) {
      p.S = S;
      p.jmax = (Ws + 31) / 32;
      break;
    }
  }
  if (p.S == 0) return false;
  // One CTA per SM leaves the second slot to the next launch (programmatic dependent
  // launch).  Matrices whose rows per warp group exceed what one batch of registers
  // holds stream for long enough that two CTAs per SM (twice the loads in flight) pay
  // off more than the overlap with the next launch.
  const int G = tw::kWarps / p.S;
  const int pre = MT == 1 ? (p.jmax <= 5 ? 8 : 6) : MT == 2 ? (p.jmax <= 2 ? 8 : 6) : (p.jmax <= 1 ? 8 : 4);
  const bool long_stream = (long long)N > (long long)num_sms * G * pre;
  const int ctas = long_stream ? 2 * num_sms : num_sms;
  p.grid = N < ctas ? N : ctas;
  p.rows_base = N / p.grid;
  p.rows_rem = N % p.grid;
  const int max_rows = p.rows_base + (p.rows_rem ? 1 : 0);
  if (max_rows > kMaxRowsPerCta) return false;
  p.xs_off = 0;
  p.acc_off = MT * Kw * 16;
  p.smem = (size_t)p.acc_off + ((size_t)max_rows * MT * 4 + 15) / 16 * 16;
  // the fused prologue stages x (and the RMSNorm gain) in shared memory when it fits; one
  // token (the decode kernel) may stage more, as long as two CTAs still fit on an SM
  const size_t stage = (size_t)(MT + (rms ? 1 : 0)) * K * 4;
  p.xf_off = -1;
  // From K = kClusterMinK (kClusterMinKRms with RMSNorm) the CTAs share the quantisation in
  // clusters of 4 CTAs (the launcher falls back to 2 when too few clusters of 4 can be
  // resident).
  p.cl = fused && K >= (rms ? kClusterMinKRms : kClusterMinK) && p.grid >= 2 ? 4 : 1;
  if (fused && p.cl == 1 && stage <= 64 * 1024) {
    p.xf_off = (int)p.smem;
    p.smem += stage;
  }
  return p.smem <= 160 * 1024;
}

// Rows per warp loaded ahead: about 40 words of weights per lane.
constexpr int pre_for(int MT, int J) { return MT == 1 ? (J <= 5 ? 8 : 6) : MT == 2 ? (J <= 2 ? 8 : 6) : (J <= 1 ? 8 : 4); }

// Clusters of C CTAs of `kern` (with `smem` bytes of dynamic shared memory each) that can be
// resident at once on the current device.  The occupancy query is made once per device,
// kernel, C and shared memory.  Clusters stay within a GPC, so on a part whose GPCs do not
// hold a multiple of C CTAs fewer than grid / C fit: on 148 SMs, 74 clusters of 2 at one or
// two CTAs per SM, but 33 of 4 at one CTA per SM and 71 of 4 at two.
int max_clusters(const void* kern, size_t smem, int C) {
  struct Entry {
    int dev;
    const void* kern;
    size_t smem;
    int C, clusters;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> g(mu);
    for (const Entry& e : cache)
      if (e.dev == dev && e.kern == kern && e.smem == smem && e.C == C) return e.clusters;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(tw::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // not sticky; the caller launches without clusters
    n = 0;
  }
  std::lock_guard<std::mutex> g(mu);
  cache.push_back(Entry{dev, kern, smem, C, n});
  return n;
}

template <int MT, int JMAX, bool FUSED, bool RMS>
cudaError_t launch(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(tw::kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if constexpr (FUSED) {
    // The largest C (from the plan's down to 2) whose resident clusters cover the grid, or at
    // least 95 % of it (the grid then shrinks to those clusters, each CTA taking a few more
    // rows); with none, one CTA per cluster (x then comes from global memory: xf_off is -1).
    auto kc = tw::gemv_stream_kernel<MT, JMAX, pre_for(MT, JMAX), FUSED, RMS, true>;
    for (int C = p.cl; C >= 2; C /= 2) {
      const int grid = p.grid / C * C;
      if (grid < C) continue;
      tw::StreamArgs b = a;
      b.rows_base = a.N / grid;
      b.rows_rem = a.N % grid;
      const int max_rows = b.rows_base + (b.rows_rem ? 1 : 0);
      if (max_rows > kMaxRowsPerCta) continue;
      const size_t smem = (size_t)p.acc_off + ((size_t)max_rows * MT * 4 + 15) / 16 * 16;
      cudaError_t e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      const long long fit = (long long)max_clusters((const void*)kc, smem, C) * C;
      if (20 * fit < 19LL * p.grid) continue;
      const int g = fit < grid ? (int)fit : grid;
      b.rows_base = a.N / g;
      b.rows_rem = a.N % g;
      const int rows_g = b.rows_base + (b.rows_rem ? 1 : 0);
      const size_t smem_g = (size_t)p.acc_off + ((size_t)rows_g * MT * 4 + 15) / 16 * 16;
      if (smem_g != smem) {
        e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_g);
        if (e != cudaSuccess) return e;
      }
      cfg.gridDim = dim3((unsigned)g);
      cfg.dynamicSmemBytes = smem_g;
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = (unsigned)C;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      cfg.numAttrs = na + 1;
      return cudaLaunchKernelEx(&cfg, kc, b);
    }
  }
  auto kern = tw::gemv_stream_kernel<MT, JMAX, pre_for(MT, JMAX), FUSED, RMS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Launch plan of the one-token decode kernel: one CTA per SM (the other slot is left to the
// next launch); the CTA's packed rows, x_q and the row totals in dynamic shared memory, at
// most kDecodeSmemMax bytes, and x in at most 4 (with RMSNorm) or 8 float4s per thread.  False otherwise
// (the caller then takes gemv_stream_kernel).
bool make_decode_plan(int N, int K, int num_sms, bool rms, Plan& p, bool epi = false) {
  if (K % 64 != 0 || K / 4 > (rms ? 4 : 8) * tw::kDecThreads) return false;
  const int Kw = K / 16;
  p.S = 0;
  for (int S : {1, 2, 4, 8, 16}) {  // divisors of the decode kernel's warp count
    const int Ws = (Kw + S - 1) / S;
    if ((Ws + 31) / 32 <= 8) {
      p.S = S;
      p.jmax = (Ws + 31) / 32;
      break;
    }
  }
  if (p.S == 0) return false;
  p.grid = N < num_sms ? N : num_sms;
  p.rows_base = N / p.grid;
  p.rows_rem = N % p.grid;
  const size_t max_rows = (size_t)p.rows_base + (p.rows_rem ? 1 : 0);
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  // the last row has lanes reading up to S * 32 * jmax - Kw words past its end (against x = 0)
  const size_t slack = (size_t)(p.S * 32 * p.jmax - Kw) * 4;
  p.xs_off = (int)up(max_rows * (size_t)(K / 4) + slack, 128);
  p.acc_off = p.xs_off + (int)up((size_t)K, 16);
  p.xf_off = -1;
  p.smem = (size_t)p.acc_off + (p.S > 1 || epi ? up(max_rows * 4, 16) : 0);
  if (epi) {  // the CTA's res_out values and g_next values
    p.h_off = (int)up(p.smem, 16);
    p.smem = (size_t)p.h_off + up(2 * max_rows * 4, 16);
  }
  return p.smem <= kDecodeSmemMax;
}

template <int JMAX, int NV, bool RMS, int MODE = 0>
cudaError_t launch_decode(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  auto kern = tw::gemv_decode_kernel<JMAX, NV, RMS, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  // every kernel of a decode chain asks for the same (largest) shared-memory carveout, so
  // that the next launch's CTA can join an SM whatever the shared memory of the running one
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(tw::kDecThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// The kernel's template arguments follow from the plan: JMAX = words per lane and row, NV =
// float4s of x per thread, ceil(K / 4 / kDecThreads) rounded up to 2, 4 or 8 (2 when one warp
// spans K, S = 1; up to 4 with two K slices; 8, without RMSNorm only, with four).
// MODE 1 and 2 (residual epilogue, finished statistics) take x in at most 4 float4s per
// thread (K <= 8192).
template <bool RMS, int MODE = 0>
cudaError_t dispatch_decode(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  const int nv = (a.K / 4 + tw::kDecThreads - 1) / tw::kDecThreads;
  if (nv <= 2) {
    switch (p.jmax) {
      case 1: return launch_decode<1, 2, RMS, MODE>(a, p, stream, pdl);
      case 2: return launch_decode<2, 2, RMS, MODE>(a, p, stream, pdl);
      case 3: return launch_decode<3, 2, RMS, MODE>(a, p, stream, pdl);
      case 4: return launch_decode<4, 2, RMS, MODE>(a, p, stream, pdl);
      case 5: return launch_decode<5, 2, RMS, MODE>(a, p, stream, pdl);
      case 6: return launch_decode<6, 2, RMS, MODE>(a, p, stream, pdl);
      case 7: return launch_decode<7, 2, RMS, MODE>(a, p, stream, pdl);
      case 8: return launch_decode<8, 2, RMS, MODE>(a, p, stream, pdl);
      default: break;
    }
  } else if (nv <= 4) {
    switch (p.jmax) {
      case 5: return launch_decode<5, 4, RMS, MODE>(a, p, stream, pdl);
      case 6: return launch_decode<6, 4, RMS, MODE>(a, p, stream, pdl);
      case 7: return launch_decode<7, 4, RMS, MODE>(a, p, stream, pdl);
      case 8: return launch_decode<8, 4, RMS, MODE>(a, p, stream, pdl);
      default: break;
    }
  } else if constexpr (!RMS && MODE == 0) {
    switch (p.jmax) {
      case 5: return launch_decode<5, 8, RMS>(a, p, stream, pdl);
      case 6: return launch_decode<6, 8, RMS>(a, p, stream, pdl);
      case 7: return launch_decode<7, 8, RMS>(a, p, stream, pdl);
      case 8: return launch_decode<8, 8, RMS>(a, p, stream, pdl);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

template <int MT, bool FUSED, bool RMS>
cudaError_t dispatch_j(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  switch (p.jmax) {
    case 1: return launch<MT, 1, FUSED, RMS>(a, p, stream, pdl);
    case 2: return launch<MT, 2, FUSED, RMS>(a, p, stream, pdl);
    case 3: if constexpr (MT <= 2) return launch<MT, 3, FUSED, RMS>(a, p, stream, pdl); break;
    case 4: if constexpr (MT == 1) return launch<MT, 4, FUSED, RMS>(a, p, stream, pdl); break;
    case 5: if constexpr (MT == 1) return launch<MT, 5, FUSED, RMS>(a, p, stream, pdl); break;
    case 6: if constexpr (MT == 1) return launch<MT, 6, FUSED, RMS>(a, p, stream, pdl); break;
    default: break;
  }
  return cudaErrorInvalidValue;
}

template <bool FUSED, bool RMS>
cudaError_t dispatch(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  if (a.M <= 1) return dispatch_j<1, FUSED, RMS>(a, p, stream, pdl);
  if (a.M <= 2) return dispatch_j<2, FUSED, RMS>(a, p, stream, pdl);
  return dispatch_j<4, FUSED, RMS>(a, p, stream, pdl);
}

void fill_plan(tw::StreamArgs& a, const Plan& p) {
  a.rows_base = p.rows_base; a.rows_rem = p.rows_rem; a.S = p.S; a.xs_off = p.xs_off; a.acc_off = p.acc_off;
  a.xf_off = p.xf_off; a.h_off = p.h_off;
}

// The one-token decode kernel with the residual epilogue or with finished statistics takes
// (N, K) when its plan fits (epilogue: with the per-row buffers) and x needs at most 4
// float4s per thread.
bool decode_mode_plan(int N, int K, int num_sms, bool rms, bool epi, Plan& p) {
  if (K / 4 > 4 * tw::kDecThreads) return false;
  return make_decode_plan(N, K, num_sms, rms, p, epi);
}

}  // namespace

// 1 when the streaming kernel handles (M, N, K) (K % 64 == 0, M <= 4, shared memory fits).
int tw_stream_supported(int M, int N, int K, int num_sms) {
  Plan p;
  return make_plan(M, N, K, num_sms, p, true) ? 1 : 0;
}

cudaError_t tw_launch_gemv_stream(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                  const float* s_x, int M, int N, int K, float* y, int32_t* acc_out,
                                  cudaStream_t stream, int num_sms, bool pdl) {
  Plan p;
  if (!make_plan(M, N, K, num_sms, p, false)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x_q_in = x_q; a.s_x_in = s_x;
  a.M = M; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  fill_plan(a, p);
  return dispatch<false, false>(a, p, stream, pdl);
}

cudaError_t tw_launch_fused_gemv(const float* x, const float* g, float eps, const uint8_t* packed,
                                 const float* w_scale, int M, int N, int K, float* y, int8_t* x_q_out,
                                 float* s_x_out, int32_t* x_sum_out, int32_t* acc_out, cudaStream_t stream,
                                 int num_sms, bool pdl) {
  Plan p;
  if (!make_plan(M, N, K, num_sms, p, true, g != nullptr)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x = x; a.g = g; a.eps = eps; a.kd = tw::make_kdiv(K);
  a.inv_k = 1.0f / (float)K;
  a.M = M; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.x_q_out = x_q_out; a.s_x_out = s_x_out; a.x_sum_out = x_sum_out;
  fill_plan(a, p);
  Plan dp;
  // one token whose CTA weight block fits in shared memory: the decode kernel
  if (M == 1 && make_decode_plan(N, K, num_sms, g != nullptr, dp)) {
    fill_plan(a, dp);
    return g ? dispatch_decode<true>(a, dp, stream, pdl) : dispatch_decode<false>(a, dp, stream, pdl);
  }
  if (g) return dispatch<true, true>(a, p, stream, pdl);
  return dispatch<true, false>(a, p, stream, pdl);
}

size_t tw_epi_ws_size() { return sizeof(float4) * tw::kMaxEpiParts; }

// Partials a residual epilogue over N outputs leaves: one per CTA of its grid.
int tw_epi_parts(int N, int num_sms) { return N < num_sms ? N : num_sms; }

// 1 when the residual-epilogue decode (rms: with RMSNorm on x) takes (N, K), N = the next
// RMSNorm's length, and the finished-statistics decode takes (N2 = any, K = N).
int tw_decode_residual_supported(int N, int K, int num_sms, int rms) {
  Plan p;
  if (N % 64 != 0 || N / 4 > 4 * tw::kDecThreads || num_sms > tw::kMaxEpiParts) return 0;
  return decode_mode_plan(N, K, num_sms, rms != 0, true, p) ? 1 : 0;
}

int tw_decode_stats_supported(int N, int K, int num_sms) {
  Plan p;
  if (num_sms > tw::kMaxEpiParts) return 0;
  return decode_mode_plan(N, K, num_sms, true, false, p) ? 1 : 0;
}

cudaError_t tw_launch_quant_gemv_residual(const float* x, const float* g, float eps, const uint8_t* packed,
                                          const float* w_scale, int N, int K, const float* res, float* res_out,
                                          const float* g_next, float* y, int32_t* acc_out, void* parts,
                                          cudaStream_t stream, int num_sms, bool pdl) {
  Plan p;
  if (!decode_mode_plan(N, K, num_sms, g != nullptr, true, p)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x = x; a.g = g; a.eps = eps; a.kd = tw::make_kdiv(K);
  a.inv_k = 1.0f / (float)K;
  a.M = 1; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.res = res; a.res_out = res_out; a.g_next = g_next; a.parts_out = static_cast<float4*>(parts);
  a.kd127 = tw::make_kdiv(127);
  fill_plan(a, p);
  return g ? dispatch_decode<true, 1>(a, p, stream, pdl) : dispatch_decode<false, 1>(a, p, stream, pdl);
}

cudaError_t tw_launch_quant_gemv_stats(const float* x, const float* g, float eps, const void* parts,
                                       const uint8_t* packed, const float* w_scale, int N, int K, float* y,
                                       int8_t* x_q_out, float* s_x_out, int32_t* x_sum_out, int32_t* acc_out,
                                       cudaStream_t stream, int num_sms, bool pdl) {
  Plan p;
  if (!decode_mode_plan(N, K, num_sms, true, false, p)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x = x; a.g = g; a.eps = eps; a.kd = tw::make_kdiv(K);
  a.inv_k = 1.0f / (float)K;
  a.M = 1; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.x_q_out = x_q_out; a.s_x_out = s_x_out; a.x_sum_out = x_sum_out;
  a.parts_in = static_cast<const float4*>(parts);
  a.nparts = tw_epi_parts(K, num_sms);
  fill_plan(a, p);
  return dispatch_decode<true, 2>(a, p, stream, pdl);
}

// Reads and clears the device status word (synchronous; diagnostics only).
cudaError_t tw_read_stream_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, tw::g_stream_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(tw::g_stream_status, &zero, sizeof(int));
}
