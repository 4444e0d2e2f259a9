// tw_act.cu -- per-token int8 activation quantisation, optionally after RMSNorm.
//
// Activations are quantised to 8 bit ("BitNet-rs" page, 技术实现细节); the RMSNorm
// kernel that precedes the ternary GEMV is named on the "1bit-systems" page
// (技术架构).  Per token m (one CTA each):
//   [RMSNorm] r = exact sum of x^2 (128-bit fixed point relative to the row's
//             largest exponent; rows with a wider exponent spread use a histogram
//             of 48-bit squared mantissas per exponent), rounded once to double,
//             ms = (float)(r / K) (the double division emulated with integers),
//             inv = 1 / sqrt(ms + eps) (IEEE fp32 sqrt and divide),
//             u = fl(fl(x * inv) * g);
//             ms is first decided from a float-float sum of squares when its error
//             bound leaves the rounding determined; the exact path above otherwise;
//   a = max |u|;  x_q = clamp(rne(fl(fl(u * 127) / a)), -128, 127);  s_x = a;
//   x_sum = sum x_q.
// All fp32 steps use the _rn intrinsics, so no contraction changes a rounding; the
// approximate steps (the float-float mean square, the approximate reciprocal of the
// quantisation) are used only where their error bound leaves the result decided, and
// the exact operation is taken otherwise.
#include "tw_common.cuh"

namespace tw {

// Exact RMSNorm scale of row xr by the whole block (rare path: the float-float mean
// square could not be decided).  The row's largest exponent E comes from mx (its
// largest magnitude's bits); 128-bit fixed point relative to E, or the exponent-bucket
// histogram when the exponents spread further.
__device__ __noinline__ float act_rms_inv_exact(const float4* xr, int K4, uint32_t mx, KDiv kd, float eps,
                                                uint32_t (*limb)[256], unsigned long long* hist,
                                                unsigned long long* red_lo, unsigned long long* red_hi,
                                                float* sh_inv) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int E = max((int)(mx >> 23), 1);
  Sum128 sq;
  sq.lo = sq.hi = 0ull;
  bool wide = false;
  for (int i = tid; i < K4; i += blockDim.x) {
    const float4 v = xr[i];
    sum128_add_square(sq, v.x, E, wide);
    sum128_add_square(sq, v.y, E, wide);
    sum128_add_square(sq, v.z, E, wide);
    sum128_add_square(sq, v.w, E, wide);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Sum128 t = sum128_shfl_xor(sq, o);
    sum128_add(sq, t.lo, t.hi);
  }
  const int any_wide = __syncthreads_or(wide ? 1 : 0);
  if (lane == 0) {
    red_lo[warp] = sq.lo;
    red_hi[warp] = sq.hi;
  }
  __syncthreads();
  if (!any_wide) {
    if (tid == 0) {
      Sum128 t;
      t.lo = t.hi = 0ull;
      for (int w = 0; w < nwarps; ++w) sum128_add(t, red_lo[w], red_hi[w]);
      *sh_inv = rms_inv_sum128(t, E, kd, eps);
    }
  } else {
    for (int i = tid; i < 256; i += blockDim.x) limb[0][i] = limb[1][i] = limb[2][i] = 0u;
    __syncthreads();
    for (int i = tid; i < K4; i += blockDim.x) {
      const float4 v = xr[i];
      const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t mm;
        int b;
        f32_bucket(e[j], mm, b);
        if (mm) {
          const unsigned long long q = (unsigned long long)mm * mm;
          atomicAdd(&limb[0][b], (uint32_t)(q & 0xffffu));
          atomicAdd(&limb[1][b], (uint32_t)((q >> 16) & 0xffffu));
          atomicAdd(&limb[2][b], (uint32_t)(q >> 32));
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < 256; i += blockDim.x)
      hist[i] = (unsigned long long)limb[0][i] + ((unsigned long long)limb[1][i] << 16) +
                ((unsigned long long)limb[2][i] << 32);
    __syncthreads();
    if (warp == 0) {
      const double r = warp_exact_hist_to_double(hist, 256, 2, -298);
      if (lane == 0) *sh_inv = rms_inv(r, kd, eps);
    }
  }
  __syncthreads();
  const float inv = *sh_inv;
  __syncthreads();
  return inv;
}

// One CTA per token.  First pass: max |x| and (RMSNorm) the float-float sum of squares;
// every warp then combines the per-warp values itself and decides the mean square when
// the float-float accuracy suffices (the exact path otherwise); second pass (RMSNorm):
// a = max |u|; last pass: quantise (conversion-free rounding, the IEEE divide only for a
// unit with a quotient near a half-integer), store, sum.
template <bool RMS>
__global__ void __launch_bounds__(512) act_quant_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ g, float eps, int K, KDiv kd,
                                                        float inv_k, int8_t* __restrict__ x_q,
                                                        float* __restrict__ s_x, int32_t* __restrict__ x_sum) {
  const int m = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int K4 = K >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)m * K);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  __shared__ uint32_t limb[RMS ? 3 : 1][RMS ? 256 : 1];
  __shared__ unsigned long long hist[RMS ? 256 : 1];
  __shared__ int red_i[32];
  __shared__ uint32_t red_u[32], red_a[32];
  __shared__ float2 red_ff[32];
  __shared__ unsigned long long red_lo[32], red_hi[32];
  __shared__ float sh_inv;

  // programmatic dependent launch: the next kernel may start its own preparation now; x may
  // come from the previous kernel, so it is read only after that kernel has finished
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // first pass
  uint32_t mx = 0u;
  FF s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f}, s2 = {0.0f, 0.0f}, s3 = {0.0f, 0.0f};
#pragma unroll 2
  for (int i = tid; i < K4; i += blockDim.x) {
    const float4 v = xr[i];
    mx = max(mx, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                     max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
    if (RMS) {
      ff_add_square(s0, v.x);
      ff_add_square(s1, v.y);
      ff_add_square(s2, v.z);
      ff_add_square(s3, v.w);
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
    red_u[warp] = mx;
    if (RMS) red_ff[warp] = make_float2(s0.hi, s0.lo);
  }
  __syncthreads();  // (1)
  mx = __reduce_max_sync(0xffffffffu, lane < nwarps ? red_u[lane] : 0u);

  float inv = 1.0f;
  uint32_t am = mx;  // without RMSNorm a = max |x|
  if constexpr (RMS) {
    FF t;
    t.hi = t.lo = 0.0f;
    if (lane < nwarps) {
      const float2 f = red_ff[lane];
      t.hi = f.x;
      t.lo = f.y;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // nwarps <= 16
      FF u;
      u.hi = __shfl_xor_sync(0xffffffffu, t.hi, o);
      u.lo = __shfl_xor_sync(0xffffffffu, t.lo, o);
      ff_add(t, u);
    }
    // lane 0's sum to every lane: the decision is the same in every thread of the block
    t.hi = __shfl_sync(0xffffffffu, t.hi, 0);
    t.lo = __shfl_sync(0xffffffffu, t.lo, 0);
    float ms = 0.0f;
    if (ff_mean_f32(t, K, inv_k, ms)) {
      inv = inv_rms_f32(ms, eps);
    } else {  // block-uniform
      inv = act_rms_inv_exact(xr, K4, mx, kd, eps, limb, hist, red_lo, red_hi, &sh_inv);
    }
    // second pass: a = max |u|
    am = 0u;
#pragma unroll 2
    for (int i = tid; i < K4; i += blockDim.x) {
      const float4 v = xr[i];
      const float4 gg = g4[i];
      const float4 u = make_float4(__fmul_rn(__fmul_rn(v.x, inv), gg.x), __fmul_rn(__fmul_rn(v.y, inv), gg.y),
                                   __fmul_rn(__fmul_rn(v.z, inv), gg.z), __fmul_rn(__fmul_rn(v.w, inv), gg.w));
      am = max(am, __float_as_uint(fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w)))));
    }
    am = __reduce_max_sync(0xffffffffu, am);
    if (lane == 0) red_a[warp] = am;
    __syncthreads();  // (2)
    am = __reduce_max_sync(0xffffffffu, lane < nwarps ? red_a[lane] : 0u);
  }

  // last pass: quantise, store, sum.  d = fl(p ra) with ra within one ulp of 1 / a
  // (rcp.approx) is within |p/a| 2^-22 < 3.1e-5 of p / a (|p/a| <= 127) and fl32(p/a)
  // within 2^-18 of it: at least 5e-5 from a half-integer, rint(d) is the rounding of
  // fl32(p / a); units with an element nearer (or a non-finite d: ra is NaN when a lies
  // outside [2^-120, 2^120]) are redone with the IEEE divide.
  const float a = __uint_as_float(am);
  float ra = a == 0.0f ? 0.0f : __int_as_float(0x7fffffff);
  if (a >= 0x1p-120f && a <= 0x1p120f) asm("rcp.approx.f32 %0, %1;" : "=f"(ra) : "f"(a));
  int sum = 0;
  uint32_t* out = reinterpret_cast<uint32_t*>(x_q + (size_t)m * K);
  for (int base = warp * 32; base < K4; base += blockDim.x) {  // warp-uniform trip count
    const int i = base + lane;
    float uu[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t pq = 0u;
    bool near = false;
    if (i < K4) {
      const float4 v = xr[i];
      float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
      if (RMS) gg = g4[i];
      uu[0] = RMS ? __fmul_rn(__fmul_rn(v.x, inv), gg.x) : v.x;
      uu[1] = RMS ? __fmul_rn(__fmul_rn(v.y, inv), gg.y) : v.y;
      uu[2] = RMS ? __fmul_rn(__fmul_rn(v.z, inv), gg.z) : v.z;
      uu[3] = RMS ? __fmul_rn(__fmul_rn(v.w, inv), gg.w) : v.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float d = __fmul_rn(__fmul_rn(uu[j], 127.0f), ra);
        const float sb = __fadd_rn(d, 12582912.0f);  // d + 1.5 2^23: rounds d to an integer
        near |= !(fabsf(__fsub_rn(d, __fsub_rn(sb, 12582912.0f))) < 0.49995f);
        const int t = (int)(__float_as_uint(sb) & 0x7fffffu) - 0x400000;
        pq |= ((uint32_t)max(-128, min(127, t)) & 0xffu) << (8 * j);
      }
    }
    if (__any_sync(0xffffffffu, near) && near) {  // rare
      pq = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = a > 0.0f ? __float2int_rn(__fdiv_rn(__fmul_rn(uu[j], 127.0f), a)) : 0;
        pq |= ((uint32_t)max(-128, min(127, t)) & 0xffu) << (8 * j);
      }
    }
    if (i < K4) {
      out[i] = pq;
      sum += (int)(int8_t)(pq & 0xffu) + (int)(int8_t)((pq >> 8) & 0xffu) + (int)(int8_t)((pq >> 16) & 0xffu) +
             (int)(int8_t)(pq >> 24);
    }
  }
  sum = warp_sum(sum);
  if (lane == 0) red_i[warp] = sum;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nwarps ? red_i[lane] : 0;
    t = warp_sum(t);
    if (lane == 0) {
      s_x[m] = a;
      if (x_sum) x_sum[m] = t;
    }
  }
}

// ---------------------------------------------------------------------------
// The same quantisation with each token shared by a thread-block cluster of C CTAs (grid C x M,
// clusters along x): rank r takes the float4 units [r gw, (r + 1) gw) of its token, gw =
// ceil(K / 4 / C), so that a long row is read and quantised by C CTAs instead of one.  Each
// rank pushes its chunk's largest |x| (with RMSNorm also its float-float sum of squares, and
// later its largest |u|) into every peer's shared memory between cluster barriers; every rank
// combines the C values in rank order, so all take the same decisions (the exact mean-square
// path, when taken, runs over the whole row in every CTA of the cluster).  The chunk's x_q go
// to global memory and its sum of x_q to rank 0, which writes s_x and x_sum.  The results are
// those of one CTA per token: the maximum does not depend on the order, and a decided
// float-float mean square is the exact one whatever the summation order.
constexpr int kActClusterMax = 8;
constexpr int kActClusterThreads = 256;

template <bool RMS>
__global__ void __launch_bounds__(kActClusterThreads) act_quant_cluster_kernel(
    const float* __restrict__ x, const float* __restrict__ g, float eps, int K, KDiv kd, float inv_k,
    int8_t* __restrict__ x_q, float* __restrict__ s_x, int32_t* __restrict__ x_sum) {
  constexpr int kNW = kActClusterThreads / 32;
  const int m = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K4 = K >> 2;
  const uint32_t rank = cl_rank(), C = cl_size();
  const int gw = (K4 + (int)C - 1) / (int)C;
  const int u0 = min(K4, (int)rank * gw), u1 = min(K4, u0 + gw);
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)m * K);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  __shared__ uint32_t c_mx[kActClusterMax], c_am[kActClusterMax];  // [source rank]
  __shared__ float2 c_ff[kActClusterMax];
  __shared__ int c_qs[kActClusterMax];
  __shared__ uint32_t red_u[kNW], red_a[kNW];
  __shared__ float2 red_ff[kNW];
  __shared__ int red_i[kNW];
  __shared__ uint32_t limb[RMS ? 3 : 1][RMS ? 256 : 1];
  __shared__ unsigned long long hist[RMS ? 256 : 1];
  __shared__ unsigned long long red_lo[32], red_hi[32];
  __shared__ float sh_inv;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  cl_arrive_relaxed();  // (0), waited for before the first remote store
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel

  // (1) the chunk's largest |x| and (RMSNorm) float-float sum of squares, one accumulator per
  // vector component
  uint32_t mx = 0u;
  FF s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f}, s2 = {0.0f, 0.0f}, s3 = {0.0f, 0.0f};
  for (int u = u0 + tid; u < u1; u += kActClusterThreads) {
    const float4 v = xr[u];
    mx = max(mx, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                     max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
    if (RMS) {
      ff_add_square(s0, v.x);
      ff_add_square(s1, v.y);
      ff_add_square(s2, v.z);
      ff_add_square(s3, v.w);
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
    red_u[warp] = mx;
    if (RMS) red_ff[warp] = make_float2(s0.hi, s0.lo);
  }
  __syncthreads();
  cl_wait();  // (0): every CTA of the cluster runs
  if (tid < (int)C) {  // the CTA's totals, warps in order, to rank tid
    uint32_t bm = 0u;
    FF t = {0.0f, 0.0f};
    for (int w = 0; w < kNW; ++w) {
      bm = max(bm, red_u[w]);
      if (RMS) ff_add(t, FF{red_ff[w].x, red_ff[w].y});
    }
    *peer(&c_mx[rank], (uint32_t)tid) = bm;
    if (RMS) *peer(&c_ff[rank], (uint32_t)tid) = make_float2(t.hi, t.lo);
  }
  cl_arrive();
  cl_wait();  // (1)
  mx = 0u;
  FF tot = {0.0f, 0.0f};
  for (uint32_t r = 0; r < C; ++r) {
    mx = max(mx, c_mx[r]);
    if (RMS) ff_add(tot, FF{c_ff[r].x, c_ff[r].y});
  }

  float inv = 1.0f;
  uint32_t am = mx;  // without RMSNorm a = max |x|
  if constexpr (RMS) {
    float ms = 0.0f;
    if (ff_mean_f32(tot, K, inv_k, ms)) {
      inv = inv_rms_f32(ms, eps);
    } else {  // cluster-uniform
      inv = act_rms_inv_exact(xr, K4, mx, kd, eps, limb, hist, red_lo, red_hi, &sh_inv);
    }
    // (2) the chunk's largest |u|
    uint32_t t = 0u;
    for (int u = u0 + tid; u < u1; u += kActClusterThreads) {
      const float4 v = xr[u];
      const float4 gg = g4[u];
      const float4 w = make_float4(__fmul_rn(__fmul_rn(v.x, inv), gg.x), __fmul_rn(__fmul_rn(v.y, inv), gg.y),
                                   __fmul_rn(__fmul_rn(v.z, inv), gg.z), __fmul_rn(__fmul_rn(v.w, inv), gg.w));
      t = max(t, __float_as_uint(fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w)))));
    }
    t = __reduce_max_sync(0xffffffffu, t);
    if (lane == 0) red_a[warp] = t;
    __syncthreads();
    if (tid < (int)C) {
      uint32_t bm = 0u;
      for (int w = 0; w < kNW; ++w) bm = max(bm, red_a[w]);
      *peer(&c_am[rank], (uint32_t)tid) = bm;
    }
    cl_arrive();
    cl_wait();  // (2)
    am = 0u;
    for (uint32_t r = 0; r < C; ++r) am = max(am, c_am[r]);
  }

  // (3) quantise the chunk: the conversion-free rounding of act_quant_kernel, with the same
  // IEEE-divide redo near a half-integer or for a non-finite quotient
  const float a = __uint_as_float(am);
  float ra = a == 0.0f ? 0.0f : __int_as_float(0x7fffffff);
  if (a >= 0x1p-120f && a <= 0x1p120f) asm("rcp.approx.f32 %0, %1;" : "=f"(ra) : "f"(a));
  int sum = 0;
  uint32_t* out = reinterpret_cast<uint32_t*>(x_q + (size_t)m * K);
  for (int base = u0 + warp * 32; base < u1; base += kActClusterThreads) {  // warp-uniform trip count
    const int i = base + lane;
    float uu[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t pq = 0u;
    bool near = false;
    if (i < u1) {
      const float4 v = xr[i];
      float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
      if (RMS) gg = g4[i];
      uu[0] = RMS ? __fmul_rn(__fmul_rn(v.x, inv), gg.x) : v.x;
      uu[1] = RMS ? __fmul_rn(__fmul_rn(v.y, inv), gg.y) : v.y;
      uu[2] = RMS ? __fmul_rn(__fmul_rn(v.z, inv), gg.z) : v.z;
      uu[3] = RMS ? __fmul_rn(__fmul_rn(v.w, inv), gg.w) : v.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float d = __fmul_rn(__fmul_rn(uu[j], 127.0f), ra);
        const float sb = __fadd_rn(d, 12582912.0f);  // d + 1.5 2^23: rounds d to an integer
        near |= !(fabsf(__fsub_rn(d, __fsub_rn(sb, 12582912.0f))) < 0.49995f);
        const int q = (int)(__float_as_uint(sb) & 0x7fffffu) - 0x400000;
        pq |= ((uint32_t)max(-128, min(127, q)) & 0xffu) << (8 * j);
      }
    }
    if (__any_sync(0xffffffffu, near) && near) {  // rare
      pq = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = a > 0.0f ? __float2int_rn(__fdiv_rn(__fmul_rn(uu[j], 127.0f), a)) : 0;
        pq |= ((uint32_t)max(-128, min(127, q)) & 0xffu) << (8 * j);
      }
    }
    if (i < u1) {
      out[i] = pq;
      sum += (int)(int8_t)(pq & 0xffu) + (int)(int8_t)((pq >> 8) & 0xffu) + (int)(int8_t)((pq >> 16) & 0xffu) +
             (int)(int8_t)(pq >> 24);
    }
  }
  sum = warp_sum(sum);
  if (lane == 0) red_i[warp] = sum;
  __syncthreads();
  if (tid == 0) {
    int t = 0;
    for (int w = 0; w < kNW; ++w) t += red_i[w];
    *peer(&c_qs[rank], 0u) = t;
  }
  cl_arrive();
  cl_wait();  // (3): every chunk sum is in rank 0's shared memory
  if (rank == 0 && tid == 0) {
    s_x[m] = a;
    if (x_sum) {
      int t = 0;
      for (uint32_t r = 0; r < C; ++r) t += c_qs[r];
      x_sum[m] = t;
    }
  }
}

}  // namespace tw

static int act_threads(long long K) {
  const long long k4 = K / 4;
  int t = 128;
  while (t < 512 && t < k4) t *= 2;
  return t;
}

// CTAs per token: one below K = 6144, for one token, or above 16 tokens (the tokens alone then
// spread over the SMs), else a cluster of 2 (K < 8192), 4 (K < 16384) or 8.  Measured in the
// benchmark's layer chains against one CTA per token: 2B at 8 tokens 48.4 -> 45.1 us per
// layer, 8B at 16 tokens 121.3 -> 117.7, 70B at 4 tokens 155.3 -> 149.7, 70B at 16 tokens
// 288.3 -> 282.7; at K = 4096 the cluster lost (8B at 16 tokens 121.3 -> 122.9), at 64 tokens
// it gained nothing, and at one token (the 2B step with separate quantisation, behind the
// one-token decode kernel) it lost 1.2 us per layer.
static int act_cluster(long long M, long long K) {
  if (M < 2 || M > 16 || K < 6144) return 1;
  return K < 8192 ? 2 : K < 16384 ? 4 : 8;
}

// Launched with programmatic dependent launch (the kernel waits before reading x).
template <bool RMS>
static cudaError_t launch_act(const float* x, const float* g, float eps, long long M, long long K, int8_t* x_q,
                              float* s_x, int32_t* x_sum, cudaStream_t stream) {
  const int C = act_cluster(M, K);
  if (C > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)M);
    cfg.blockDim = dim3(tw::kActClusterThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tw::act_quant_cluster_kernel<RMS>, x, g, eps, (int)K, tw::make_kdiv((int)K),
                              1.0f / (float)K, x_q, s_x, x_sum);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M);
  cfg.blockDim = dim3((unsigned)act_threads(K));
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tw::act_quant_kernel<RMS>, x, g, eps, (int)K, tw::make_kdiv((int)K),
                            1.0f / (float)K, x_q, s_x, x_sum);
}

cudaError_t tw_launch_quant_act(const float* x, long long M, long long K, int8_t* x_q, float* s_x,
                                int32_t* x_sum, cudaStream_t stream) {
  return launch_act<false>(x, nullptr, 0.0f, M, K, x_q, s_x, x_sum, stream);
}

cudaError_t tw_launch_rmsnorm_quant_act(const float* x, const float* g, float eps, long long M, long long K,
                                        int8_t* x_q, float* s_x, int32_t* x_sum, cudaStream_t stream) {
  return launch_act<true>(x, g, eps, M, K, x_q, s_x, x_sum, stream);
}
