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
//   a = max |u|;  x_q = clamp(rne(fl(fl(u * 127) / a)), -128, 127);  s_x = a;
//   x_sum = sum x_q.
// All fp32 steps use the _rn intrinsics, so no contraction or approximate
// division changes a rounding.
#include "tw_common.cuh"

namespace tw {

template <bool RMS>
__global__ void __launch_bounds__(512) act_quant_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ g, float eps, int K, KDiv kd,
                                                        int8_t* __restrict__ x_q, float* __restrict__ s_x,
                                                        int32_t* __restrict__ x_sum) {
  const int m = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int K4 = K >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)m * K);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  // exact sum of squares: per exponent bucket, m^2 (< 2^48) split into three 16-bit
  // limbs summed with native 32-bit shared atomics (K <= 65532 keeps each < 2^32)
  __shared__ uint32_t limb[RMS ? 3 : 1][RMS ? 256 : 1];
  __shared__ unsigned long long hist[RMS ? 256 : 1];
  __shared__ float red_f[32];
  __shared__ int red_i[32];
  __shared__ uint32_t red_u[32];
  __shared__ unsigned long long red_lo[32], red_hi[32];
  __shared__ float sh_inv, sh_amax;

  float inv = 1.0f;
  if (RMS) {
    // E = largest biased exponent of the row (from the largest magnitude's bits)
    uint32_t mx = 0u;
    for (int i = tid; i < K4; i += blockDim.x) {
      const float4 v = xr[i];
      mx = max(mx, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                       max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) red_u[warp] = mx;
    __syncthreads();
    mx = 0u;
    for (int w = 0; w < nwarps; ++w) mx = max(mx, red_u[w]);
    const int E = max((int)(mx >> 23), 1);
    // exact sum of squares in 128-bit fixed point (fast path)
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
        sh_inv = rms_inv_sum128(t, E, kd, eps);
      }
    } else {
      // exponents spread too far for 128 bits: exact exponent-bucket histogram
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
        if (lane == 0) sh_inv = rms_inv(r, kd, eps);
      }
    }
    __syncthreads();
    inv = sh_inv;
  }

  auto norm = [&](float v, float gg) -> float { return RMS ? __fmul_rn(__fmul_rn(v, inv), gg) : v; };

  // pass: a = max |u|
  float a = 0.0f;
  for (int i = tid; i < K4; i += blockDim.x) {
    const float4 v = xr[i];
    float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
    if (RMS) gg = g4[i];
    a = fmaxf(a, fabsf(norm(v.x, gg.x)));
    a = fmaxf(a, fabsf(norm(v.y, gg.y)));
    a = fmaxf(a, fabsf(norm(v.z, gg.z)));
    a = fmaxf(a, fabsf(norm(v.w, gg.w)));
  }
  a = warp_max(a);
  if (lane == 0) red_f[warp] = a;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nwarps ? red_f[lane] : 0.0f;
    t = warp_max(t);
    if (lane == 0) sh_amax = t;
  }
  __syncthreads();
  a = sh_amax;

  // pass: quantise, store, sum
  const float ra = a > 0.0f ? __frcp_rn(a) : 0.0f;
  int sum = 0;
  char4* out = reinterpret_cast<char4*>(x_q + (size_t)m * K);
  for (int i = tid; i < K4; i += blockDim.x) {
    const float4 v = xr[i];
    float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
    if (RMS) gg = g4[i];
    const float u[4] = {norm(v.x, gg.x), norm(v.y, gg.y), norm(v.z, gg.z), norm(v.w, gg.w)};
    int q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = 0;
      if (a > 0.0f) t = quant_div(__fmul_rn(u[j], 127.0f), a, ra);
      q[j] = max(-128, min(127, t));
      sum += q[j];
    }
    out[i] = make_char4((signed char)q[0], (signed char)q[1], (signed char)q[2], (signed char)q[3]);
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

}  // namespace tw

static int act_threads(long long K) {
  const long long k4 = K / 4;
  int t = 128;
  while (t < 512 && t < k4) t *= 2;
  return t;
}

cudaError_t tw_launch_quant_act(const float* x, long long M, long long K, int8_t* x_q, float* s_x,
                                int32_t* x_sum, cudaStream_t stream) {
  tw::act_quant_kernel<false><<<(unsigned)M, act_threads(K), 0, stream>>>(x, nullptr, 0.0f, (int)K, tw::make_kdiv((int)K), x_q, s_x,
                                                                         x_sum);
  return cudaGetLastError();
}

cudaError_t tw_launch_rmsnorm_quant_act(const float* x, const float* g, float eps, long long M, long long K,
                                        int8_t* x_q, float* s_x, int32_t* x_sum, cudaStream_t stream) {
  tw::act_quant_kernel<true><<<(unsigned)M, act_threads(K), 0, stream>>>(x, g, eps, (int)K, tw::make_kdiv((int)K), x_q, s_x, x_sum);
  return cudaGetLastError();
}
