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

struct StreamArgs {
  const uint8_t* packed;
  const float* w_scale;
  const float* x;         // fused: fp32 activations [M][K] (NULL -> use x_q_in)
  const float* g;         // fused RMSNorm gain [K] or NULL
  float eps;
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
};

// Block-wide reductions of MT values (every thread gets the results).
template <int MT>
__device__ __forceinline__ void breduce_max_u32(uint32_t (&v)[MT], uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    v[m] = __reduce_max_sync(0xffffffffu, v[m]);
    if (lane == 0) red[warp * MT + m] = v[m];
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    uint32_t t = red[m];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) t = max(t, red[w * MT + m]);
    v[m] = t;
  }
  __syncthreads();
}
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
__device__ double row_sumsq_hist(const float4* xr, int K4, uint32_t (*limb)[256], unsigned long long* hist,
                                 double* out) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256; i += kThreads) limb[0][i] = limb[1][i] = limb[2][i] = 0u;
  __syncthreads();
  for (int i = tid; i < K4; i += kThreads) {
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
  for (int i = tid; i < 256; i += kThreads)
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

// Quantise the activations of MT tokens (after RMSNorm when RMS) into xs
// (byte-transposed 16-element groups); scales to s_scale.  CTA 0 also stores
// x_q, s_x and x_sum when asked.  When xf is not NULL the first pass copies x (and
// the gain) into shared memory and the later passes read it from there.
template <int MT, bool RMS>
__device__ __forceinline__ void fused_prologue(const StreamArgs& a, uint4* xs, float* xf, float* s_scale,
                                               uint32_t* red_u, int* red_i, unsigned long long* red_lo,
                                               unsigned long long* red_hi, uint32_t (*limb)[256],
                                               unsigned long long* hist, double* s_dbl, float* s_inv) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4, K4 = K >> 2;
  const bool staged = xf != nullptr;
  float4* xf4 = reinterpret_cast<float4*>(xf);  // [MT][K4] then the gain [K4]
  const float4* g4 = staged && RMS ? xf4 + (size_t)MT * K4 : reinterpret_cast<const float4*>(a.g);
  auto xsrc = [&](int m) -> const float4* {
    return staged ? xf4 + (size_t)m * K4 : reinterpret_cast<const float4*>(a.x + (size_t)m * K);
  };
  // first pass: from global memory (staging copy), largest magnitude per token as bits
  uint32_t mx[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    mx[m] = 0u;
    if (m < a.M) {
      const float4* xg = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
      for (int i = tid; i < K4; i += kThreads) {
        const float4 v = xg[i];
        if (staged) xf4[(size_t)m * K4 + i] = v;
        mx[m] = max(mx[m], max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                               max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
      }
    }
  }
  if (RMS && staged) {
    const float4* gg = reinterpret_cast<const float4*>(a.g);
    for (int i = tid; i < K4; i += kThreads) xf4[(size_t)MT * K4 + i] = gg[i];
  }
  breduce_max_u32<MT>(mx, red_u);  // its barriers also publish the staged copy
  float inv[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) inv[m] = 1.0f;
  if constexpr (RMS) {
    uint32_t wide[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      Sum128 sq;
      sq.lo = sq.hi = 0ull;
      bool wd = false;
      const int E = max((int)(mx[m] >> 23), 1);
      if (m < a.M) {
        const float4* xr = xsrc(m);
        for (int i = tid; i < K4; i += kThreads) {
          const float4 v = xr[i];
          sum128_add_square(sq, v.x, E, wd);
          sum128_add_square(sq, v.y, E, wd);
          sum128_add_square(sq, v.z, E, wd);
          sum128_add_square(sq, v.w, E, wd);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const Sum128 t = sum128_shfl_xor(sq, o);
        sum128_add(sq, t.lo, t.hi);
      }
      wide[m] = wd ? 1u : 0u;
      if (lane == 0) {
        red_lo[warp * MT + m] = sq.lo;
        red_hi[warp * MT + m] = sq.hi;
      }
    }
    breduce_max_u32<MT>(wide, red_u);  // its barrier also publishes red_lo / red_hi
    // warp m combines the per-warp sums of token m; its lane 0 rounds the total and
    // forms 1/sqrt(ms + eps) (double arithmetic is scarce on this part)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= a.M) continue;
      if (wide[m]) {
        const double r = row_sumsq_hist(xsrc(m), K4, limb, hist, s_dbl);
        if (tid == 0) s_inv[m] = rms_inv(r, K, a.eps);
      } else if (warp == m) {
        Sum128 t;
        t.lo = lane < kWarps ? red_lo[lane * MT + m] : 0ull;
        t.hi = lane < kWarps ? red_hi[lane * MT + m] : 0ull;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {  // kWarps <= 16
          const Sum128 u = sum128_shfl_xor(t, o);
          sum128_add(t, u.lo, u.hi);
        }
        if (lane == 0) s_inv[m] = rms_inv(sum128_to_double(t, max((int)(mx[m] >> 23), 1)), K, a.eps);
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < MT; ++m) inv[m] = s_inv[m];
  }
  auto norm = [&](float v, float gg, int m) -> float { return RMS ? __fmul_rn(__fmul_rn(v, inv[m]), gg) : v; };
  uint32_t am[MT];  // a = max |u| per token (u >= 0 compares as its bits)
  if constexpr (RMS) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      am[m] = 0u;
      if (m < a.M) {
        const float4* xr = xsrc(m);
        for (int i = tid; i < K4; i += kThreads) {
          const float4 v = xr[i];
          const float4 gg = g4[i];
          const float t = fmaxf(fmaxf(fabsf(norm(v.x, gg.x, m)), fabsf(norm(v.y, gg.y, m))),
                                fmaxf(fabsf(norm(v.z, gg.z, m)), fabsf(norm(v.w, gg.w, m))));
          am[m] = max(am[m], __float_as_uint(t));
        }
      }
    }
    breduce_max_u32<MT>(am, red_u);
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m) am[m] = mx[m];  // without RMSNorm u = x: the first pass found max |x|
  }
  // quantise: thread by thread over 4-element units u (k = 4u .. 4u+3); element k of
  // 16-element group k/16 goes to byte (k/4) % 4 of word k % 4 of that group in xs
  unsigned char* xsb = reinterpret_cast<unsigned char*>(xs);
  int qsum[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    qsum[m] = 0;
    const float amax = __uint_as_float(am[m]);
    const float ra = amax > 0.0f ? __frcp_rn(amax) : 0.0f;
    const float4* xr = xsrc(m);
    for (int u = tid; u < K4; u += kThreads) {
      uint32_t pq = 0u;
      if (m < a.M) {
        const float4 v = xr[u];
        float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
        if (RMS) gg = g4[u];
        const float uu[4] = {norm(v.x, gg.x, m), norm(v.y, gg.y, m), norm(v.z, gg.z, m), norm(v.w, gg.w, m)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int t = amax > 0.0f ? quant_div(__fmul_rn(uu[e], 127.0f), amax, ra) : 0;
          t = max(-128, min(127, t));
          qsum[m] += t;
          pq |= ((uint32_t)t & 0xffu) << (8 * e);
        }
        if (blockIdx.x == 0 && a.x_q_out) reinterpret_cast<uint32_t*>(a.x_q_out + (size_t)m * K)[u] = pq;
      }
      unsigned char* gb = xsb + (size_t)m * Kw * 16 + (u >> 2) * 16 + (u & 3);
#pragma unroll
      for (int e = 0; e < 4; ++e) gb[4 * e] = (unsigned char)(pq >> (8 * e));
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

template <int MT, int JMAX, int PRE, bool FUSED, bool RMS>
__global__ void __launch_bounds__(kThreads, 2) gemv_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4;
  const int c = blockIdx.x;
  const int nrows = a.rows_base + (c < a.rows_rem ? 1 : 0);
  const int row0 = c * a.rows_base + min(c, a.rows_rem);
  uint4* xs = reinterpret_cast<uint4*>(smem + a.xs_off);  // [MT][Kw] byte-transposed x_q
  int* sacc = reinterpret_cast<int*>(smem + a.acc_off);   // [nrows][MT] row totals
  __shared__ uint32_t red_u[kWarps * MT];
  __shared__ int red_i[kWarps * MT];
  __shared__ unsigned long long red_lo[RMS ? kWarps * MT : 1], red_hi[RMS ? kWarps * MT : 1];
  __shared__ float s_scale[MT];
  __shared__ float s_inv[MT];
  __shared__ double s_dbl;
  __shared__ uint32_t limb[RMS ? 3 : 1][256];
  __shared__ unsigned long long hist[RMS ? 256 : 1];

  pdl_launch_dependents();

  // ---------------------------------------------------------------- rows of this warp
  const int S = a.S, G = kWarps / S;
  const int sl = warp % S, gr = warp / S;
  const int Ws = (Kw + S - 1) / S;
  const int ws0 = sl * Ws, ws1 = min(Kw, ws0 + Ws);
  const int nr = nrows > gr ? (nrows - gr + G - 1) / G : 0;  // rows of this group
  const uint32_t* Wp = reinterpret_cast<const uint32_t*>(a.packed) + (size_t)row0 * Kw;
  const uint64_t pol = l2_evict_first_policy();

  uint32_t wv[PRE][JMAX];
  auto load_batch = [&](int b) {
#pragma unroll
    for (int p = 0; p < PRE; ++p) {
      const int i = b * PRE + p;
      const uint32_t* rowp = Wp + (size_t)(gr + (i < nr ? i : 0) * G) * Kw;
#pragma unroll
      for (int j = 0; j < JMAX; ++j) {
        const int wi = ws0 + lane + 32 * j;
        wv[p][j] = (i < nr && wi < ws1) ? ld_stream_u32(rowp + wi, pol) : 0x55555555u;
      }
    }
  };
  // weights (and their scale) do not depend on the previous kernel: start streaming now
  if (nr > 0) load_batch(0);
  const float gam = __ldg(a.w_scale);

  for (int i = tid; i < nrows * MT; i += kThreads) sacc[i] = 0;
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
  } else {
    float* xf = a.xf_off >= 0 ? reinterpret_cast<float*>(smem + a.xf_off) : nullptr;
    fused_prologue<MT, RMS>(a, xs, xf, s_scale, red_u, red_i, red_lo, red_hi, limb, hist, &s_dbl, s_inv);
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
  const int nb = (nr + PRE - 1) / PRE;
  for (int b = 0; b < nb; ++b) {
    if (b > 0) load_batch(b);
#pragma unroll
    for (int p = 0; p < PRE; ++p) {
      if (b * PRE + p >= nr) break;  // warp-uniform
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0;
#pragma unroll
      for (int j = 0; j < JMAX; ++j) {
        const uint32_t w = wv[p][j];
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
      const int i = b * PRE + p;
      // padding words hold code 1 (weight 0) against x = 0; lane_xsum covers exactly the
      // words this lane multiplied.  acc[m][s] is 4^s times an integer: the shifts are exact.
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int t = acc[m][0] + (acc[m][1] >> 2) + (acc[m][2] >> 4) + (acc[m][3] >> 6) - lane_xsum[m];
        const int tot = __reduce_add_sync(0xffffffffu, t);
        if (lane == 0 && i < nr) {
          const int r = gr + i * G;
          if (S == 1) sacc[r * MT + m] = tot;
          else atomicAdd(&sacc[r * MT + m], tot);
        }
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- epilogue (coalesced)
  for (int i = tid; i < a.M * nrows; i += kThreads) {
    const int m = i / nrows, r = i - m * nrows;
    const int acc = sacc[r * MT + m];
    const float sm = s_scale[m];
    const size_t o = (size_t)m * a.N + row0 + r;
    a.y[o] = dequant(acc, dequant_scale(gam, sm), gam, sm);
    if (a.acc_out) a.acc_out[o] = acc;
  }
}

}  // namespace tw

namespace {

struct Plan {
  int grid, rows_base, rows_rem, S, jmax;
  int xs_off, acc_off, xf_off;
  size_t smem;
};

constexpr int kMaxRowsPerCta = 8192;

// Largest number of 32-bit words of x (per token) a lane keeps in registers.
int jmax_cap(int MT) { return MT == 1 ? 6 : MT == 2 ? 3 : 2; }

// Returns false when the shape is outside what the streaming kernel handles.
bool make_plan(int M, int N, int K, int num_sms, Plan& p, bool fused) {
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
  // the fused prologue stages x (and the RMSNorm gain) in shared memory when it fits
  const size_t stage = (size_t)(MT + 1) * K * 4;
  p.xf_off = -1;
  if (fused && stage <= 64 * 1024) {
    p.xf_off = (int)p.smem;
    p.smem += stage;
  }
  return p.smem <= 160 * 1024;
}

// Rows per warp loaded ahead: about 40 words of weights per lane.
constexpr int pre_for(int MT, int J) { return MT == 1 ? (J <= 5 ? 8 : 6) : MT == 2 ? (J <= 2 ? 8 : 6) : (J <= 1 ? 8 : 4); }

template <int MT, int JMAX, bool FUSED, bool RMS>
cudaError_t launch(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  auto kern = tw::gemv_stream_kernel<MT, JMAX, pre_for(MT, JMAX), FUSED, RMS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(tw::kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
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
  a.xf_off = p.xf_off;
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
  if (!make_plan(M, N, K, num_sms, p, true)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x = x; a.g = g; a.eps = eps;
  a.M = M; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.x_q_out = x_q_out; a.s_x_out = s_x_out; a.x_sum_out = x_sum_out;
  fill_plan(a, p);
  if (g) return dispatch<true, true>(a, p, stream, pdl);
  return dispatch<true, false>(a, p, stream, pdl);
}

// Reads and clears the device status word (synchronous; diagnostics only).
cudaError_t tw_read_stream_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, tw::g_stream_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(tw::g_stream_status, &zero, sizeof(int));
}
