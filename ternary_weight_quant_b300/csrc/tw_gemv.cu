// tw_gemv.cu -- ternary x int8 matrix-vector product for 1..16 tokens (dp4a).
//
// The product needs no multiplier: each ternary weight selects +x, -x or nothing
// (bitnet.cpp CPU tutorial, m.qwbw.cn/news/64613, section 1.1), and the kernel is
// bound by streaming the packed weights ("1bit-systems" page, 性能实测).  On the
// GPU the sign-and-add is done four weights at a time with dp4a on the 2-bit
// codes c = t + 1 in {0, 1, 2}:
//     acc = sum_k c[k] * x_q[k] - sum_k x_q[k]  (= sum_k t[k] * x_q[k], exact int32),
// so unpacking a 32-bit word of 16 weights costs one shift and one AND per four
// weights.  (w >> 2s) & 0x03030303 presents weights 4j + s (j = 0..3) of the
// word's 16-weight group, so the activations are staged in shared memory with
// each 16-byte group byte-transposed to the same order (permute_group).
//
// Work split: a CTA owns `rows_per_cta` consecutive output rows; each warp takes
// 4 rows at a time with its lanes striding over the 32-bit words of K (coalesced
// 128-byte loads per row, no imbalance between lanes beyond one word); U words
// per lane per row are loaded before any is used, so 4*U loads are in flight per
// lane.  Partial sums are reduced with redux.sync and kept per row in shared
// memory across K chunks (a chunk is the part of x_q that fits in shared memory
// for all tokens).  Epilogue: y = (float)acc * fl(fl(gamma * s_x) / 127) (dequant()).
#include "tw_common.cuh"

namespace tw {

template <int MT, int U>
__global__ void __launch_bounds__(256) gemv_dp4a_kernel(const uint32_t* __restrict__ Wp,
                                                        const float* __restrict__ w_scale,
                                                        const int8_t* __restrict__ x_q,
                                                        const float* __restrict__ s_x,
                                                        const int32_t* __restrict__ x_sum, int M, int N,
                                                        int K, int rows_per_cta, int chunk_words,
                                                        float* __restrict__ y, int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);                     // [MT][chunk_words]
  int* part = reinterpret_cast<int*>(xs + (size_t)MT * chunk_words);  // [rows_per_cta][MT]
  __shared__ int xsum_s[MT];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int Kw = K >> 4;
  const int row0 = blockIdx.x * rows_per_cta;
  const int rows = min(rows_per_cta, N - row0);
  const bool need_sum = (x_sum == nullptr);
  const uint64_t pol = l2_evict_first_policy();

  for (int i = tid; i < rows_per_cta * MT; i += blockDim.x) part[i] = 0;
  if (tid < MT) xsum_s[tid] = 0;

  for (int w0 = 0; w0 < Kw; w0 += chunk_words) {
    const int cw = min(chunk_words, Kw - w0);
    __syncthreads();
    // stage x_q[:, 16*w0 .. 16*(w0+cw)) permuted; tokens >= M are zero
    for (int i = tid; i < MT * cw; i += blockDim.x) {
      const int m = i / cw, j = i - m * cw;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < M) v = *reinterpret_cast<const uint4*>(x_q + (size_t)m * K + 16 * (size_t)(w0 + j));
      xs[m * chunk_words + j] = permute_group(v);
      if (need_sum && m < M) atomicAdd(&xsum_s[m], byte_sum16(v));
    }
    __syncthreads();

    for (int rb = warp * 4; rb < rows; rb += 4 * nwarps) {
      const uint32_t* wr[4];
      bool rv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        rv[r] = rb + r < rows;
        wr[r] = Wp + (size_t)(row0 + (rv[r] ? rb + r : rb)) * Kw + w0;
      }
      int acc[4][MT];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0;

      for (int j0 = lane; j0 < cw; j0 += 32 * U) {
        uint32_t wv[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + 32 * u;
#pragma unroll
          for (int r = 0; r < 4; ++r) wv[u][r] = (j < cw && rv[r]) ? ld_stream_u32(wr[r] + j, pol) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + 32 * u;
          if (j < cw) {
            uint32_t c[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              c[r][0] = wv[u][r] & 0x03030303u;
              c[r][1] = (wv[u][r] >> 2) & 0x03030303u;
              c[r][2] = (wv[u][r] >> 4) & 0x03030303u;
              c[r][3] = (wv[u][r] >> 6) & 0x03030303u;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint4 xv = xs[m * chunk_words + j];
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                int a = acc[r][m];
                a = __dp4a((int)c[r][0], (int)xv.x, a);
                a = __dp4a((int)c[r][1], (int)xv.y, a);
                a = __dp4a((int)c[r][2], (int)xv.z, a);
                a = __dp4a((int)c[r][3], (int)xv.w, a);
                acc[r][m] = a;
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int s = __reduce_add_sync(0xffffffffu, acc[r][m]);
          if (lane == ((r * MT + m) & 31) && rv[r]) part[(rb + r) * MT + m] += s;
        }
    }
  }
  __syncthreads();

  const float gam = *w_scale;
  for (int i = tid; i < M * rows; i += blockDim.x) {
    const int m = i / rows, r = i - m * rows;
    const int xsm = need_sum ? xsum_s[m] : x_sum[m];
    const int a = part[r * MT + m] - xsm;
    const float sm = s_x[m];
    y[(size_t)m * N + row0 + r] = dequant(a, dequant_scale(gam, sm), gam, sm);
    if (acc_out) acc_out[(size_t)m * N + row0 + r] = a;
  }
}

// Any K % 4 == 0, any alignment, any M: one warp per output row, byte loads.
__global__ void __launch_bounds__(256) gemv_generic_kernel(const uint8_t* __restrict__ packed,
                                                           const float* __restrict__ w_scale,
                                                           const int8_t* __restrict__ x_q,
                                                           const float* __restrict__ s_x, int M, int N,
                                                           int K, float* __restrict__ y,
                                                           int32_t* __restrict__ acc_out) {
  const long long wg = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wg >= N) return;
  const int n = (int)wg;
  const int Kb = K >> 2;
  const float gam = *w_scale;
  for (int m = 0; m < M; ++m) {
    int acc = 0;
    for (int k = lane; k < K; k += 32) {
      const uint32_t code = ((uint32_t)packed[(size_t)n * Kb + (k >> 2)] >> (2 * (k & 3))) & 3u;
      acc += ((int)code - 1) * (int)x_q[(size_t)m * K + k];
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      const float sm = s_x[m];
      y[(size_t)m * N + n] = dequant(acc, dequant_scale(gam, sm), gam, sm);
      if (acc_out) acc_out[(size_t)m * N + n] = acc;
    }
  }
}

template <int MT, int U>
static cudaError_t launch_dp4a(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                               const float* s_x, const int32_t* x_sum, int M, int N, int K, float* y,
                               int32_t* acc_out, cudaStream_t stream) {
  const int Kw = K / 16;
  const int rows_per_cta = 32;
  int chunk_words = (96 * 1024) / (16 * MT);
  if (chunk_words > Kw) chunk_words = Kw;
  const size_t smem = (size_t)MT * chunk_words * 16 + (size_t)rows_per_cta * MT * 4;
  auto kern = gemv_dp4a_kernel<MT, U>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int grid = (N + rows_per_cta - 1) / rows_per_cta;
  kern<<<grid, 256, smem, stream>>>(reinterpret_cast<const uint32_t*>(packed), w_scale, x_q, s_x, x_sum, M,
                                    N, K, rows_per_cta, chunk_words, y, acc_out);
  return cudaGetLastError();
}

}  // namespace tw

// M in [1, 16].  Fast path when K % 16 == 0 and the pointers are aligned.
cudaError_t tw_launch_gemv(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                           const int32_t* x_sum, int M, int N, int K, float* y, int32_t* acc_out,
                           cudaStream_t stream) {
  using namespace tw;
  const bool fast = (K % 16 == 0) && ((uintptr_t)packed % 4 == 0) && ((uintptr_t)x_q % 16 == 0);
  if (!fast) {
    const long long threads = (long long)N * 32;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    gemv_generic_kernel<<<grid, 256, 0, stream>>>(packed, w_scale, x_q, s_x, M, N, K, y, acc_out);
    return cudaGetLastError();
  }
  if (M == 1) return launch_dp4a<1, 8>(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  if (M == 2) return launch_dp4a<2, 8>(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  if (M <= 4) return launch_dp4a<4, 4>(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  if (M <= 8) return launch_dp4a<8, 2>(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  return launch_dp4a<16, 2>(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
}

// Exact generic path for any M (used when K % 16 != 0).
cudaError_t tw_launch_gemv_generic(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                   const float* s_x, int M, int N, int K, float* y, int32_t* acc_out,
                                   cudaStream_t stream) {
  const long long threads = (long long)N * 32;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  tw::gemv_generic_kernel<<<grid, 256, 0, stream>>>(packed, w_scale, x_q, s_x, M, N, K, y, acc_out);
  return cudaGetLastError();
}
