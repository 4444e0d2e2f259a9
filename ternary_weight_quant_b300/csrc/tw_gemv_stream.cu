// tw_gemv_stream.cu -- batch 1..4 ternary GEMV that streams the packed weights
// through shared memory with bulk asynchronous copies, optionally with the
// activation quantisation (and RMSNorm) fused in front.
//
// The GEMV is bound by reading the packed weights once ("1bit-systems" page,
// 性能实测: the ternary GEMV saturates the memory system; only fewer bytes make
// it faster).  Design for B300:
//   * one CTA per SM (grid <= #SMs); CTA c owns a contiguous block of rows, which
//     is a contiguous byte range of the packed tensor (rows are K/4 bytes);
//   * the block is cut into chunks of whole rows (~8 KB) that cp.async.bulk moves
//     from HBM into a ring of shared-memory stages, completion tracked by one
//     mbarrier per stage (transaction bytes); up to 8 chunks are in flight;
//   * the first chunks are issued BEFORE griddepcontrol.wait, so under
//     programmatic dependent launch the weight stream of this GEMV overlaps the
//     tail of the kernel before it (weights never depend on that kernel);
//   * the activations (fp32 x, fused quantisation; or int8 x_q) are read only
//     after the wait, quantised into shared memory, and each warp keeps the
//     words of its K slice in registers for all rows (x is reused N times);
//   * inner loop: one LDS.32 of 16 packed weights, 4 x (shift, and) to get the
//     codes c = t + 1, 4 dp4a per token; sum c*x - sum x = sum t*x exactly;
//   * warps split K into S slices (so a lane holds at most JMAX words of x) and
//     the rows of a chunk among 8/S groups; per-row sums by redux.sync, slices
//     combined in shared memory.
// Every mbarrier wait is bounded; on expiry the kernel records TW_ERR_TIMEOUT in
// a device status word, drains its own copies (bounded) and returns.
#include "tw_common.cuh"

namespace tw {

__device__ int g_stream_status;  // 0 or a tw_status recorded by a kernel (sticky until read)

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 8;
constexpr long long kSpinLimit = 1LL << 25;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
  int chunk_rows, nstages, S;
  float* y;
  int32_t* acc_out;
  int8_t* x_q_out;        // fused: written by CTA 0 when non-NULL
  float* s_x_out;
  int32_t* x_sum_out;
};

// Block-wide reductions over 256 threads (all threads get the result).
__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < kWarps ? red[lane] : 0.0f;
  return warp_max(t);
}
__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = lane < kWarps ? red[lane] : 0;
  return warp_sum(t);
}

template <int MT, int JMAX, bool FUSED, bool RMS>
__global__ void __launch_bounds__(kThreads) gemv_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, Kw = K >> 4, rowB = K >> 2;
  const int c = blockIdx.x;
  const int nrows = a.rows_base + (c < a.rows_rem ? 1 : 0);
  const int row0 = c * a.rows_base + min(c, a.rows_rem);
  const int chunk_bytes = a.chunk_rows * rowB;
  const int nchunks = (nrows + a.chunk_rows - 1) / a.chunk_rows;

  // shared memory carve-up (offsets are multiples of 16)
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                             // [kMaxStages]
  unsigned char* ring = smem + 128;                                              // [nstages][chunk_bytes]
  uint4* xs = reinterpret_cast<uint4*>(ring + (size_t)a.nstages * chunk_bytes);  // [MT][Kw] permuted
  int* part = reinterpret_cast<int*>(xs + (size_t)MT * Kw);                      // [chunk_rows][S][MT]
  __shared__ float red_f[kWarps];
  __shared__ int red_i[kWarps];
  __shared__ float s_scale[MT];
  __shared__ uint32_t limb[RMS ? 3 : 1][RMS ? 256 : 1];
  __shared__ unsigned long long hist[RMS ? 256 : 1];

  const uint64_t pol = l2_evict_first_policy();
  if (tid == 0) {
    for (int s = 0; s < a.nstages; ++s) mbar_init(&bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();

  // prefetch the first chunks (independent of any earlier kernel)
  const unsigned char* src0 = a.packed + (size_t)row0 * rowB;
  if (tid == 0) {
    for (int ch = 0; ch < nchunks && ch < a.nstages; ++ch) {
      const int r = min(a.chunk_rows, nrows - ch * a.chunk_rows);
      mbar_arrive_expect_tx(&bar[ch], (uint32_t)(r * rowB));
      bulk_g2s(ring + (size_t)ch * chunk_bytes, src0 + (size_t)ch * chunk_bytes, (uint32_t)(r * rowB), &bar[ch],
               pol);
    }
  }

  pdl_wait();  // activations and outputs may belong to the previous kernel

  // ---------------------------------------------------------------- activations -> xs
  const int G16 = K >> 4;  // 16-element groups per token
  for (int m = 0; m < MT; ++m) {
    if (m >= a.M) {
      for (int i = tid; i < G16; i += kThreads) xs[m * Kw + i] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    if (!FUSED) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x_q_in + (size_t)m * K);
      for (int i = tid; i < G16; i += kThreads) xs[m * Kw + i] = permute_group(src[i]);
      if (tid == 0) s_scale[m] = a.s_x_in[m];
      continue;
    }
    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)m * K);
    const float4* g4 = reinterpret_cast<const float4*>(a.g);
    float inv = 1.0f;
    if (RMS) {
      for (int i = tid; i < 256; i += kThreads) limb[0][i] = limb[1][i] = limb[2][i] = 0u;
      __syncthreads();
      for (int i = tid; i < (K >> 2); i += kThreads) {
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
        if (lane == 0) red_f[0] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn((float)(r / (double)K), a.eps)));
      }
      __syncthreads();
      inv = red_f[0];
      __syncthreads();
    }
    auto norm = [&](float v, float gg) -> float { return RMS ? __fmul_rn(__fmul_rn(v, inv), gg) : v; };
    float amax = 0.0f;
    for (int i = tid; i < (K >> 2); i += kThreads) {
      const float4 v = xr[i];
      float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
      if (RMS) gg = g4[i];
      amax = fmaxf(amax, fabsf(norm(v.x, gg.x)));
      amax = fmaxf(amax, fabsf(norm(v.y, gg.y)));
      amax = fmaxf(amax, fabsf(norm(v.z, gg.z)));
      amax = fmaxf(amax, fabsf(norm(v.w, gg.w)));
    }
    amax = block_max(amax, red_f);
    int qsum = 0;
    for (int i = tid; i < G16; i += kThreads) {
      uint32_t wq[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 v = xr[4 * i + q4];
        float4 gg = make_float4(1.f, 1.f, 1.f, 1.f);
        if (RMS) gg = g4[4 * i + q4];
        const float u[4] = {norm(v.x, gg.x), norm(v.y, gg.y), norm(v.z, gg.z), norm(v.w, gg.w)};
        uint32_t packedq = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int t = 0;
          if (amax > 0.0f) t = __float2int_rn(__fdiv_rn(__fmul_rn(u[j], 127.0f), amax));
          t = max(-128, min(127, t));
          qsum += t;
          packedq |= ((uint32_t)t & 0xffu) << (8 * j);
        }
        wq[q4] = packedq;
      }
      const uint4 grp = make_uint4(wq[0], wq[1], wq[2], wq[3]);
      xs[m * Kw + i] = permute_group(grp);
      if (c == 0 && a.x_q_out) reinterpret_cast<uint4*>(a.x_q_out + (size_t)m * K)[i] = grp;
    }
    if (c == 0 && a.x_sum_out) {
      qsum = block_sum(qsum, red_i);
      if (tid == 0) a.x_sum_out[m] = qsum;
    }
    if (tid == 0) {
      s_scale[m] = amax;
      if (c == 0 && a.s_x_out) a.s_x_out[m] = amax;
    }
    __syncthreads();
  }
  __syncthreads();

  // ---------------------------------------------------------------- x slice -> registers
  const int S = a.S, G = kWarps / S;
  const int sl = warp % S, grp = warp / S;
  const int Ws = (Kw + S - 1) / S;
  const int ws0 = sl * Ws, ws1 = min(Kw, ws0 + Ws);
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
  const float gam = *a.w_scale;
  float cm[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) cm[m] = dequant_scale(gam, s_scale[m]);

  // ---------------------------------------------------------------- weight chunks
  for (int ch = 0; ch < nchunks; ++ch) {
    const int stage = ch % a.nstages;
    const uint32_t parity = (uint32_t)((ch / a.nstages) & 1);
    const bool ok = mbar_wait_bounded(&bar[stage], parity);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicExch(&g_stream_status, (int)TW_ERR_TIMEOUT);
        // drain the copies this CTA still has in flight (bounded) before leaving
        for (int k2 = ch + 1; k2 < nchunks && k2 < ch + a.nstages; ++k2)
          mbar_wait_bounded(&bar[k2 % a.nstages], (uint32_t)((k2 / a.nstages) & 1));
      }
      return;
    }
    const int crow0 = ch * a.chunk_rows;
    const int crows = min(a.chunk_rows, nrows - crow0);
    const uint32_t* wbase = reinterpret_cast<const uint32_t*>(ring + (size_t)stage * chunk_bytes);
    for (int r = grp; r < crows; r += G) {
      const uint32_t* wrow = wbase + (size_t)r * Kw;
      int acc[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = 0;
#pragma unroll
      for (int j = 0; j < JMAX; ++j) {
        const int wi = ws0 + lane + 32 * j;
        if (wi < ws1) {
          const uint32_t w = wrow[wi];
          const uint32_t c0 = w & 0x03030303u, c1 = (w >> 2) & 0x03030303u;
          const uint32_t c2 = (w >> 4) & 0x03030303u, c3 = (w >> 6) & 0x03030303u;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            int s = acc[m];
            s = __dp4a((int)c0, (int)xr[j][m].x, s);
            s = __dp4a((int)c1, (int)xr[j][m].y, s);
            s = __dp4a((int)c2, (int)xr[j][m].z, s);
            s = __dp4a((int)c3, (int)xr[j][m].w, s);
            acc[m] = s;
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int tot = __reduce_add_sync(0xffffffffu, acc[m] - lane_xsum[m]);
        if (lane == m && m < a.M) {
          if (S == 1) {
            const size_t o = (size_t)m * a.N + row0 + crow0 + r;
            a.y[o] = dequant(tot, cm[m], gam, s_scale[m]);
            if (a.acc_out) a.acc_out[o] = tot;
          } else {
            part[(r * S + sl) * MT + m] = tot;
          }
        }
      }
    }
    __syncthreads();  // every warp is done with this stage (and part[] is complete)
    if (S > 1) {
      for (int i = tid; i < crows * a.M; i += kThreads) {
        const int m = i / crows, r = i - m * crows;
        int tot = 0;
        for (int s2 = 0; s2 < S; ++s2) tot += part[(r * S + s2) * MT + m];
        const size_t o = (size_t)m * a.N + row0 + crow0 + r;
        a.y[o] = dequant(tot, cm[m], gam, s_scale[m]);
        if (a.acc_out) a.acc_out[o] = tot;
      }
      __syncthreads();
    }
    if (tid == 0) {
      const int nxt = ch + a.nstages;
      if (nxt < nchunks) {
        const int r = min(a.chunk_rows, nrows - nxt * a.chunk_rows);
        mbar_arrive_expect_tx(&bar[stage], (uint32_t)(r * rowB));
        bulk_g2s(ring + (size_t)stage * chunk_bytes, src0 + (size_t)nxt * chunk_bytes, (uint32_t)(r * rowB),
                 &bar[stage], pol);
      }
    }
  }
}

}  // namespace tw

namespace {

struct Plan {
  int grid, rows_base, rows_rem, chunk_rows, nstages, S;
  size_t smem;
};

constexpr int kChunkTarget = 8 * 1024;
constexpr int kRingBudget = 64 * 1024;

int jmax_for(int MT) { return MT == 1 ? 8 : MT == 2 ? 4 : 2; }

// Returns false when the shape is outside what the streaming kernel handles.
bool make_plan(int M, int N, int K, int num_sms, Plan& p) {
  const int MT = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  if (M > 4 || K % 64 != 0) return false;
  const int Kw = K / 16, rowB = K / 4;
  const int jmax = jmax_for(MT);
  p.S = 0;
  for (int S = 1; S <= 8; S *= 2) {
    const int Ws = (Kw + S - 1) / S;
    if ((Ws + 31) / 32 <= jmax) {
      p.S = S;
      break;
    }
  }
  if (p.S == 0) return false;
  p.grid = N < num_sms ? N : num_sms;
  p.rows_base = N / p.grid;
  p.rows_rem = N % p.grid;
  const int max_rows = p.rows_base + (p.rows_rem ? 1 : 0);
  p.chunk_rows = kChunkTarget / rowB;
  if (p.chunk_rows < 1) p.chunk_rows = 1;
  if (p.chunk_rows > max_rows) p.chunk_rows = max_rows;
  const int chunk_bytes = p.chunk_rows * rowB;
  const int nchunks = (max_rows + p.chunk_rows - 1) / p.chunk_rows;
  p.nstages = kRingBudget / chunk_bytes;
  if (p.nstages < 2) p.nstages = 2;
  if (p.nstages > tw::kMaxStages) p.nstages = tw::kMaxStages;
  if (p.nstages > nchunks) p.nstages = nchunks;
  p.smem = 128 + (size_t)p.nstages * chunk_bytes + (size_t)MT * Kw * 16 + (size_t)p.chunk_rows * p.S * MT * 4;
  return p.smem <= 200 * 1024;
}

template <int MT, int JMAX, bool FUSED, bool RMS>
cudaError_t launch(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  auto kern = tw::gemv_stream_kernel<MT, JMAX, FUSED, RMS>;
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

template <bool FUSED, bool RMS>
cudaError_t dispatch(const tw::StreamArgs& a, const Plan& p, cudaStream_t stream, bool pdl) {
  if (a.M <= 1) return launch<1, 8, FUSED, RMS>(a, p, stream, pdl);
  if (a.M <= 2) return launch<2, 4, FUSED, RMS>(a, p, stream, pdl);
  return launch<4, 2, FUSED, RMS>(a, p, stream, pdl);
}

}  // namespace

// 1 when the streaming kernel handles (M, N, K) (K % 64 == 0, M <= 4, shared memory fits).
int tw_stream_supported(int M, int N, int K, int num_sms) {
  Plan p;
  return make_plan(M, N, K, num_sms, p) ? 1 : 0;
}

cudaError_t tw_launch_gemv_stream(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                  const float* s_x, int M, int N, int K, float* y, int32_t* acc_out,
                                  cudaStream_t stream, int num_sms, bool pdl) {
  Plan p;
  if (!make_plan(M, N, K, num_sms, p)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x_q_in = x_q; a.s_x_in = s_x;
  a.M = M; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.rows_base = p.rows_base; a.rows_rem = p.rows_rem; a.chunk_rows = p.chunk_rows; a.nstages = p.nstages; a.S = p.S;
  return dispatch<false, false>(a, p, stream, pdl);
}

cudaError_t tw_launch_fused_gemv(const float* x, const float* g, float eps, const uint8_t* packed,
                                 const float* w_scale, int M, int N, int K, float* y, int8_t* x_q_out,
                                 float* s_x_out, int32_t* x_sum_out, int32_t* acc_out, cudaStream_t stream,
                                 int num_sms, bool pdl) {
  Plan p;
  if (!make_plan(M, N, K, num_sms, p)) return cudaErrorInvalidValue;
  tw::StreamArgs a = {};
  a.packed = packed; a.w_scale = w_scale; a.x = x; a.g = g; a.eps = eps;
  a.M = M; a.N = N; a.K = K; a.y = y; a.acc_out = acc_out;
  a.x_q_out = x_q_out; a.s_x_out = s_x_out; a.x_sum_out = x_sum_out;
  a.rows_base = p.rows_base; a.rows_rem = p.rows_rem; a.chunk_rows = p.chunk_rows; a.nstages = p.nstages; a.S = p.S;
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
