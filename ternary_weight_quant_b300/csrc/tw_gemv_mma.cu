// tw_gemv_mma.cu -- the ternary product for a small token batch (5 .. 16 tokens) on the
// tensor cores through mma.sync (m16n8k16, f16 operands, f32 accumulation).
//
// Past a few tokens the dp4a GEMV is bound by integer issue (four dp4a per 16 weights and
// token, and integer instructions issue at half rate here), while the product is a dense
// contraction ("1-bit 大模型官方推理框架" page, FAQ 2: the weights are restored to a wider
// type for accumulation).  The int8 form of mma.sync issues very slowly on this part
// (measured: one m16n8k32 per 65 cycles per scheduler, 0.14 POP/s for the GPU), the f16 form
// at one m16n8k16 per 8 cycles (0.55 PFLOP/s), so the operands are f16.  Both are exact here:
//
//   * A (weights): the 2-bit code c = t + 1 of a weight is used as the bit pattern of an f16
//     without any conversion.  For a packed word w of 16 codes (code i in bits 2i, 2i+1),
//     w & (0x00030003 << 2s) holds codes s and s + 8 in the two f16 halves with the values
//     c 4^s 2^-24 (f16 subnormals for s <= 4; for s = 5 the code sits in the two low exponent
//     bits, and the values 0, 2^-14, 2^-13 are again c 4^5 2^-24).  Codes 6, 7, 14 and 15
//     use the word shifted right by 12.  Lane q of a quad takes masks 2q and 2q + 1 (the
//     shifted pair for q = 3): one AND per register (and one shift per word).
//   * B (activations): x_q * 4^-s for the same k positions (x_q * 1 and x_q / 4 for the
//     shifted pair), exact in f16; converted from int8 by placing x + 128 in the mantissa of
//     1024 (a byte permute) and one f16 fused multiply-add: (1024 + x + 128) sc - 1152 sc.
//   * Each product is c x 2^-24 exactly, and every partial sum is a multiple of 2^-24 below
//     1 in magnitude (|sum c x| <= 256 K < 2^24 for K <= 65532): fp32 holds it exactly, in
//     any order.  acc = 2^24 * sum - sum_k x_q  (= sum t x_q, exact int32).
// The k order inside a 16-step is therefore a permutation (kk = 2q, 2q+1, 2q+8, 2q+9 of
// lane q hold codes o0, o0 + 8, o1, o1 + 8 with o0 = 2q, o1 = 2q + 1, or 6 and 7 for q = 3);
// B is gathered in the same order, so the sum is unchanged.
//
// Work split: a CTA owns blocks of TC consecutive tiles of 16 rows; its 8 warps are G groups
// x SL K slices; group g takes tiles g, g + G, ... (up to TWM per warp), slice s a range of
// 64-k steps.  A block's rows are copied into shared memory by bulk copies, one per row into
// rows padded by 16 bytes (the eight rows a warp reads at once then fall in different
// banks), all in flight together and completing on one mbarrier (bounded wait).  Small
// matrices take one block per CTA; large ones a persistent grid with two buffers, the next
// block's copies running under the current block's computation; without room for even one
// tile each warp loads its rows' words from global memory one group of four 16-steps ahead.  A quad's four lanes share each 16-byte load.  The activations come
// straight from global memory (x_q is small and stays in L1).  Slices meet in shared memory
// through float atomics (exact: integer multiples of 2^-24 below 1).  Epilogue: per row and
// token, the accumulator minus sum x_q, dequantised as everywhere else.
#include "tw_common.cuh"

namespace tw {
namespace mma {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Args {
  const uint8_t* packed;
  const float* w_scale;
  const int8_t* x_q;
  const float* s_x;
  int M, N, K;
  int TC, G, SL;  // tiles per CTA, tile groups, K slices (G * SL = kWarps)
  int wrow;       // SMEM: byte stride of a row in shared memory (K / 4 + 16)
  float* y;
  int32_t* acc_out;
};

__device__ int g_mma_status;  // 0 or TW_ERR_TIMEOUT (sticky until read)

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Bounded wait on an mbarrier phase (2 s of wall time).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 63u) == 63u) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// NT (1 or 2) n-tiles of 8 tokens (M <= 8 NT); TWM tiles of 16 rows per warp (TC = G * TWM).
// STAGE 0: rows read from global memory one group ahead; 1: the CTA's block of TC tiles is
// staged in shared memory once; 2 (persistent): the CTA takes blocks blockIdx.x, + gridDim.x,
// ... through two shared-memory buffers, the copies of block b + 2 issued as soon as block b
// is computed, so that they run under the computation of block b + 1.
template <int NT, int TWM, int STAGE>
__global__ void __launch_bounds__(kThreads, 2) gemv_mma_kernel(Args a) {
  static_assert(NT == 1 || NT == 2, "8 or 16 tokens per kernel");
  constexpr bool SMEM = STAGE > 0;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // [SL][TC][16][8 NT] partial sums of each K slice (units of 2^-24), summed in the epilogue
  float* dsum = reinterpret_cast<float*>(smem_raw);
  unsigned char* wbase = smem_raw + (size_t)a.SL * a.TC * 16 * (8 * NT) * sizeof(float);  // [1 or 2][TC*16][wrow]
  const size_t bufsz = (size_t)a.TC * 16 * a.wrow;
  __shared__ int xsum_s[8 * NT];
  __shared__ float cs_s[8 * NT];  // per token: the dequantisation scale fl(fl(gamma s_x) / 127)
  __shared__ __align__(8) unsigned long long wbar[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = lane & 3, rq = lane >> 2;
  const int MP = 8 * NT;
  const int K = a.K, Kw = K >> 4, T4 = K >> 6;  // 16-steps (words) per row, groups of four
  const int g = warp / a.SL, sl = warp % a.SL;
  const int ntiles_all = (a.N + 15) >> 4;
  const int nblk_all = (ntiles_all + a.TC - 1) / a.TC;
  const uint32_t rb = (uint32_t)(K >> 2);

  // warp 0: the rows of block blk into buffer buf, all copies completing on wbar[buf]: one
  // bulk copy per row into padded rows, or (unpadded, wrow = K / 4) the block's contiguous
  // bytes in pieces of up to 32 KB
  auto issue = [&](int blk, int buf) {
    const int rows = min(a.TC * 16, a.N - blk * a.TC * 16);
    const uint32_t bar = smem_u32(&wbar[buf]);
    const uint32_t total = (uint32_t)rows * rb;
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(total) : "memory");
    __syncwarp();
    unsigned char* dst = wbase + (size_t)buf * bufsz;
    const unsigned char* src = a.packed + (size_t)blk * a.TC * 16 * rb;
    if ((uint32_t)a.wrow == rb) {
      for (uint32_t off = 32768u * (uint32_t)lane; off < total; off += 32768u * 32u)
        asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(dst + off)),
                     "l"(src + off), "r"(min(32768u, total - off)), "r"(bar)
                     : "memory");
    } else {
      for (int r = lane; r < rows; r += 32)
        asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(dst + (size_t)r * a.wrow)),
                     "l"(src + (size_t)r * rb), "r"(rb), "r"(bar)
                     : "memory");
    }
  };

  // programmatic dependent launch: the weights are parameters and are fetched at once; the
  // activations, their scales and the outputs belong to the previous kernel until the wait
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (SMEM && warp == 0) {
    if (lane == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&wbar[0])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&wbar[1])) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (blockIdx.x < nblk_all) issue(blockIdx.x, 0);
    if (STAGE == 2 && blockIdx.x + gridDim.x < nblk_all) issue(blockIdx.x + gridDim.x, 1);
  }
  const float gam = __ldg(a.w_scale);
  if (tid < MP) xsum_s[tid] = 0;
  __syncthreads();  // the mbarriers' initialisation and the zeroed sums, before the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the dequantisation scales are read only by the epilogue, behind the barrier that ends
  // the products: their loads need not hold anything up here
  if (tid < MP) cs_s[tid] = tid < a.M ? dequant_scale(gam, a.s_x[tid]) : 0.0f;

  // per-lane constants of the A masks and B scales (see the header)
  const uint32_t sh = q == 3 ? 12u : 0u;
  const uint32_t m0 = q == 3 ? 0x00030003u : (0x00030003u << (4 * q));
  const uint32_t m1 = q == 3 ? 0x000C000Cu : (0x000C000Cu << (4 * q));
  // f16x2 scale pairs sc = 4^-(2q), 4^-(2q+1) (1 and 1/4 for q = 3) and -1152 sc
  const uint32_t e0 = q == 3 ? 15u : (uint32_t)(15 - 4 * q), e1 = q == 3 ? 13u : (uint32_t)(13 - 4 * q);
  const uint32_t sc0 = (e0 << 10) * 0x10001u, sc1 = (e1 << 10) * 0x10001u;
  // -1152 sc = -(1.125 * 2^10) sc: sign, exponent 25 - (15 - e), mantissa 0.125
  const uint32_t nb0 = (0x8000u | ((e0 + 10u) << 10) | 0x80u) * 0x10001u;
  const uint32_t nb1 = (0x8000u | ((e1 + 10u) << 10) | 0x80u) * 0x10001u;
  // bytes of a 16-group: lanes q < 2 use words 0 and 2, lanes q >= 2 words 1 and 3
  const int xw_lo = q < 2 ? 0 : 1;
  const uint32_t xsel = (q & 1) ? 0x7362u : 0x5140u;

  // this warp's K range (in groups of four 16-steps)
  const int gs = (T4 + a.SL - 1) / a.SL;
  const int g0 = sl * gs, g1 = min(T4, g0 + gs);
  const uint32_t* W = reinterpret_cast<const uint32_t*>(a.packed);
  const uint32_t* X = reinterpret_cast<const uint32_t*>(a.x_q);
  int xs_lane[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) xs_lane[n] = 0;

  int b = 0;
  for (int blk = blockIdx.x; blk < nblk_all; blk += gridDim.x, ++b) {
    const int tile0 = blk * a.TC;
    const int buf = STAGE == 2 ? (b & 1) : 0;
    const unsigned char* wsm = wbase + (size_t)buf * bufsz;
    int rowA[TWM], rowB[TWM];  // rows rq and rq + 8 of each tile (clamped into the matrix)
#pragma unroll
    for (int i = 0; i < TWM; ++i) {
      const int tile = min(tile0 + g + i * a.G, ntiles_all - 1);
      rowA[i] = min(tile * 16 + rq, a.N - 1);
      rowB[i] = min(tile * 16 + rq + 8, a.N - 1);
      if (SMEM) {  // as rows of the staged block
        rowA[i] -= tile0 * 16;
        rowB[i] -= tile0 * 16;
      }
    }
    float acc[TWM][NT][4];
#pragma unroll
    for (int i = 0; i < TWM; ++i)
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.0f;

    uint4 wa[TWM], wb[TWM];  // words of the current group (four 16-steps) for rows A and B
    auto load_w = [&](int gi) {
#pragma unroll
      for (int i = 0; i < TWM; ++i) {
        if (SMEM) {
          wa[i] = *reinterpret_cast<const uint4*>(wsm + (size_t)rowA[i] * a.wrow + 16 * gi);
          wb[i] = *reinterpret_cast<const uint4*>(wsm + (size_t)rowB[i] * a.wrow + 16 * gi);
        } else {
          wa[i] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)rowA[i] * Kw) + gi);
          wb[i] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)rowB[i] * Kw) + gi);
        }
      }
    };
    bool ok = true;
    if (SMEM) {  // warp-uniform: a warp gives up as a whole (outputs then left unwritten)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&wbar[buf]), STAGE == 2 ? (uint32_t)((b >> 1) & 1) : 0u));
      if (!ok && lane == 0) atomicCAS(&g_mma_status, 0, (int)TW_ERR_TIMEOUT);
    }
    // the activation words of a group (four 16-steps) for this lane's quad position (plain
    // loads: x_q was written by the previous kernel, read after the dependency wait); with 8
    // tokens they are requested one group ahead, like the weight words (16 tokens: registers)
    constexpr bool kXAhead = NT == 1;
    uint32_t xlo_n[4][NT], xhi_n[4][NT];
    auto load_x = [&](int gi) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const uint32_t* xp = X + ((size_t)min(n * 8 + rq, a.M - 1) * K >> 2) + 16 * gi;
        const bool in = n * 8 + rq < a.M;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          xlo_n[s4][n] = in ? xp[4 * s4 + xw_lo] : 0u;
          xhi_n[s4][n] = in ? xp[4 * s4 + xw_lo + 2] : 0u;
        }
      }
    };
    if (ok && g0 < g1) {
      load_w(g0);
      if (kXAhead) load_x(g0);
    }
    for (int gi = ok ? g0 : g1; gi < g1; ++gi) {
      uint4 ca[TWM], cb[TWM];
#pragma unroll
      for (int i = 0; i < TWM; ++i) {
        ca[i] = wa[i];
        cb[i] = wb[i];
      }
      // the next group's words are in flight during this one; with 16 tokens the weight words
      // are requested before this group's activation words
      if (!kXAhead) {
        if (gi + 1 < g1) load_w(gi + 1);
        load_x(gi);
      }
      uint32_t xlo[4][NT], xhi[4][NT];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          xlo[s4][n] = xlo_n[s4][n];
          xhi[s4][n] = xhi_n[s4][n];
        }
      if (kXAhead && gi + 1 < g1) {
        load_w(gi + 1);
        load_x(gi + 1);
      }
      // B for token n * 8 + rq: this lane's four activations x[o0], x[o0 + 8], x[o1], x[o1 + 8]
      // of a 16-step, scaled and in f16 (tokens past M: x = 0).  Sums of x_q: first block only.
      auto make_b = [&](uint32_t lo, uint32_t hi, int n, uint32_t& b0, uint32_t& b1) {
        const uint32_t xb = __byte_perm(lo, hi, xsel);
        if (b == 0 && n * 8 + rq < a.M) xs_lane[n] = __dp4a((int)xb, 0x01010101, xs_lane[n]);
        const uint32_t u = xb ^ 0x80808080u;  // x + 128 as bytes
        b0 = hfma2_bits(__byte_perm(u, 0x6464u, 0x4140u), sc0, nb0);
        b1 = hfma2_bits(__byte_perm(u, 0x6464u, 0x4342u), sc1, nb1);
      };
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) make_b(xlo[s4][n], xhi[s4][n], n, b0[n], b1[n]);
#pragma unroll
        for (int i = 0; i < TWM; ++i) {
          const uint32_t w_a = (s4 == 0 ? ca[i].x : s4 == 1 ? ca[i].y : s4 == 2 ? ca[i].z : ca[i].w) >> sh;
          const uint32_t w_b = (s4 == 0 ? cb[i].x : s4 == 1 ? cb[i].y : s4 == 2 ? cb[i].z : cb[i].w) >> sh;
#pragma unroll
          for (int n = 0; n < NT; ++n) mma_f16(acc[i][n], w_a & m0, w_b & m0, w_a & m1, w_b & m1, b0[n], b1[n]);
        }
      }
    }

    // each slice's partial sums to its own slot: D[row][token] of tile i is (c0, c1) at row rq,
    // tokens 2q, 2q + 1 and (c2, c3) at row rq + 8
#pragma unroll
    for (int i = 0; i < TWM; ++i) {
      float* d = dsum + ((size_t)sl * a.TC + g + i * a.G) * 16 * MP;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int tk = n * 8 + 2 * q;
        *reinterpret_cast<float2*>(&d[rq * MP + tk]) = make_float2(ok ? acc[i][n][0] : 0.f, ok ? acc[i][n][1] : 0.f);
        *reinterpret_cast<float2*>(&d[(rq + 8) * MP + tk]) =
            make_float2(ok ? acc[i][n][2] : 0.f, ok ? acc[i][n][3] : 0.f);
      }
    }
    // sum of x_q per token: the slices of group 0 cover K once; a quad covers a 16-group
    if (b == 0 && g == 0) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        int v = xs_lane[n];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (q == 0 && n * 8 + rq < a.M) atomicAdd(&xsum_s[n * 8 + rq], v);
      }
    }
    if (__syncthreads_or(!ok)) {  // a bounded wait gave up: no more outputs; copies must land first
      if (SMEM) {
        mbar_wait_bounded(smem_u32(&wbar[buf]), STAGE == 2 ? (uint32_t)((b >> 1) & 1) : 0u);
        if (STAGE == 2 && blk + gridDim.x < nblk_all)  // the other buffer's block was issued too
          mbar_wait_bounded(smem_u32(&wbar[buf ^ 1]), (uint32_t)(((b + 1) >> 1) & 1));
      }
      return;
    }
    // this buffer is free again (every warp has passed the barrier above, so its reads are
    // done): its next block starts loading under the next computation
    if (STAGE == 2 && warp == 0 && blk + 2 * (int)gridDim.x < nblk_all) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(blk + 2 * gridDim.x, buf);
    }

    const size_t slot = (size_t)a.TC * 16 * MP;
    for (int i = tid; i < a.TC * 16 * MP; i += kThreads) {
      const int tk = i % MP, r = i / MP;
      const int row = tile0 * 16 + r;
      if (tk >= a.M || row >= a.N) continue;
      float d = 0.0f;  // exact: multiples of 2^-24 below 1
      for (int k = 0; k < a.SL; ++k) d += dsum[k * slot + i];
      // 2^24 times a multiple of 2^-24 below 1: an exact integer
      const int acc_i = __float2int_rn(__fmul_rn(d, 16777216.0f)) - xsum_s[tk];
      const size_t o = (size_t)tk * a.N + row;
      a.y[o] = dequant(acc_i, cs_s[tk], gam, a.s_x[tk]);
      if (a.acc_out) a.acc_out[o] = acc_i;
    }
    if (STAGE < 2) break;
    __syncthreads();  // dsum is written again by the next block
  }
}

}  // namespace mma
}  // namespace tw

namespace {

template <int NT, int TWM, int STAGE>
cudaError_t launch_mma(const tw::mma::Args& a, size_t smem, int grid, cudaStream_t stream) {
  auto kern = tw::mma::gemv_mma_kernel<NT, TWM, STAGE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(tw::mma::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int NT, int STAGE>
cudaError_t launch_mma_tw(const tw::mma::Args& a, int tw, size_t smem, int grid, cudaStream_t stream) {
  if constexpr (NT == 1) {
    if (tw == 4) return launch_mma<NT, 4, STAGE>(a, smem, grid, stream);
  }
  if constexpr (NT <= 2) {
    if (tw == 3) return launch_mma<NT, 3, STAGE>(a, smem, grid, stream);
  }
  if (tw == 2) return launch_mma<NT, 2, STAGE>(a, smem, grid, stream);
  return launch_mma<NT, 1, STAGE>(a, smem, grid, stream);
}

template <int NT>
cudaError_t launch_mma_nt(const tw::mma::Args& a, int tw, size_t smem, int grid, int stage, cudaStream_t stream) {
  if (stage == 2) return launch_mma_tw<NT, 2>(a, tw, smem, grid, stream);
  return stage == 1 ? launch_mma_tw<NT, 1>(a, tw, smem, grid, stream) : launch_mma_tw<NT, 0>(a, tw, smem, grid, stream);
}

// Shared memory a CTA may use: two CTAs per SM.
constexpr size_t kMmaSmemMax = 110 * 1024;

}  // namespace

// 1 when the tensor-core GEMV takes (M, N, K): 1 <= M <= 16, K % 64 == 0.
int tw_mma_supported(int M, int N, int K) { return (M >= 1 && M <= 16 && N >= 1 && K % 64 == 0) ? 1 : 0; }

// G groups of tiles: one while a warp can take all TC tiles (each warp forms the activation
// operand once per 16-step for all its tiles, so more tiles per warp share that work), else
// a power of two dividing TC, at most kWarps.
static void split_groups(int TC, int twmax, int& G) {
  G = 1;
  if (TC <= twmax) return;
  while (G * 2 <= tw::mma::kWarps && TC % (G * 2) == 0) G *= 2;
}

// Launch plan.  One block of TC tiles per CTA, about two CTAs per SM, staged in shared memory
// when it fits (else read from global memory); tiles per CTA split into G groups (at most 4
// or 3 tiles per warp for 8 or 16 tokens: the accumulators are registers) and SL = 8 / G
// slices of K.  When that takes more than one wave of CTAs, a persistent grid instead walks
// through the blocks with two shared-memory buffers (two CTAs per SM when both buffers fit in
// kMmaSmemMax, else one CTA with up to twice that), loading one block while computing another.
namespace {
struct MmaPlan {
  int NT, TC, G, grid, stage;
  size_t wrow;
};

MmaPlan make_mma_plan(int M, int N, int K, int num_sms) {
  const int NT = M <= 8 ? 1 : 2;  // n-tiles of 8 tokens
  const int twmax = NT == 1 ? 4 : 3;
  const int tiles = (N + 15) / 16;
  const int target = 2 * num_sms;
  const size_t wrow = (size_t)K / 4 + 16;
  const size_t dsum_tile = (size_t)tw::mma::kWarps * 16 * (8 * NT) * sizeof(float);  // up to 8 slices
  // rows + partial sums of up to 8 slices
  const size_t tile_bytes = 16 * wrow + dsum_tile;
  const int fit = (int)(kMmaSmemMax / tile_bytes);
  int stage = fit >= 1 ? 1 : 0;
  int TC = (tiles + target - 1) / target;
  if (stage && TC > fit) TC = fit;
  int G;
  split_groups(TC, twmax, G);
  while (TC / G > twmax) {  // too many tiles per warp: fewer tiles per CTA, more CTAs
    TC -= 1;
    split_groups(TC, twmax, G);
  }
  int grid = (tiles + TC - 1) / TC;
  size_t wrow_used = wrow;
  // More than one wave of CTAs: the persistent double-buffered plan, where it measured faster
  // than one block per CTA (rows of up to 4096 weights, or 16 tokens).  Two CTAs per SM
  // within kMmaSmemMax each, or one with twice that: the one that gives a warp more tiles
  // (one tile per warp repeats the activation operand's work for every 256 weights); ties:
  // two CTAs.
  if (grid > target && (K <= 4096 || NT == 2)) {
    const size_t wr = (size_t)K / 4;  // unpadded: one contiguous copy per block
    int best_tw = 0;
    for (int cps = 2; cps >= 1; --cps) {
      const size_t budget = cps == 2 ? kMmaSmemMax : 2 * kMmaSmemMax;
      int tc = (int)(budget / (2 * 16 * wr + dsum_tile));
      if (tc < 1) continue;
      if (tc > twmax) tc = twmax;  // one group: every warp takes all tiles of its K slice
      if (tc <= best_tw) continue;
      best_tw = tc;
      const int nblk = (tiles + tc - 1) / tc;
      stage = 2;
      TC = tc;
      G = 1;
      grid = nblk < cps * num_sms ? nblk : cps * num_sms;
      wrow_used = wr;
    }
  }
  MmaPlan p;
  p.NT = NT; p.TC = TC; p.G = G; p.grid = grid; p.stage = stage; p.wrow = wrow_used;
  return p;
}
}  // namespace

// 1 when the launch plan of (M, N, K) is the persistent double-buffered one.
int tw_mma_persistent(int M, int N, int K, int num_sms) {
  if (!tw_mma_supported(M, N, K)) return 0;
  return make_mma_plan(M, N, K, num_sms).stage == 2 ? 1 : 0;
}

cudaError_t tw_launch_gemv_mma(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                               int M, int N, int K, float* y, int32_t* acc_out, cudaStream_t stream,
                               int num_sms) {
  if (!tw_mma_supported(M, N, K)) return cudaErrorInvalidValue;
  const MmaPlan p = make_mma_plan(M, N, K, num_sms);
  tw::mma::Args a = {};
  a.packed = packed; a.w_scale = w_scale; a.x_q = x_q; a.s_x = s_x;
  a.M = M; a.N = N; a.K = K; a.TC = p.TC; a.G = p.G; a.SL = tw::mma::kWarps / p.G; a.wrow = (int)p.wrow;
  a.y = y; a.acc_out = acc_out;
  const size_t smem = (size_t)a.SL * p.TC * 16 * (8 * p.NT) * sizeof(float) +
                      (size_t)(p.stage == 2 ? 2 : p.stage) * p.TC * 16 * p.wrow;
  const int tw = p.TC / p.G;
  return p.NT == 1 ? launch_mma_nt<1>(a, tw, smem, p.grid, p.stage, stream)
                   : launch_mma_nt<2>(a, tw, smem, p.grid, p.stage, stream);
}

// Reads and clears the tensor-core GEMV's device status word (synchronous; diagnostics only).
cudaError_t tw_read_mma_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, tw::mma::g_mma_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(tw::mma::g_mma_status, &zero, sizeof(int));
}
