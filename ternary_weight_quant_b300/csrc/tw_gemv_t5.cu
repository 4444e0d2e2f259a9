// tw_gemv_t5.cu -- the ternary GEMV over weights stored five trits per byte (1.6 bits).
//
// "BitNet 1 位 LLM 独立推理引擎：位串行 GEMM 内核与 LUT 优化工程实践" (正文 paragraph 3)
// describes TL2: several ternary weights share one small index, looked up in a table, so
// the product loads fewer weight bytes; the "1bit-systems" page (性能实测) notes that the
// bandwidth-bound GEMV only gets faster by reading fewer bytes.  Five trits fit one byte
// (3^5 = 243 <= 256): 1.6 bits per weight, 20 % fewer bytes than the 2-bit layout.
//
// Layout (written by tw_pack_ternary_t5): a row takes RB = 16 ceil(K / 80) bytes; byte i
// holds the weights 4i..4i+3 as base-3 digits 0..3 and the weight 4 RB + i as digit 4,
// each digit t + 1.  The layout is chosen for dp4a: digits 0..3 of one byte are four
// consecutive weights, one dp4a against one 32-bit word of x_q; digit 4 of four
// consecutive bytes are four consecutive weights of the tail, one more dp4a.
//
// Decode: a 256-entry table maps a byte to its five weights as int8 (digits 0..3 in a
// 32-bit word, digit 4 in a second word).  Entry v takes the 256 bytes at v * 256 and holds
// 32 copies, lane l reading the 8-byte copy l: the lanes of each half-warp always hit
// different bank pairs, whatever their bytes, and the address v * 256 + 8 l is one byte
// permute of the weight word and a register holding 8 l.  Per 4 weight bytes (20 weights) a
// lane does four such permutes, four table reads, three byte permutes to gather digit 4 and
// five dp4a per token.  On this part the integer pipe runs at half the fp32 rate and each
// table read is two shared-memory wavefronts, so the decode, not the byte count, bounds
// this kernel before HBM does.
//
// Work split: lane l of a warp covers the 16-byte chunk c = 32 s + l of every row (slice s
// of 32 chunks, 2560 weights); its x_q words stay in registers for the whole kernel.  The
// CTA has S x G warps (S slices, G warps per slice); warps of one slice take rows in turn,
// four rows per batch, the next batch's chunks requested before the current one is decoded.  Each (slice, row) total goes to shared memory; the
// CTA adds the slices of its rows and dequantises.  With programmatic dependent launch the
// table is built before griddepcontrol.wait, x_q and s_x are read after it.
#include "tw_common.cuh"

namespace tw {
namespace t5 {

constexpr int kLutCopies = 32;
constexpr int kLutBytes = 256 * kLutCopies * 8;  // 64 KB
constexpr int kMaxWarps = 16;
constexpr int kRows = 4;  // rows in flight per warp

struct Args {
  const uint4* p5;  // [N][U] 16-byte chunks
  const float* w_scale;
  const int8_t* x_q;
  const float* s_x;
  int M, N, K, RB, U, S, G;
  int rows_base, rows_rem, rows_cap;
  float* y;
  int32_t* acc_out;
};

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// lane8 = 8 * lane: byte 0 of the address, the weight byte b as byte 1, zeros above
__device__ __forceinline__ uint2 lut_read(const unsigned char* lut, uint32_t word, uint32_t lane8, uint32_t sel) {
  return *reinterpret_cast<const uint2*>(lut + __byte_perm(word, lane8, sel));
}

template <int MT>
__device__ __forceinline__ void dot_word(uint32_t word, const unsigned char* lut, uint32_t lane8,
                                         const uint4 (&xq)[MT][4], const uint4 (&xt)[MT], int q, int (&acc)[MT]) {
  const uint2 e0 = lut_read(lut, word, lane8, 0x6504u);
  const uint2 e1 = lut_read(lut, word, lane8, 0x6514u);
  const uint2 e2 = lut_read(lut, word, lane8, 0x6524u);
  const uint2 e3 = lut_read(lut, word, lane8, 0x6534u);
  // digit 4 of the four bytes: byte 0 of each .y, gathered into one word
  const uint32_t f = __byte_perm(__byte_perm(e0.y, e1.y, 0x0040u), __byte_perm(e2.y, e3.y, 0x0040u), 0x5410u);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int s = __dp4a((int)e0.x, (int)xq[m][q].x, acc[m]);
    s = __dp4a((int)e1.x, (int)xq[m][q].y, s);
    s = __dp4a((int)e2.x, (int)xq[m][q].z, s);
    s = __dp4a((int)e3.x, (int)xq[m][q].w, s);
    acc[m] = __dp4a((int)f, (int)comp(xt[m], q), s);
  }
}

template <int MT>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) gemv_t5_kernel(Args a) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint2* lut = reinterpret_cast<uint2*>(smem);           // [256][kLutCopies]
  int* part = reinterpret_cast<int*>(smem + kLutBytes);  // [S][rows_cap][MT]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_launch_dependents();

  // byte v -> digits 0..3 as int8 in .x, digit 4 as int8 in byte 0 of .y (bytes 243..255
  // never occur in a packed tensor; they decode to zeros).  Each entry is worked out by two
  // threads, each storing half of its copies.
  for (int e = tid; e < 2 * 256; e += blockDim.x) {
    const int v = e >> 1;
    uint32_t lo = 0, hi = 0;
    if (v < 243) {
      int r = v;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= (uint32_t)(uint8_t)(int8_t)(r % 3 - 1) << (8 * j);
        r /= 3;
      }
      hi = (uint32_t)(uint8_t)(int8_t)(r - 1);
    }
    const uint2 val = make_uint2(lo, hi);
    uint2* dst = lut + v * kLutCopies + (e & 1) * (kLutCopies / 2);
#pragma unroll
    for (int c2 = 0; c2 < kLutCopies / 2; ++c2) dst[c2] = val;
  }

  const int c = blockIdx.x;
  const int nrows = a.rows_base + (c < a.rows_rem ? 1 : 0);
  const int row0 = c * a.rows_base + min(c, a.rows_rem);
  const int s = warp % a.S, g = warp / a.S;
  const int chunk = 32 * s + lane;
  const bool active = chunk < a.U;
  const int K = a.K;
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);

  // the packed weights are parameters: the first rows' chunks are fetched before the wait
  const uint4* base = a.p5 + (size_t)row0 * a.U + chunk;
  uint4 w[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int rr = g + r * a.G;
    w[r] = (active && rr < nrows) ? ld_stream_v4(base + (size_t)rr * a.U) : z4;
  }

  pdl_wait();

  // x_q of this lane's weights: digits 0..3 of its 16 bytes are x_q[64 chunk .. +63],
  // digit 4 is x_q[4 RB + 16 chunk .. +15]; zero past K (K % 16 == 0)
  uint4 xq[MT][4], xt[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int8_t* xr = a.x_q + (size_t)m * K;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k0 = 64 * chunk + 16 * q;
      xq[m][q] = (active && m < a.M && k0 < K) ? *reinterpret_cast<const uint4*>(xr + k0) : z4;
    }
    const int kt = 4 * a.RB + 16 * chunk;
    xt[m] = (active && m < a.M && kt < K) ? *reinterpret_cast<const uint4*>(xr + kt) : z4;
  }
  __syncthreads();  // the table is complete

  const unsigned char* lutb = smem;
  const uint32_t lane8 = 8u * (uint32_t)lane;
  for (int i = g; i < nrows; i += kRows * a.G) {
    // the next rows' chunks are requested before this batch is decoded
    uint4 nx[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int rr = i + (kRows + r) * a.G;
      nx[r] = (active && rr < nrows) ? ld_stream_v4(base + (size_t)rr * a.U) : z4;
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int rr = i + r * a.G;
      if (rr >= nrows) break;  // warp-uniform
      int acc[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = 0;
      dot_word<MT>(w[r].x, lutb, lane8, xq, xt, 0, acc);
      dot_word<MT>(w[r].y, lutb, lane8, xq, xt, 1, acc);
      dot_word<MT>(w[r].z, lutb, lane8, xq, xt, 2, acc);
      dot_word<MT>(w[r].w, lutb, lane8, xq, xt, 3, acc);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int tot = __reduce_add_sync(0xffffffffu, acc[m]);
        if (lane == 0) part[((size_t)s * a.rows_cap + rr) * MT + m] = tot;
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) w[r] = nx[r];
  }
  __syncthreads();

  const float gam = *a.w_scale;
  for (int e = tid; e < nrows * a.M; e += blockDim.x) {
    const int rr = e / a.M, m = e - rr * a.M;
    int acc = 0;
    for (int s2 = 0; s2 < a.S; ++s2) acc += part[((size_t)s2 * a.rows_cap + rr) * MT + m];
    const float sx = a.s_x[m];
    const size_t o = (size_t)m * a.N + row0 + rr;
    a.y[o] = dequant(acc, dequant_scale(gam, sx), gam, sx);
    if (a.acc_out) a.acc_out[o] = acc;
  }
}

}  // namespace t5
}  // namespace tw

// Cases the kernel takes: 1 or 2 tokens, K % 16 == 0, and at most 16 slices of 2560
// weights (K <= 40960).
int tw_t5_supported(int M, int N, int K) {
  if (M < 1 || M > 2 || N < 1 || K < 16 || K % 16 != 0) return 0;
  const int RB = 16 * ((K + 79) / 80);
  const int S = (RB / 16 + 31) / 32;
  return S <= tw::t5::kMaxWarps;
}

cudaError_t tw_launch_gemv_t5(const uint8_t* packed5, const float* w_scale, const int8_t* x_q, const float* s_x,
                              int M, int N, int K, float* y, int32_t* acc_out, cudaStream_t stream, int num_sms) {
  using namespace tw::t5;
  Args a{};
  a.p5 = reinterpret_cast<const uint4*>(packed5);
  a.w_scale = w_scale;
  a.x_q = x_q;
  a.s_x = s_x;
  a.M = M;
  a.N = N;
  a.K = K;
  a.RB = 16 * ((K + 79) / 80);
  a.U = a.RB / 16;
  a.S = (a.U + 31) / 32;
  a.G = kMaxWarps / a.S;
  a.y = y;
  a.acc_out = acc_out;
  const int MT = M == 1 ? 1 : 2;
  // one CTA per SM (its table is 64 KB); a CTA keeps at most 1024 rows so the per-row
  // totals stay small
  long long grid = (long long)num_sms;
  if (grid > N) grid = N;
  const long long need = ((long long)N + 1023) / 1024;
  if (grid < need) grid = need;
  a.rows_base = (int)(N / grid);
  a.rows_rem = (int)(N % grid);
  a.rows_cap = a.rows_base + (a.rows_rem ? 1 : 0);
  const size_t smem = (size_t)kLutBytes + (size_t)a.S * a.rows_cap * MT * sizeof(int);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)(32 * a.S * a.G));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (MT == 1) {
    cudaError_t e = cudaFuncSetAttribute(gemv_t5_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, gemv_t5_kernel<1>, a);
  }
  cudaError_t e = cudaFuncSetAttribute(gemv_t5_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, gemv_t5_kernel<2>, a);
}
