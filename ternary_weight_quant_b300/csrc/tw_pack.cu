// tw_pack.cu -- absmean ternarisation and 2-bit packing of a weight tensor.
//
// Conversion step of the bitnet.cpp CPU tutorial (m.qwbw.cn/news/64613) section 3.2:
// every weight is absmean-quantised onto {-1, 0, +1}; stored 2 bits per weight
// (section 1.1; the I2_S format of "BitNet 1 位 LLM 独立推理引擎" 正文 para 4).
//
// gamma = (float)(S / (N*K)) where S = sum |W| is accumulated EXACTLY: each |W|
// is an integer m < 2^24 times 2^(b-1-149), so a 256-bucket histogram of the
// mantissas by exponent holds the sum without error in any order; one warp then
// turns the histogram into the correctly rounded double.  The result is
// therefore the same bit pattern for every grid size.
//
// Kernel 1 (absmean_hist): grid-stride float4 loads, per-CTA shared histogram
//   (two 12-bit limbs per bucket, native 32-bit shared atomics), merged into the
//   workspace histogram with 64-bit global atomics; the last CTA to arrive
//   (completion counter, no waiting) computes gamma.
// Kernel 2 (pack): one thread per 32-bit output word (16 weights, 64 bytes of W).

#include "tw_common.cuh"

namespace tw {

struct PackWorkspace {
  unsigned long long hist[256];
  unsigned int done;
  unsigned int pad[63];
};
static_assert(sizeof(PackWorkspace) == 2304, "workspace layout");

__global__ void __launch_bounds__(512) absmean_hist_kernel(const float4* __restrict__ W4, long long n4,
                                                           PackWorkspace* ws, float* w_scale,
                                                           long long nk) {
  // m (< 2^24) split into two 12-bit limbs summed with native 32-bit shared atomics;
  // a CTA sees at most 2^20 elements (see the launcher), so each limb sum is < 2^32.
  __shared__ uint32_t hl[256], hh[256];
  __shared__ unsigned long long hs[256];
  __shared__ bool is_last;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hl[i] = hh[i] = 0u;
  __syncthreads();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldcs(W4 + i);
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t m;
      int b;
      f32_bucket(e[j], m, b);
      if (m) {
        atomicAdd(&hl[b], m & 0xfffu);
        atomicAdd(&hh[b], m >> 12);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const unsigned long long v = (unsigned long long)hl[i] + ((unsigned long long)hh[i] << 12);
    if (v) atomicAdd(&ws->hist[i], v);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(&ws->done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hs[i] = __ldcg(&ws->hist[i]);
  __syncthreads();
  if (threadIdx.x < 32) {
    const double S = warp_exact_hist_to_double(hs, 256, 1, -149);
    if (threadIdx.x == 0) *w_scale = (float)(S / (double)nk);
  }
}

__device__ __forceinline__ uint32_t ternary_code(float w, float gamma) {
  // t = clamp(rne(w / gamma), -1, 1); code = t + 1.  gamma == 0 -> t = 0.
  if (gamma == 0.0f) return 1u;
  int t = __float2int_rn(__fdiv_rn(w, gamma));
  t = max(-1, min(1, t));
  return (uint32_t)(t + 1);
}

__device__ __forceinline__ uint32_t pack4(float4 v, float gamma) {
  return ternary_code(v.x, gamma) | (ternary_code(v.y, gamma) << 2) | (ternary_code(v.z, gamma) << 4) |
         (ternary_code(v.w, gamma) << 6);
}

// One thread per output word (4 bytes = 16 weights); `nbytes` = N*K/4.  Byte i
// of the packed tensor holds W[4i .. 4i+3] (rows are contiguous in both).
__global__ void __launch_bounds__(256) pack_kernel(const float4* __restrict__ W4, long long nbytes,
                                                   const float* __restrict__ w_scale,
                                                   uint8_t* __restrict__ packed) {
  const float gamma = *w_scale;
  const long long nwords = nbytes / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  uint32_t* out = reinterpret_cast<uint32_t*>(packed);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nwords; i += stride) {
    const float4* src = W4 + 4 * i;
    const uint32_t b0 = pack4(__ldcs(src + 0), gamma);
    const uint32_t b1 = pack4(__ldcs(src + 1), gamma);
    const uint32_t b2 = pack4(__ldcs(src + 2), gamma);
    const uint32_t b3 = pack4(__ldcs(src + 3), gamma);
    out[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
  // tail bytes (nbytes % 4), handled by the first threads of block 0
  if (blockIdx.x == 0) {
    const long long i = nwords * 4 + threadIdx.x;
    if (i < nbytes) packed[i] = (uint8_t)pack4(__ldcs(W4 + i), gamma);
  }
}

// Five trits per byte (the 1.6-bit layout).  A row takes RB = 16 ceil(K / 80) bytes; byte
// i holds the weights 4i..4i+3 as base-3 digits 0..3 and the weight 4 RB + i as digit 4,
// each digit t + 1 (t = 0 past K).  One thread per 4-byte word of the output (20 weights):
// the 16 weights of digits 0..3 are four float4 loads, the 4 of digit 4 one more.
__global__ void __launch_bounds__(256) pack_t5_kernel(const float* __restrict__ W, long long N, int K, int RB,
                                                      const float* __restrict__ w_scale,
                                                      uint32_t* __restrict__ out) {
  const float gamma = *w_scale;
  const int wpr = RB / 4;
  const long long total = N * wpr;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);  // t = 0 for any gamma
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long n = i / wpr;
    const int q = (int)(i - n * wpr);
    const float* row = W + n * (long long)K;
    const int kf = 4 * RB + 4 * q;
    const float4 f = kf < K ? __ldcs(reinterpret_cast<const float4*>(row + kf)) : zero;
    const float fifth[4] = {f.x, f.y, f.z, f.w};
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int kq = 16 * q + 4 * b;
      const float4 v = kq < K ? __ldcs(reinterpret_cast<const float4*>(row + kq)) : zero;
      const uint32_t byte = ternary_code(v.x, gamma) + 3u * ternary_code(v.y, gamma) +
                            9u * ternary_code(v.z, gamma) + 27u * ternary_code(v.w, gamma) +
                            81u * ternary_code(fifth[b], gamma);
      word |= byte << (8 * b);
    }
    out[i] = word;
  }
}

}  // namespace tw

// Host launcher (called from tw_api.cu after argument checks).
// absmean: clears the workspace, then the histogram kernel writes gamma to w_scale.
static cudaError_t launch_absmean(const float* W, long long N, long long K, float* w_scale, void* workspace,
                                  cudaStream_t stream, int num_sms) {
  using namespace tw;
  PackWorkspace* ws = static_cast<PackWorkspace*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, sizeof(PackWorkspace), stream);
  if (err != cudaSuccess) return err;
  const long long n = N * K;
  const long long n4 = n / 4;
  // at least 4 CTAs per SM, and enough CTAs that none sees more than 2^20 elements
  long long blocks = (long long)num_sms * 4;
  const long long need = (n4 + 512LL * 256 - 1) / (512LL * 256);
  if (blocks < need) blocks = need;
  if (blocks > (n4 + 511) / 512) blocks = (n4 + 511) / 512;
  if (blocks < 1) blocks = 1;
  absmean_hist_kernel<<<(unsigned)blocks, 512, 0, stream>>>(reinterpret_cast<const float4*>(W), n4, ws,
                                                            w_scale, n);
  return cudaGetLastError();
}

cudaError_t tw_launch_pack(const float* W, long long N, long long K, uint8_t* packed, float* w_scale,
                           void* workspace, cudaStream_t stream, int num_sms) {
  using namespace tw;
  cudaError_t err = launch_absmean(W, N, K, w_scale, workspace, stream, num_sms);
  if (err != cudaSuccess) return err;
  const long long nbytes = N * K / 4;
  long long pblocks = (nbytes / 4 + 255) / 256;
  const long long pmax = (long long)num_sms * 8;
  if (pblocks > pmax) pblocks = pmax;
  if (pblocks < 1) pblocks = 1;
  pack_kernel<<<(unsigned)pblocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(W), nbytes, w_scale,
                                                     packed);
  return cudaGetLastError();
}

size_t tw_pack_ws_size() { return sizeof(tw::PackWorkspace); }

// The same absmean, then the five-trits-per-byte layout (RB = 16 ceil(K / 80) bytes per row).
cudaError_t tw_launch_pack_t5(const float* W, long long N, long long K, uint8_t* packed5, float* w_scale,
                              void* workspace, cudaStream_t stream, int num_sms) {
  using namespace tw;
  cudaError_t err = launch_absmean(W, N, K, w_scale, workspace, stream, num_sms);
  if (err != cudaSuccess) return err;
  const int RB = (int)(16 * ((K + 79) / 80));
  const long long words = N * (RB / 4);
  long long blocks = (words + 255) / 256;
  const long long bmax = (long long)num_sms * 8;
  if (blocks > bmax) blocks = bmax;
  if (blocks < 1) blocks = 1;
  pack_t5_kernel<<<(unsigned)blocks, 256, 0, stream>>>(W, N, (int)K, RB, w_scale,
                                                       reinterpret_cast<uint32_t*>(packed5));
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Allocation-free variant: the same two kernels with their scratch in a
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they convert weights (a
// plug-in inside a host framework that owns every device allocation, a service
// whose memory pools are fixed at start-up, a loop that forbids allocation after
// initialisation); they pass only the tensors.  The scratch is one histogram plus
// a completion counter (sizeof(PackWorkspace) = 2304 bytes); every GPU that
// loads the library keeps it until the process exits.
namespace {

static __device__ __align__(256) tw::PackWorkspace g_pack_scratch;

}  // namespace

// Device address of g_pack_scratch in the current device's current context (in
// host code the symbol names a host-side stand-in, never the device memory
// itself).  Looked up on every call rather than cached: after cudaDeviceReset, or
// with another driver context made current, the module is loaded afresh and its
// variables move, so an address kept from an earlier call could point into memory
// that now belongs to someone else.
cudaError_t tw_pack_scratch_address(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_pack_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

size_t tw_pack_scratch_bytes() { return sizeof(g_pack_scratch); }
