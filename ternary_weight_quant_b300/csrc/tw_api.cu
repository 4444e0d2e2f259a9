// tw_api.cu -- the C ABI of libtw.so: argument checks, then kernel launches.
//
// This is the boundary between a host runtime and the kernels, the role the
// "1bit-systems" page gives its FFI layer (系统组件全景).  Every entry point
// checks its arguments on the host in a fixed order -- NULL pointers, shapes,
// alignment, then (with one CUDA query per pointer) that each pointer is device
// memory -- and enqueues nothing when a check fails.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/ternary_w158a8.h"

cudaError_t tw_launch_pack(const float* W, long long N, long long K, uint8_t* packed, float* w_scale,
                           void* workspace, cudaStream_t stream, int num_sms);
size_t tw_pack_ws_size();
cudaError_t tw_pack_scratch_address(void** out);
size_t tw_pack_scratch_bytes();
cudaError_t tw_launch_quant_act(const float* x, long long M, long long K, int8_t* x_q, float* s_x,
                                int32_t* x_sum, cudaStream_t stream);
cudaError_t tw_launch_rmsnorm_quant_act(const float* x, const float* g, float eps, long long M, long long K,
                                        int8_t* x_q, float* s_x, int32_t* x_sum, cudaStream_t stream);
cudaError_t tw_launch_gemv(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                           const int32_t* x_sum, int M, int N, int K, float* y, int32_t* acc_out,
                           cudaStream_t stream);
cudaError_t tw_launch_gemv_generic(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                   const float* s_x, int M, int N, int K, float* y, int32_t* acc_out,
                                   cudaStream_t stream);
int tw_stream_supported(int M, int N, int K, int num_sms);
cudaError_t tw_launch_gemv_stream(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                  const float* s_x, int M, int N, int K, float* y, int32_t* acc_out,
                                  cudaStream_t stream, int num_sms, bool pdl);
cudaError_t tw_launch_fused_gemv(const float* x, const float* g, float eps, const uint8_t* packed,
                                 const float* w_scale, int M, int N, int K, float* y, int8_t* x_q_out,
                                 float* s_x_out, int32_t* x_sum_out, int32_t* acc_out, cudaStream_t stream,
                                 int num_sms, bool pdl);
cudaError_t tw_read_stream_status(int* out);
int tw_mma_supported(int M, int N, int K);
int tw_mma_persistent(int M, int N, int K, int num_sms);
cudaError_t tw_launch_gemv_mma(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                               int M, int N, int K, float* y, int32_t* acc_out, cudaStream_t stream,
                               int num_sms);
cudaError_t tw_read_gemm_status(int* out);
cudaError_t tw_set_gemm_abort_test(int on);
cudaError_t tw_read_mma_status(int* out);
cudaError_t tw_launch_gemm(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                           int M, int N, int K, float* y, int32_t* acc_out, void* workspace, cudaStream_t stream,
                           int num_sms, int* unsupported);
size_t tw_gemm_ws_size(long long M, long long K);
size_t tw_epi_ws_size();
int tw_decode_residual_supported(int N, int K, int num_sms, int rms);
int tw_decode_stats_supported(int N, int K, int num_sms);
cudaError_t tw_launch_quant_gemv_residual(const float* x, const float* g, float eps, const uint8_t* packed,
                                          const float* w_scale, int N, int K, const float* res, float* res_out,
                                          const float* g_next, float* y, int32_t* acc_out, void* parts,
                                          cudaStream_t stream, int num_sms, bool pdl);
cudaError_t tw_launch_quant_gemv_stats(const float* x, const float* g, float eps, const void* parts,
                                       const uint8_t* packed, const float* w_scale, int N, int K, float* y,
                                       int8_t* x_q_out, float* s_x_out, int32_t* x_sum_out, int32_t* acc_out,
                                       cudaStream_t stream, int num_sms, bool pdl);
cudaError_t tw_launch_pack_t5(const float* W, long long N, long long K, uint8_t* packed5, float* w_scale,
                              void* workspace, cudaStream_t stream, int num_sms);
int tw_t5_supported(int M, int N, int K);
cudaError_t tw_launch_gemv_t5(const uint8_t* packed5, const float* w_scale, const int8_t* x_q, const float* s_x,
                              int M, int N, int K, float* y, int32_t* acc_out, cudaStream_t stream, int num_sms);

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];  // 0 = unknown, -1 = not sm_103, else SM count

// Current device must be an sm_103 part; returns its SM count or a status.
tw_status device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return TW_ERR_UNSUPPORTED;
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return TW_ERR_CUDA;
    }
    v = (major == 10 && minor == 3) ? n : -1;
    g_sms[dev].store(v, std::memory_order_relaxed);
  }
  if (v < 0) return TW_ERR_UNSUPPORTED;
  *sms = v;
  return TW_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device or managed memory only (pageable or pinned host memory is rejected).
tw_status check_device_ptr(const void* p) {
  if (!p) return TW_OK;
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_NOT_DEVICE_PTR;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return TW_ERR_NOT_DEVICE_PTR;
  return TW_OK;
}

template <typename... P>
tw_status check_device_ptrs(const P*... ps) {
  tw_status st = TW_OK;
  ((st = (st == TW_OK ? check_device_ptr(ps) : st)), ...);
  return st;
}

tw_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TW_OK : TW_ERR_CUDA; }

tw_status check_kdim(int64_t K) {
  if (K < 4 || K > TW_MAX_K || K % 4 != 0) return TW_ERR_SHAPE;
  return TW_OK;
}

tw_status check_product_args(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                             const float* s_x, int64_t M, int64_t N, int64_t K, float* y) {
  if (!packed || !w_scale || !x_q || !s_x || !y) return TW_ERR_NULL;
  if (M < 1 || N < 1 || check_kdim(K) != TW_OK) return TW_ERR_SHAPE;
  if (N > (1LL << 31) - 1 || M > (1LL << 31) - 1 || N * K >= TW_MAX_NK) return TW_ERR_SHAPE;
  if (M * N >= (1LL << 40) || M * K >= (1LL << 40)) return TW_ERR_SHAPE;
  if (!aligned(w_scale, 4) || !aligned(s_x, 4) || !aligned(y, 4)) return TW_ERR_ALIGN;
  return TW_OK;
}

}  // namespace

// Tokens from which tw_ternary_gemv takes the tensor-core (mma.sync) kernel (up to 16): below
// it the integer product of the streaming kernel is cheaper than an 8-token tensor tile.  At 3
// and 4 tokens the mma.sync kernel still wins on rows of up to 8192 weights whose plan is one
// block per CTA (measured on B300, us per call in a graph: 70B gate|up 57344 x 8192 at 4
// tokens 75 against 126, 70B q|k|v 10240 x 8192 17 against 26, 2B gate|up 13824 x 2560 9.0
// against 11.8; the streaming kernel at 4096 x 14336 13.7 against 18.7 and at the persistent
// plan of 28672 x 4096 24.1 against 28.2).
static const int64_t kMmaMinM = 5;
static const int64_t kMmaMinMShortRows = 3;

extern "C" {

TW_API const char* tw_status_string(int status) {
  switch (status) {
    case TW_OK: return "TW_OK";
    case TW_ERR_NULL: return "TW_ERR_NULL: a required pointer is NULL";
    case TW_ERR_SHAPE: return "TW_ERR_SHAPE: M, N or K out of range, K % 4 != 0, or size overflow";
    case TW_ERR_ALIGN: return "TW_ERR_ALIGN: a pointer lacks its required alignment";
    case TW_ERR_NOT_DEVICE_PTR: return "TW_ERR_NOT_DEVICE_PTR: a pointer is not device memory";
    case TW_ERR_CUDA: return "TW_ERR_CUDA: the CUDA runtime reported an error";
    case TW_ERR_UNSUPPORTED: return "TW_ERR_UNSUPPORTED: no sm_103 device or unsupported case";
    case TW_ERR_TIMEOUT: return "TW_ERR_TIMEOUT: a bounded device-side wait gave up";
    case TW_ERR_WORKSPACE: return "TW_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown tw_status";
  }
}

TW_API int tw_version(void) { return 100; }

TW_API size_t tw_pack_workspace_bytes(int64_t N, int64_t K) {
  if (N < 1 || check_kdim(K) != TW_OK || N * K >= TW_MAX_NK) return 0;
  return tw_pack_ws_size();
}

TW_API tw_status tw_pack_ternary(const float* W, int64_t N, int64_t K, uint8_t* packed, float* w_scale,
                                 void* workspace, size_t ws_bytes, tw_stream_t stream) {
  if (!W || !packed || !w_scale) return TW_ERR_NULL;
  if (N < 1 || check_kdim(K) != TW_OK || N * K >= TW_MAX_NK) return TW_ERR_SHAPE;
  if (!workspace || ws_bytes < tw_pack_ws_size()) return TW_ERR_WORKSPACE;
  if (!aligned(W, 16) || !aligned(packed, 4) || !aligned(w_scale, 4) || !aligned(workspace, 8))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(W, packed, w_scale, static_cast<const uint8_t*>(workspace));
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_pack(W, N, K, packed, w_scale, workspace, (cudaStream_t)stream, sms));
}

TW_API tw_status tw_pack_ternary_noalloc(const float* W, int64_t N, int64_t K, uint8_t* packed,
                                         float* w_scale, tw_stream_t stream) {
  if (!W || !packed || !w_scale) return TW_ERR_NULL;
  if (N < 1 || check_kdim(K) != TW_OK || N * K >= TW_MAX_NK) return TW_ERR_SHAPE;
  if (tw_pack_scratch_bytes() < tw_pack_ws_size()) return TW_ERR_WORKSPACE;
  if (!aligned(W, 16) || !aligned(packed, 4) || !aligned(w_scale, 4)) return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(W, packed, w_scale);
  if (st != TW_OK) return st;
  void* scratch = nullptr;
  if (tw_pack_scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_CUDA;
  }
  return from_cuda(tw_launch_pack(W, N, K, packed, w_scale, scratch, (cudaStream_t)stream, sms));
}

TW_API tw_status tw_quant_act(const float* x, int64_t M, int64_t K, int8_t* x_q, float* s_x, int32_t* x_sum,
                              tw_stream_t stream) {
  if (!x || !x_q || !s_x) return TW_ERR_NULL;
  if (M < 1 || M > (1LL << 20) || check_kdim(K) != TW_OK) return TW_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(x_q, 4) || !aligned(s_x, 4) || !aligned(x_sum, 4)) return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(x, x_q, s_x, x_sum);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_quant_act(x, M, K, x_q, s_x, x_sum, (cudaStream_t)stream));
}

TW_API tw_status tw_rmsnorm_quant_act(const float* x, const float* g, float eps, int64_t M, int64_t K,
                                      int8_t* x_q, float* s_x, int32_t* x_sum, tw_stream_t stream) {
  if (!x || !g || !x_q || !s_x) return TW_ERR_NULL;
  if (M < 1 || M > (1LL << 20) || check_kdim(K) != TW_OK) return TW_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(x_q, 4) || !aligned(s_x, 4) || !aligned(x_sum, 4))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(x, g, x_q, s_x, x_sum);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_rmsnorm_quant_act(x, g, eps, M, K, x_q, s_x, x_sum, (cudaStream_t)stream));
}

TW_API tw_status tw_ternary_gemv(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                 const float* s_x, const int32_t* x_sum, int64_t M, int64_t N, int64_t K,
                                 float* y, int32_t* acc_out, tw_stream_t stream) {
  tw_status st = check_product_args(packed, w_scale, x_q, s_x, M, N, K, y);
  if (st != TW_OK) return st;
  if (M > TW_GEMV_MAX_M) return TW_ERR_SHAPE;
  if (!aligned(x_sum, 4) || !aligned(acc_out, 4)) return TW_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(packed, w_scale, x_q, s_x, x_sum, y, acc_out);
  if (st != TW_OK) return st;
  const bool mma_m = M >= kMmaMinM ||
                     (M >= kMmaMinMShortRows && K <= 8192 && !tw_mma_persistent((int)M, (int)N, (int)K, sms));
  if (mma_m && aligned(packed, 16) && aligned(x_q, 16) && tw_mma_supported((int)M, (int)N, (int)K))
    return from_cuda(tw_launch_gemv_mma(packed, w_scale, x_q, s_x, (int)M, (int)N, (int)K, y, acc_out,
                                        (cudaStream_t)stream, sms));
  if (aligned(packed, 16) && aligned(x_q, 16) && tw_stream_supported((int)M, (int)N, (int)K, sms))
    return from_cuda(tw_launch_gemv_stream(packed, w_scale, x_q, s_x, (int)M, (int)N, (int)K, y, acc_out,
                                           (cudaStream_t)stream, sms, true));
  return from_cuda(tw_launch_gemv(packed, w_scale, x_q, s_x, x_sum, (int)M, (int)N, (int)K, y, acc_out,
                                  (cudaStream_t)stream));
}

TW_API tw_status tw_quant_gemv(const float* x, const float* g, float eps, const uint8_t* packed,
                               const float* w_scale, int64_t M, int64_t N, int64_t K, float* y, int8_t* x_q_out,
                               float* s_x_out, int32_t* x_sum_out, int32_t* acc_out, tw_stream_t stream) {
  if (!x || !packed || !w_scale || !y) return TW_ERR_NULL;
  if (M < 1 || M > TW_QUANT_GEMV_MAX_M || N < 1 || N > (1LL << 31) - 1 || check_kdim(K) != TW_OK ||
      K % 64 != 0 || N * K >= TW_MAX_NK)
    return TW_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(packed, 16) || !aligned(w_scale, 4) || !aligned(y, 4) ||
      !aligned(x_q_out, 16) || !aligned(s_x_out, 4) || !aligned(x_sum_out, 4) || !aligned(acc_out, 4))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  if (!tw_stream_supported((int)M, (int)N, (int)K, sms)) return TW_ERR_UNSUPPORTED;
  st = check_device_ptrs(x, g, packed, w_scale, y, x_q_out, s_x_out, x_sum_out, acc_out);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_fused_gemv(x, g, eps, packed, w_scale, (int)M, (int)N, (int)K, y, x_q_out, s_x_out,
                                        x_sum_out, acc_out, (cudaStream_t)stream, sms, true));
}

TW_API size_t tw_gemm_workspace_bytes(int64_t M, int64_t K) {
  if (M < 1 || M > (1LL << 31) - 1 || check_kdim(K) != TW_OK || M * K >= (1LL << 40)) return 0;
  return tw_gemm_ws_size(M, K);
}

TW_API tw_status tw_ternary_gemm(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                 const float* s_x, const int32_t* x_sum, int64_t M, int64_t N, int64_t K,
                                 float* y, int32_t* acc_out, void* workspace, size_t ws_bytes, tw_stream_t stream) {
  (void)x_sum;
  tw_status st = check_product_args(packed, w_scale, x_q, s_x, M, N, K, y);
  if (st != TW_OK) return st;
  if (K % 16 != 0) return TW_ERR_SHAPE;
  if (workspace && ws_bytes < tw_gemm_ws_size(M, K)) return TW_ERR_WORKSPACE;
  if (!aligned(x_q, 16) || !aligned(packed, 16) || !aligned(acc_out, 4) || !aligned(workspace, 256))
    return TW_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(packed, w_scale, x_q, s_x, y, acc_out, static_cast<const uint8_t*>(workspace));
  if (st != TW_OK) return st;
  int unsupported = 0;
  cudaError_t e = tw_launch_gemm(packed, w_scale, x_q, s_x, (int)M, (int)N, (int)K, y, acc_out, workspace,
                                 (cudaStream_t)stream, sms, &unsupported);
  if (unsupported) return TW_ERR_UNSUPPORTED;
  return from_cuda(e);
}

// Token count from which the tcgen05 GEMM takes over from the GEMV kernels (the mma.sync
// kernel from 5 to 16 tokens).  Measured on B300, microseconds per call chained in a graph, at
// 12 and 16 tokens (mma.sync against GEMM): 70B q|k|v 10240 x 8192 34.5 / 33.7 against 42.6 /
// 42.8, 70B gate|up 57344 x 8192 141 against 150, 8B down 4096 x 14336 29.4 / 37.7 against
// 43.5 / 43.7; but 70B down 8192 x 28672 (rows too long to stage) 75 / 83 against 69 and
// 2560 x 6912 16.8 / 20.5 against 16.0 / 15.9.  So from 12 tokens the GEMM takes rows longer
// than 16384 weights, and narrow matrices (N < 4096) with rows of 6912 or more, when it can
// use its workspace; 17 tokens and more always go to the GEMM.
static const int64_t kGemmCrossoverM = 17;
static const int64_t kGemmCrossoverLargeM = 12;
static const int64_t kLargeWeights = (int64_t)1 << 24;

static bool prefer_gemm(int64_t M, int64_t N, int64_t K, const void* workspace, size_t ws_bytes) {
  if (M >= kGemmCrossoverM || M > TW_GEMV_MAX_M) return true;
  return M >= kGemmCrossoverLargeM && (K > 16384 || (N < 4096 && K >= 6912)) && N * K >= kLargeWeights &&
         K % 64 == 0 && workspace != nullptr && ws_bytes >= tw_gemm_ws_size((int)M, (int)K);
}

TW_API tw_status tw_ternary_matmul(const uint8_t* packed, const float* w_scale, const int8_t* x_q,
                                   const float* s_x, const int32_t* x_sum, int64_t M, int64_t N, int64_t K,
                                   float* y, int32_t* acc_out, void* workspace, size_t ws_bytes,
                                   tw_stream_t stream) {
  tw_status st = check_product_args(packed, w_scale, x_q, s_x, M, N, K, y);
  if (st != TW_OK) return st;
  if (!prefer_gemm(M, N, K, workspace, ws_bytes))
    return tw_ternary_gemv(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  if (K % 16 == 0 && aligned(x_q, 16) && aligned(packed, 16))
    return tw_ternary_gemm(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, workspace, ws_bytes, stream);
  if (M <= TW_GEMV_MAX_M)
    return tw_ternary_gemv(packed, w_scale, x_q, s_x, x_sum, M, N, K, y, acc_out, stream);
  if (!aligned(acc_out, 4)) return TW_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(packed, w_scale, x_q, s_x, y, acc_out);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_gemv_generic(packed, w_scale, x_q, s_x, (int)M, (int)N, (int)K, y, acc_out,
                                          (cudaStream_t)stream));
}

TW_API size_t tw_t5_row_bytes(int64_t K) {
  if (check_kdim(K) != TW_OK) return 0;
  return (size_t)(16 * ((K + 79) / 80));
}

TW_API tw_status tw_pack_ternary_t5(const float* W, int64_t N, int64_t K, uint8_t* packed5, float* w_scale,
                                    void* workspace, size_t ws_bytes, tw_stream_t stream) {
  if (!W || !packed5 || !w_scale) return TW_ERR_NULL;
  if (N < 1 || check_kdim(K) != TW_OK || N * K >= TW_MAX_NK) return TW_ERR_SHAPE;
  if (!workspace || ws_bytes < tw_pack_ws_size()) return TW_ERR_WORKSPACE;
  if (!aligned(W, 16) || !aligned(packed5, 16) || !aligned(w_scale, 4) || !aligned(workspace, 8))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(W, packed5, w_scale, static_cast<const uint8_t*>(workspace));
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_pack_t5(W, N, K, packed5, w_scale, workspace, (cudaStream_t)stream, sms));
}

TW_API tw_status tw_ternary_gemv_t5(const uint8_t* packed5, const float* w_scale, const int8_t* x_q,
                                    const float* s_x, int64_t M, int64_t N, int64_t K, float* y,
                                    int32_t* acc_out, tw_stream_t stream) {
  tw_status st = check_product_args(packed5, w_scale, x_q, s_x, M, N, K, y);
  if (st != TW_OK) return st;
  if (M > 2 || !tw_t5_supported((int)M, (int)N, (int)K)) return TW_ERR_SHAPE;
  if (!aligned(packed5, 16) || !aligned(x_q, 16) || !aligned(acc_out, 4)) return TW_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != TW_OK) return st;
  st = check_device_ptrs(packed5, w_scale, x_q, s_x, y, acc_out);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_gemv_t5(packed5, w_scale, x_q, s_x, (int)M, (int)N, (int)K, y, acc_out,
                                     (cudaStream_t)stream, sms));
}

TW_API size_t tw_epilogue_workspace_bytes(void) { return tw_epi_ws_size(); }

TW_API tw_status tw_quant_gemv_residual(const float* x, const float* g, float eps, const uint8_t* packed,
                                        const float* w_scale, int64_t N, int64_t K, const float* h, float* h_out,
                                        const float* g_next, float* y, int32_t* acc_out, void* workspace,
                                        size_t ws_bytes, tw_stream_t stream) {
  if (!x || !packed || !w_scale || !h || !h_out || !g_next) return TW_ERR_NULL;
  if (N < 64 || N > 8192 || N % 64 != 0 || check_kdim(K) != TW_OK || K % 64 != 0 || K > 8192) return TW_ERR_SHAPE;
  if (!workspace || ws_bytes < tw_epi_ws_size()) return TW_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(packed, 16) || !aligned(w_scale, 4) || !aligned(h, 16) ||
      !aligned(h_out, 16) || !aligned(g_next, 4) || !aligned(y, 4) || !aligned(acc_out, 4) ||
      !aligned(workspace, 16))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  if (!tw_decode_residual_supported((int)N, (int)K, sms, g != nullptr)) return TW_ERR_UNSUPPORTED;
  st = check_device_ptrs(x, g, packed, w_scale, h, h_out, g_next, y, acc_out, static_cast<const uint8_t*>(workspace));
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_quant_gemv_residual(x, g, eps, packed, w_scale, (int)N, (int)K, h, h_out, g_next, y,
                                                 acc_out, workspace, (cudaStream_t)stream, sms, true));
}

TW_API tw_status tw_quant_gemv_stats(const float* x, const float* g, float eps, const void* workspace,
                                     const uint8_t* packed, const float* w_scale, int64_t N, int64_t K, float* y,
                                     int8_t* x_q_out, float* s_x_out, int32_t* x_sum_out, int32_t* acc_out,
                                     tw_stream_t stream) {
  if (!x || !g || !workspace || !packed || !w_scale || !y) return TW_ERR_NULL;
  if (N < 1 || N > (1LL << 31) - 1 || check_kdim(K) != TW_OK || K % 64 != 0 || K > 8192 || N * K >= TW_MAX_NK)
    return TW_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(workspace, 16) || !aligned(packed, 16) ||
      !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(x_q_out, 16) || !aligned(s_x_out, 4) ||
      !aligned(x_sum_out, 4) || !aligned(acc_out, 4))
    return TW_ERR_ALIGN;
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  if (!tw_decode_stats_supported((int)N, (int)K, sms)) return TW_ERR_UNSUPPORTED;
  st = check_device_ptrs(x, g, static_cast<const uint8_t*>(workspace), packed, w_scale, y, x_q_out, s_x_out,
                         x_sum_out, acc_out);
  if (st != TW_OK) return st;
  return from_cuda(tw_launch_quant_gemv_stats(x, g, eps, workspace, packed, w_scale, (int)N, (int)K, y, x_q_out,
                                              s_x_out, x_sum_out, acc_out, (cudaStream_t)stream, sms, true));
}

TW_API tw_status tw_debug_gemm_abort(int on) {
  int sms = 0;
  tw_status st = device_info(&sms);
  if (st != TW_OK) return st;
  if (tw_set_gemm_abort_test(on) != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_CUDA;
  }
  return TW_OK;
}

TW_API tw_status tw_device_status(int32_t* status) {
  if (!status) return TW_ERR_NULL;
  int v = 0, g = 0, m = 0;
  if (tw_read_stream_status(&v) != cudaSuccess || tw_read_gemm_status(&g) != cudaSuccess ||
      tw_read_mma_status(&m) != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_CUDA;
  }
  *status = v ? v : g ? g : m;
  return TW_OK;
}

}  // extern "C"
