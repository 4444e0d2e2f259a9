// tw_gemm.cu -- ternary x int8 product for larger token batches on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// The product is a sign check and an add per weight (bitnet.cpp CPU tutorial,
// m.qwbw.cn/news/64613, section 1.1); for many tokens it is a dense contraction,
// so ternary weights are widened for the accumulation ("1-bit 大模型官方推理框架"
// page, FAQ 2) and fed to the tensor cores:
//   * weights {-1, 0, +1} and int8 activations are exact in bf16, and every partial
//     sum of the fp32 accumulation is an integer of magnitude <= 128*K < 2^24, so
//     the bf16 MMA with fp32 accumulation (kind::f16) yields the exact int32 dot
//     product in any summation order;
//   * the tile is "swapped": the MMA's M side (128 lanes of tensor memory) is 128
//     weight rows and its N side is up to 256 tokens, so batches from 16 tokens up
//     fill the tensor core without padding the weight side;
//   * four producer warps read the 2-bit packed weights and the int8 activations
//     from global memory, widen them to bf16 in registers (the weights with two
//     byte-permutes per four codes) and store them into shared memory in the
//     128-byte-swizzled K-major layout the MMA reads; a fifth warp allocates
//     tensor memory and issues tcgen05.mma from one thread; stages are handed over
//     with mbarriers (producers -> MMA: thread arrivals; MMA -> producers:
//     tcgen05.commit);
//   * within each group of 16 k the widened weights are stored in the order
//     0,4,1,5,2,6,3,7,8,12,9,13,10,14,11,15 (what the byte permutes produce) and the
//     activations are stored in the same order, so the dot product is unchanged;
//   * K may be split across a cluster of CTAs (thread-block cluster along K); each
//     CTA leaves its partial accumulators in its shared memory and the CTAs of the
//     cluster sum them through distributed shared memory, each finishing a slice of
//     the tokens -- no global scratch;
//   * epilogue: tcgen05.ld of the accumulators, exact conversion to int32, then
//     y = acc * fl(fl(gamma * s_x) / 127) (the same roundings as the GEMV, dequant()).
// Every mbarrier wait is bounded (2 s); a CTA that gives up records TW_ERR_TIMEOUT in a
// device status word, waits (bounded) for the MMAs it issued, frees its tensor
// memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "tw_common.cuh"

namespace tw {
namespace gemm {

__device__ int g_gemm_status;  // 0 or TW_ERR_TIMEOUT (sticky until read)
// Diagnostic switch (tw_debug_gemm_abort): when set, every GEMM launch starts with its abort
// flag raised, so it takes the path of a bounded wait that gave up before it issues any
// copy or product.
__device__ int g_gemm_abort_test;

constexpr int BM = 128;            // weight rows per CTA (MMA M)
constexpr int BK = 64;             // k per stage: one 128-byte swizzle row of bf16
constexpr int kProducers = 128;    // threads of warps 0-3
constexpr int kThreads = 160;      // + warp 4 (TMEM allocation, MMA issue)
constexpr int kMaxStages = 8;
constexpr int kMaxCluster = 8;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int kScaleOff = 256;                // per-token scales: this far into the control block
constexpr int kCtrlBytes = kScaleOff + 2 * 256 * 4;
constexpr int kMaxBUnits = 256 * 4 / kProducers;  // 16-byte activation units per producer thread

struct Args {
  const uint8_t* packed;
  const float* w_scale;
  const int8_t* x_q;
  const float* s_x;
  int M, N, K;
  int BN;          // tokens per CTA tile (multiple of 16, <= 256)
  int nstages;
  int ksplit;      // CTAs of a cluster along K (1 = no split)
  int kstages_per_split;
  uint32_t ctrl_off;  // byte offset of the barriers after the stage / partials area
  uint32_t tmem_cols;
  float* y;
  int32_t* acc_out;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait (kTimeoutNs of wall time); with abort_flag it also gives up as soon as
// another role of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag = nullptr) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (abort_flag && *abort_flag) return false;
      const uint64_t t = global_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kTimeoutNs) return false;
    }
  }
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                     // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// 16 packed codes (one 32-bit word, k = 0..15) -> 16 bf16 in the order
// 0,4,1,5,2,6,3,7 | 8,12,9,13,10,14,11,15.  Selector byte b of s is c*0x11 + 0x40:
// nibble c picks the low bf16 byte from T0, nibble c + 4 the high byte from T1.
__device__ __forceinline__ void widen_codes(uint32_t w, uint4& lo, uint4& hi) {
  const uint32_t T0 = 0x00800080u;  // low bytes of bf16(-1), bf16(0), bf16(+1)
  const uint32_t T1 = 0x003F00BFu;  // high bytes
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = ((w >> (2 * j)) & 0x03030303u) * 0x11u + 0x40404040u;
    o[j] = __byte_perm(T0, T1, s);
    o[4 + j] = __byte_perm(T0, T1, s >> 16);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ uint32_t bf16x2_s8(uint32_t w, int i) {
  const float a = (float)(int)(int8_t)(w >> (8 * i));
  const float b = (float)(int)(int8_t)(w >> (8 * (i + 1)));
  return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);  // exact: small integers
}

// 16 int8 activations (k = 0..15) -> 16 bf16 in the same order as widen_codes.
__device__ __forceinline__ void widen_acts(uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w0 = __byte_perm(v.x, v.y, 0x5140);  // x0 x4 x1 x5
  const uint32_t w1 = __byte_perm(v.x, v.y, 0x7362);  // x2 x6 x3 x7
  const uint32_t w2 = __byte_perm(v.z, v.w, 0x5140);
  const uint32_t w3 = __byte_perm(v.z, v.w, 0x7362);
  lo = make_uint4(bf16x2_s8(w0, 0), bf16x2_s8(w0, 2), bf16x2_s8(w1, 0), bf16x2_s8(w1, 2));
  hi = make_uint4(bf16x2_s8(w2, 0), bf16x2_s8(w2, 2), bf16x2_s8(w3, 0), bf16x2_s8(w3, 2));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Epilogue shared by the GEMM kernels.  Warps 0 .. EPI-1 read the accumulators (warp
// w may only address tensor-memory lanes 32 (w % 4) .. +31; with 8 warps the two
// halves of the token columns go to warps w and w + 4).  Without a K split they
// dequantise and store y directly; with one, every CTA of the cluster leaves its
// partials in its own shared memory and finishes a slice of the tokens from all of
// them through distributed shared memory.  Called by all NTHR threads of the CTA.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Epilogue shared by the GEMM kernels.  Warps 0 .. EPI-1 read the accumulators (warp
// w may only address tensor-memory lanes 32 (w % 4) .. +31; with 8 warps the two
// halves of the token columns go to warps w and w + 4).  Without a K split they
// dequantise and store y directly; with one, every CTA of the cluster leaves its
// partials in its own shared memory and finishes a slice of the tokens from all of
// them through distributed shared memory.  Called by all NTHR threads of the CTA;
// `scale` holds, per token of the tile, s_x and fl(fl(gamma * s_x) / 127)
// (2 x BN floats, filled before the main loop).
template <int EPI, int NTHR>
__device__ __forceinline__ void epilogue(const Args& a, uint32_t tmem, float* part, volatile int* abort_flag,
                                         int any_fail, int nk, int n0, int m0, uint32_t crank,
                                         const float* scale) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BN = a.BN;
  const int quarter = warp & 3, half = warp >> 2;
  const int cols = BN / (EPI / 4), c_begin = half * cols;
  const int row = quarter * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
  const float gam = __ldg(a.w_scale);
  const float* sxs = scale;       // [BN] s_x of the tile's tokens
  const float* cs = scale + BN;   // [BN] dequantisation scales
  int cluster_fail = any_fail;
  if (a.ksplit > 1) {
    // publish this CTA's failure state and partials, then combine across the cluster
    if (warp < EPI && !any_fail) {
      for (int c0 = c_begin; c0 < c_begin + cols; c0 += 8) {
        uint32_t v[8];
        if (nk > 0) {
          tmem_ld8(taddr + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) v[t] = 0u;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) part[(size_t)(c0 + t) * BM + row] = __uint_as_float(v[t]);
      }
    }
    if (tid == 0) *abort_flag = any_fail;
    cluster_sync();
    for (int rk = 0; rk < a.ksplit; ++rk)
      cluster_fail |= *static_cast<volatile int*>(__cluster_map_shared_rank((void*)abort_flag, (unsigned)rk));
    if (!cluster_fail) {
      // CTA crank finishes tokens [t0, t1) of the tile for all 128 rows; that slice is
      // contiguous in every CTA's [BN][BM] partials, read 4 floats at a time
      const int per = (((BN + a.ksplit - 1) / a.ksplit) + 7) & ~7;
      const int t0 = min(BN, (int)crank * per), t1 = min(BN, t0 + per);
      const float4* src[kMaxCluster];
#pragma unroll
      for (int rk = 0; rk < kMaxCluster; ++rk)
        src[rk] = static_cast<const float4*>(
            __cluster_map_shared_rank((void*)(part + (size_t)t0 * BM), (unsigned)(rk < a.ksplit ? rk : 0)));
      const int nvec = (t1 - t0) * BM / 4;
      for (int e = tid; e < nvec; e += NTHR) {
        float4 v[kMaxCluster];  // every rank's partials in flight together
#pragma unroll
        for (int rk = 0; rk < kMaxCluster; ++rk) v[rk] = rk < a.ksplit ? src[rk][e] : make_float4(0.f, 0.f, 0.f, 0.f);
        // integers below 2^24 in magnitude: the fp32 sums are exact
        float4 acc = v[0];
#pragma unroll
        for (int rk = 1; rk < kMaxCluster; ++rk) {
          acc.x = __fadd_rn(acc.x, v[rk].x); acc.y = __fadd_rn(acc.y, v[rk].y);
          acc.z = __fadd_rn(acc.z, v[rk].z); acc.w = __fadd_rn(acc.w, v[rk].w);
        }
        const int j = t0 + (4 * e) / BM, rr = (4 * e) % BM;
        const int m = m0 + j;
        if (m < a.M) {
          const float sm = sxs[j], c = cs[j];
          const float av[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int n = n0 + rr + t;
            if (n < a.N) {
              a.y[(size_t)m * a.N + n] = dequant_f(av[t], c, gam, sm);
              if (a.acc_out) a.acc_out[(size_t)m * a.N + n] = __float2int_rn(av[t]);
            }
          }
        }
      }
    }
    cluster_sync();  // no CTA leaves while others still read its shared memory
  } else if (warp < EPI && !any_fail) {
    const int n = n0 + row;
    const bool nv = n < a.N;
    if ((cols & 31) == 0) {
      for (int c0 = c_begin; c0 < c_begin + cols; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int j = c0 + t, m = m0 + j;
          if (m < a.M && nv) {
            const float acc = __uint_as_float(v[t]);
            a.y[(size_t)m * a.N + n] = dequant_f(acc, cs[j], gam, sxs[j]);
            if (a.acc_out) a.acc_out[(size_t)m * a.N + n] = __float2int_rn(acc);
          }
        }
      }
    } else {
      for (int c0 = c_begin; c0 < c_begin + cols; c0 += 8) {
        uint32_t v[8];
        tmem_ld8(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int j = c0 + t, m = m0 + j;
          if (m < a.M && nv) {
            const float acc = __uint_as_float(v[t]);
            a.y[(size_t)m * a.N + n] = dequant_f(acc, cs[j], gam, sxs[j]);
            if (a.acc_out) a.acc_out[(size_t)m * a.N + n] = __float2int_rn(acc);
          }
        }
      }
    }
  }
  if (tid == 0 && cluster_fail) atomicExch(&g_gemm_status, (int)TW_ERR_TIMEOUT);
}

// Per-token scales of the tile into shared memory (called by `nthr` threads).
__device__ __forceinline__ void load_scales(const Args& a, int m0, float* scale, int t, int nthr) {
  const float gam = __ldg(a.w_scale);
  for (int j = t; j < a.BN; j += nthr) {
    const float sm = (m0 + j < a.M) ? __ldg(a.s_x + m0 + j) : 0.0f;
    scale[j] = sm;
    scale[a.BN + j] = dequant_scale(gam, sm);
  }
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(Args a) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const int BN = a.BN, NS = a.nstages;
  const uint32_t b_stage_bytes = (uint32_t)BN * BK * 2;
  const uint32_t stage_bytes = A_STAGE_BYTES + b_stage_bytes;
  // control block after the stages (or the split-K partials, whichever is larger)
  unsigned char* ctrl = gbase + a.ctrl_off;
  const uint32_t bar_full = smem_u32(ctrl);        // [NS]
  const uint32_t bar_empty = bar_full + 8 * kMaxStages;  // [NS]
  const uint32_t bar_done = bar_empty + 8 * kMaxStages;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctrl + 16 * kMaxStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 16 * kMaxStages + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = a.ksplit > 1 ? cluster_ctarank() : 0u;
  const int n0 = blockIdx.x / a.ksplit * BM;  // clusters are consecutive blocks along x
  const int m0 = blockIdx.y * BN;
  const int kst0 = (int)crank * a.kstages_per_split;
  const int nkst_total = (a.K + BK - 1) / BK;
  const int nk = max(0, min(a.kstages_per_split, nkst_total - kst0));

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, kProducers);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = g_gemm_abort_test;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp < 4) {
    // ------------------------------------------------------------ producers
    // Each thread owns weight row r of the tile and BN/32 16-byte units of the
    // activations per stage.  The global loads of stage i+1 are issued before
    // stage i is widened and stored, so their latency overlaps that work.
    const int K = a.K, Kw = K >> 4;  // 32-bit packed words per row
    const int r = tid;               // weight row of this thread within the tile
    const int n = n0 + r;
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(a.packed) + (size_t)(n < a.N ? n : 0) * Kw;
    const int bunits = BN * 4;       // 16-byte units of int8 activations per stage
    const bool vec_ok = (Kw & 3) == 0;
    auto load_stage = [&](int i, uint32_t (&pw)[4], uint4 (&bv)[kMaxBUnits]) {
      const int kw0 = (kst0 + i) * (BK / 16);
      if (n < a.N && vec_ok && kw0 + 4 <= Kw) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(wrow + kw0));
        pw[0] = v.x; pw[1] = v.y; pw[2] = v.z; pw[3] = v.w;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) pw[q] = (n < a.N && kw0 + q < Kw) ? __ldg(wrow + kw0 + q) : 0x55555555u;
      }
#pragma unroll
      for (int t = 0; t < kMaxBUnits; ++t) {
        const int u = tid + t * kProducers;
        bv[t] = make_uint4(0u, 0u, 0u, 0u);
        if (u < bunits) {
          const int m = m0 + (u >> 2), k = (kw0 + (u & 3)) * 16;
          if (m < a.M && k < K) bv[t] = __ldg(reinterpret_cast<const uint4*>(a.x_q + (size_t)m * K + k));
        }
      }
    };
    load_scales(a, m0, reinterpret_cast<float*>(ctrl + kScaleOff), tid, kProducers);
    uint32_t pw[4];
    uint4 bv[kMaxBUnits];
    if (nk > 0) load_stage(0, pw, bv);
    for (int i = 0; i < nk; ++i) {
      const int s = i % NS;
      uint32_t pw_n[4];
      uint4 bv_n[kMaxBUnits];
      if (i + 1 < nk) load_stage(i + 1, pw_n, bv_n);
      if (i >= NS) {
        if (!mbar_wait(bar_empty + 8 * s, (uint32_t)(((i / NS) - 1) & 1), abort_flag)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
      }
      if (*abort_flag) {
        ok = false;
        break;
      }
      const uint32_t As = base + (uint32_t)s * stage_bytes;
      const uint32_t Bs = As + A_STAGE_BYTES;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 lo, hi;
        widen_codes(pw[q], lo, hi);  // 0x55555555 = sixteen zero codes
        st_shared_v4(As + sw128_off(r, 2 * q), lo);
        st_shared_v4(As + sw128_off(r, 2 * q + 1), hi);
      }
#pragma unroll
      for (int t = 0; t < kMaxBUnits; ++t) {
        const int u = tid + t * kProducers;
        if (u < bunits) {
          const int j = u >> 2, q = u & 3;
          uint4 lo, hi;
          widen_acts(bv[t], lo, hi);
          st_shared_v4(Bs + sw128_off(j, 2 * q), lo);
          st_shared_v4(Bs + sw128_off(j, 2 * q + 1), hi);
        }
      }
      fence_async_smem();
      mbar_arrive(bar_full + 8 * s);
      if (i + 1 < nk) {
#pragma unroll
        for (int q = 0; q < 4; ++q) pw[q] = pw_n[q];
#pragma unroll
        for (int t = 0; t < kMaxBUnits; ++t) bv[t] = bv_n[t];
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BN);
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % NS;
        if (!mbar_wait(bar_full + 8 * s, (uint32_t)((i / NS) & 1), abort_flag) || *abort_flag) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t As = base + (uint32_t)s * stage_bytes;
        const uint32_t Bs = As + A_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          mma_bf16(tmem, sw128_desc(As + 32 * kk), sw128_desc(Bs + 32 * kk), idesc, (i | kk) ? 1u : 0u);
        }
        mma_commit(bar_empty + 8 * s);
        ++issued;
      }
      (void)issued;
      mma_commit(bar_done);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ epilogue
  // All threads wait until the accumulators are final (or the MMAs issued before an
  // abort have drained), so tensor memory is never freed under a running MMA.
  const bool done_ok = mbar_wait(bar_done, 0);
  tc_fence_after();
  __syncthreads();
  const bool failed = !done_ok || *abort_flag != 0 || !ok;
  const int any_fail = __syncthreads_or(failed ? 1 : 0);
  epilogue<4, kThreads>(a, tmem, reinterpret_cast<float*>(gbase), abort_flag, any_fail, nk, n0, m0, crank,
                        reinterpret_cast<const float*>(ctrl + kScaleOff));

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}


// ----------------------------------------------------------------------------
// TMA-fed variant (K % 64 == 0).  One thread issues 2-D tensor copies
// (cp.async.bulk.tensor) of the activation tiles: with the workspace, the bf16 copy
// straight into the operand stage (128-byte swizzle done by the copy engine);
// without it, raw int8 tiles into a small ring.  The packed weight tile is only 16
// bytes per row and stage, a poor shape for the copy engine, so each converter
// thread fetches its own 8 bytes with cp.async, kARing stages ahead, and widens
// exactly what it fetched.  One thread issues the MMAs.
constexpr int kTmaConv = 256;     // converter threads (warps 0-7); also the epilogue
constexpr int kTmaThreads = 320;  // + warp 8 (tensor copies) + warp 9 (TMEM, MMA)
constexpr int kRawStages = 4;                 // raw int8 activation tiles in flight (no workspace)
constexpr int A_RAW_BYTES = BM * (BK / 4);    // 2 KB of packed codes per stage
constexpr int kARing = 8;                     // stages of packed codes in flight (cp.async)

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// kBPre: the activations were widened beforehand (bf16, MMA K order) and mapB
// describes that copy with 128-byte swizzle, so its tiles land directly in the
// operand stage and the converters widen only the weights.
template <bool kBPre>
__global__ void __launch_bounds__(kTmaThreads, 1)
    gemm_tma_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, Args a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw0 = smem_u32(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw0);
  const int BN = a.BN, NS = a.nstages, RS = kRawStages;
  (void)mapA;
  const uint32_t op_bytes = A_STAGE_BYTES + (uint32_t)BN * BK * 2;   // multiple of 1024
  const uint32_t raw_bytes = kBPre ? 0u : (uint32_t)BN * BK;         // raw int8 activations
  const uint32_t op0 = base;
  const uint32_t araw = base + (uint32_t)NS * op_bytes;              // [kARing][128 rows][16 B]
  const uint32_t rawbase = araw + (uint32_t)kARing * A_RAW_BYTES;    // [RS][raw_bytes]
  unsigned char* ctrl = gbase + a.ctrl_off;
  const uint32_t raw_full = smem_u32(ctrl);           // [kRawStages]
  const uint32_t raw_empty = raw_full + 8 * kRawStages;
  const uint32_t op_full = raw_empty + 8 * kRawStages;  // [kMaxStages]
  const uint32_t op_empty = op_full + 8 * kMaxStages;
  const uint32_t bar_done = op_empty + 8 * kMaxStages;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctrl + 16 * kRawStages + 16 * kMaxStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 16 * kRawStages + 16 * kMaxStages + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = a.ksplit > 1 ? cluster_ctarank() : 0u;
  const int n0 = blockIdx.x / a.ksplit * BM;
  const int m0 = blockIdx.y * BN;
  const int kst0 = (int)crank * a.kstages_per_split;
  const int nkst_total = a.K / BK;
  const int nk = max(0, min(a.kstages_per_split, nkst_total - kst0));

  if (tid == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(raw_full + 8 * s, 1);
      mbar_init(raw_empty + 8 * s, kTmaConv / 32);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(op_full + 8 * s, kTmaConv / 32 + (kBPre ? 1 : 0));
      mbar_init(op_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = g_gemm_abort_test;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 8) {
    // ------------------------------------------------------------ tensor copies
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)) : "memory");
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int kb = (kst0 + i) * BK;  // first k of the stage
        if constexpr (kBPre) {
          const int s = i % NS;
          if (i >= NS && !mbar_wait(op_empty + 8 * s, (uint32_t)(((i / NS) - 1) & 1), abort_flag)) {
            ok = false;
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(op_full + 8 * s, (uint32_t)BN * BK * 2);
          tma_load_2d(op0 + (uint32_t)s * op_bytes + A_STAGE_BYTES, &mapB, kb, m0, op_full + 8 * s);
        } else {
          const int rs = i % RS;
          if (i >= RS && !mbar_wait(raw_empty + 8 * rs, (uint32_t)(((i / RS) - 1) & 1), abort_flag)) {
            ok = false;
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(raw_full + 8 * rs, raw_bytes);
          tma_load_2d(rawbase + (uint32_t)rs * raw_bytes, &mapB, kb, m0, raw_full + 8 * rs);
        }
        issued = i + 1;
      }
      // never leave with tensor copies in flight into this CTA's shared memory
      if constexpr (kBPre) {
        for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(op_full + 8 * (i % NS), (uint32_t)((i / NS) & 1));
      } else {
        for (int i = max(0, issued - RS); i < issued; ++i) mbar_wait(raw_full + 8 * (i % RS), (uint32_t)((i / RS) & 1));
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % NS;
        if (!mbar_wait(op_full + 8 * s, (uint32_t)((i / NS) & 1), abort_flag) || *abort_flag) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t As = op0 + (uint32_t)s * op_bytes;
        const uint32_t Bs = As + A_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16(tmem, sw128_desc(As + 32 * kk), sw128_desc(Bs + 32 * kk), idesc, (i | kk) ? 1u : 0u);
        mma_commit(op_empty + 8 * s);
      }
      mma_commit(bar_done);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ converters (warps 0-7)
    load_scales(a, m0, reinterpret_cast<float*>(ctrl + kScaleOff), tid, kTmaConv);
    const int bunits = BN * 4;  // 16-byte units of raw activations per stage
    // thread t owns 8 bytes (32 codes) of weight row t / 2 in every stage
    const int r = tid >> 1, h = tid & 1;
    const bool rowv = n0 + r < a.N;
    const uint8_t* gA = a.packed + (size_t)(rowv ? n0 + r : 0) * (a.K / 4) + h * 8;
    const uint32_t aslot = araw + (uint32_t)(r * 16 + h * 8);
    auto fetch = [&](int i) {  // stage i of this CTA -> ring slot i % kARing (one group per stage)
      if (i < nk && rowv) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(aslot + (uint32_t)(i % kARing) * A_RAW_BYTES),
                     "l"(gA + (size_t)(kst0 + i) * (BK / 4))
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int i = 0; i < kARing; ++i) fetch(i);
    for (int i = 0; i < nk; ++i) {
      const int rs = i % RS, s = i % NS;
      asm volatile("cp.async.wait_group %0;" ::"n"(kARing - 1) : "memory");  // this thread's stage i
      int okw = 1;
      if (lane == 0) {
        okw = (kBPre || mbar_wait(raw_full + 8 * rs, (uint32_t)((i / RS) & 1), abort_flag)) &&
              (i < NS || mbar_wait(op_empty + 8 * s, (uint32_t)(((i / NS) - 1) & 1), abort_flag));
      }
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      const uint32_t rB = rawbase + (uint32_t)rs * raw_bytes;
      const uint32_t As = op0 + (uint32_t)s * op_bytes, Bs = As + A_STAGE_BYTES;
      {  // weights: widen the 32 codes this thread fetched into 4 chunks of its row
        uint32_t w0, w1;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(w0), "=r"(w1)
                     : "r"(aslot + (uint32_t)(i % kARing) * A_RAW_BYTES));
        if (!rowv) w0 = w1 = 0x55555555u;  // rows past N: zero codes (their outputs are dropped)
        uint4 lo, hi;
        widen_codes(w0, lo, hi);
        st_shared_v4(As + sw128_off(r, 4 * h + 0), lo);
        st_shared_v4(As + sw128_off(r, 4 * h + 1), hi);
        widen_codes(w1, lo, hi);
        st_shared_v4(As + sw128_off(r, 4 * h + 2), lo);
        st_shared_v4(As + sw128_off(r, 4 * h + 3), hi);
      }
      fetch(i + kARing);  // the slot just read is free again
      for (int u = tid; u < (kBPre ? 0 : bunits); u += kTmaConv) {  // activations: 16 int8 -> 16 bf16
        const int j = u >> 2, q = u & 3;
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(rB + (uint32_t)(16 * u)));
        uint4 lo, hi;
        widen_acts(v, lo, hi);
        st_shared_v4(Bs + sw128_off(j, 2 * q), lo);
        st_shared_v4(Bs + sw128_off(j, 2 * q + 1), hi);
      }
      fence_async_smem();  // this thread's operand stores become visible to the tensor cores
      __syncwarp();
      if (lane == 0) {     // one arrival per warp (after all its lanes fenced)
        mbar_arrive(op_full + 8 * s);
        if (!kBPre) mbar_arrive(raw_empty + 8 * rs);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may land after this CTA is gone
  }

  // ------------------------------------------------------------ epilogue
  const bool done_ok = mbar_wait(bar_done, 0);
  tc_fence_after();
  __syncthreads();
  const bool failed = !done_ok || *abort_flag != 0 || !ok;
  const int any_fail = __syncthreads_or(failed ? 1 : 0);
  epilogue<8, kTmaThreads>(a, tmem, reinterpret_cast<float*>(gbase), abort_flag, any_fail, nk, n0, m0, crank,
                           reinterpret_cast<const float*>(ctrl + kScaleOff));

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}


// ----------------------------------------------------------------------------
// Tokens-on-M variant (1 <= M <= 128, K % 64 == 0, activations pre-widened into the
// workspace).  One tcgen05.mma costs the same time whatever its N, so the
// instruction count is what matters: with the tokens (padded to 128) as the MMA's
// M side and 256 weight rows as its N side, a weight tile needs half the
// instructions of a 128-row tile.  The accumulators are [128 tokens][256 rows]
// in tensor memory: each thread of the epilogue owns one token.
// Pipeline: the activation tiles (TMA, 16 KB) have a ring of their own, deep enough
// (kTokNA stages) to hide the copy latency behind the MMAs; the widened weight tiles
// (32 KB) need only kTokNB stages, since their packed codes are fetched kTokARing
// stages ahead with cp.async.  Launched with programmatic dependent launch: the
// weight fetches start before the widening kernel in front of it has finished.
constexpr int TBN = 256;                       // weight rows per CTA (MMA N)
constexpr int TB_STAGE = TBN * BK * 2;         // 32 KB of widened weights per stage
constexpr int TA_STAGE = 128 * BK * 2;         // 16 KB of activations per stage
constexpr int TW_RAW = TBN * (BK / 4);         // 4 KB of packed codes per stage
constexpr int kTokNA = 6, kTokNB = 3, kTokARing = 4;
constexpr int kPartStride = TBN + 4;           // floats per token row of the staged partials
constexpr int kTokThreads = 320;               // warps 0-7 convert + epilogue, 8: TMA, 9: MMA

__device__ __forceinline__ void pdl_wait_all() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Epilogue of the tokens-on-M kernel.  Warp w reads tensor-memory lanes 32 (w % 4)
// .. +31 (its tokens) and the weight-row half w / 4, 32 columns at a time, and
// stages them in its own CTA's shared memory as part[token][row] (rows padded to
// 260 floats: conflict-free for one token per lane).  The 256 rows of the tile are
// finished by the ksplit CTAs of the cluster, W = 256 / ksplit each: after a cluster
// barrier every CTA reads its rows of every rank's partials, four consecutive rows of
// a token per thread (each warp reads and stores 512 contiguous bytes), adds them in
// fp32 (the partial sums are integers below 2^24 in magnitude, so every sum is
// exact) and stores them dequantised as one float4; a second barrier keeps every CTA
// until its peers are done reading.  The flags of all ranks are read before the
// second barrier.
__device__ __forceinline__ void tok_epilogue(const Args& a, uint32_t tmem, float* part, volatile int* abort_flag,
                                             int any_fail, int nk, int n0, uint32_t crank, const float* scale) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int m = quarter * 32 + lane;  // token of this thread
  const int ks = a.ksplit, W = TBN / ks;
  const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
  const float gam = __ldg(a.w_scale);
  const bool vec = (a.N & 3) == 0 && (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.acc_out) & 15) == 0;  // 16-byte stores allowed
  if (warp < 8 && quarter * 32 < a.M && !any_fail) {
    for (int c0 = half * 128; c0 < half * 128 + 128; c0 += 32) {
      uint32_t v[32];
      if (nk > 0) {
        tmem_ld32(taddr + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = 0u;
      }
      uint4* dst = reinterpret_cast<uint4*>(part + (size_t)m * kPartStride + c0);
#pragma unroll
      for (int t = 0; t < 8; ++t) dst[t] = make_uint4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
    }
  }
  if (tid == 0) *abort_flag = any_fail;
  if (ks > 1) cluster_sync();
  else __syncthreads();
  int cluster_fail = any_fail;
  if (ks > 1) {
    for (int rk = 0; rk < ks; ++rk)
      cluster_fail |= *static_cast<volatile int*>(__cluster_map_shared_rank((void*)abort_flag, (unsigned)rk));
  }
  if (!cluster_fail) {
    const int per4 = W / 4;
    const int r0 = (int)crank * W;
    const float* src[kMaxCluster];
#pragma unroll
    for (int rk = 0; rk < kMaxCluster; ++rk)
      src[rk] = ks > 1 ? static_cast<const float*>(__cluster_map_shared_rank((void*)part, (unsigned)(rk < ks ? rk : 0)))
                       : part;
    for (int it = tid; it < a.M * per4; it += kTokThreads) {
      const int mm = it / per4, c = r0 + 4 * (it % per4);
      float4 acc = *reinterpret_cast<const float4*>(src[0] + (size_t)mm * kPartStride + c);
#pragma unroll
      for (int rk = 1; rk < kMaxCluster; ++rk) {
        if (rk < ks) {
          const float4 f = *reinterpret_cast<const float4*>(src[rk] + (size_t)mm * kPartStride + c);
          acc.x = __fadd_rn(acc.x, f.x); acc.y = __fadd_rn(acc.y, f.y);
          acc.z = __fadd_rn(acc.z, f.z); acc.w = __fadd_rn(acc.w, f.w);
        }
      }
      const int n = n0 + c;
      const float sm = scale[mm], cs = scale[128 + mm];
      float* yrow = a.y + (size_t)mm * a.N;
      if (vec && n + 4 <= a.N) {
        *reinterpret_cast<float4*>(yrow + n) = make_float4(dequant_f(acc.x, cs, gam, sm), dequant_f(acc.y, cs, gam, sm),
                                                           dequant_f(acc.z, cs, gam, sm), dequant_f(acc.w, cs, gam, sm));
        if (a.acc_out)
          *reinterpret_cast<int4*>(a.acc_out + (size_t)mm * a.N + n) =
              make_int4(__float2int_rn(acc.x), __float2int_rn(acc.y), __float2int_rn(acc.z), __float2int_rn(acc.w));
      } else {
        const float av[4] = {acc.x, acc.y, acc.z, acc.w};
        for (int q = 0; q < 4; ++q) {
          if (n + q < a.N) {
            yrow[n + q] = dequant_f(av[q], cs, gam, sm);
            if (a.acc_out) a.acc_out[(size_t)mm * a.N + n + q] = __float2int_rn(av[q]);
          }
        }
      }
    }
  }
  if (ks > 1) cluster_sync();  // no CTA leaves while others still read its shared memory
  if (tid == 0 && cluster_fail) atomicExch(&g_gemm_status, (int)TW_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kTokThreads, 1)
    gemm_tok_kernel(const __grid_constant__ CUtensorMap mapX, Args a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw0 = smem_u32(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw0);
  const uint32_t a0 = base;                                         // [kTokNA][16 KB] activations
  const uint32_t b0 = a0 + (uint32_t)kTokNA * TA_STAGE;             // [kTokNB][32 KB] widened weights
  const uint32_t wraw = b0 + (uint32_t)kTokNB * TB_STAGE;           // [kTokARing][256 rows][16 B]
  unsigned char* ctrl = gbase + a.ctrl_off;
  const uint32_t a_full = smem_u32(ctrl);                            // [kTokNA]
  const uint32_t a_empty = a_full + 8 * kTokNA;
  const uint32_t b_full = a_empty + 8 * kTokNA;                      // [kTokNB]
  const uint32_t b_empty = b_full + 8 * kTokNB;
  const uint32_t bar_done = b_empty + 8 * kTokNB;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctrl + 16 * (kTokNA + kTokNB) + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 16 * (kTokNA + kTokNB) + 12);
  float* scale = reinterpret_cast<float*>(ctrl + kScaleOff);  // [128] s_x, [128] dequantisation scales

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = a.ksplit > 1 ? cluster_ctarank() : 0u;
  const int n0 = blockIdx.x / a.ksplit * TBN;
  const int kst0 = (int)crank * a.kstages_per_split;
  const int nk = max(0, min(a.kstages_per_split, a.K / BK - kst0));

  if (tid == 0) {
    for (int s = 0; s < kTokNA; ++s) {
      mbar_init(a_full + 8 * s, 1);
      mbar_init(a_empty + 8 * s, 1);
    }
    for (int s = 0; s < kTokNB; ++s) {
      mbar_init(b_full + 8 * s, kTmaConv / 32);
      mbar_init(b_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = g_gemm_abort_test;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  pdl_trigger();

  if (warp == 8) {
    // ------------------------------------------------------------ activation tiles
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapX)) : "memory");
      pdl_wait_all();  // the widened activations come from the kernel in front
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kTokNA;
        if (i >= kTokNA && !mbar_wait(a_empty + 8 * s, (uint32_t)(((i / kTokNA) - 1) & 1), abort_flag)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(a_full + 8 * s, (uint32_t)TA_STAGE);
        tma_load_2d(a0 + (uint32_t)s * TA_STAGE, &mapX, (kst0 + i) * BK, 0, a_full + 8 * s);
        issued = i + 1;
      }
      for (int i = max(0, issued - kTokNA); i < issued; ++i)
        mbar_wait(a_full + 8 * (i % kTokNA), (uint32_t)((i / kTokNA) & 1));
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TBN >> 3) << 17) | ((128u >> 4) << 24);
      for (int i = 0; i < nk; ++i) {
        const int sa = i % kTokNA, sb = i % kTokNB;
        if (!mbar_wait(a_full + 8 * sa, (uint32_t)((i / kTokNA) & 1), abort_flag) ||
            !mbar_wait(b_full + 8 * sb, (uint32_t)((i / kTokNB) & 1), abort_flag) || *abort_flag) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t As = a0 + (uint32_t)sa * TA_STAGE, Bs = b0 + (uint32_t)sb * TB_STAGE;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16(tmem, sw128_desc(As + 32 * kk), sw128_desc(Bs + 32 * kk), idesc, (i | kk) ? 1u : 0u);
        mma_commit(a_empty + 8 * sa);
        mma_commit(b_empty + 8 * sb);
      }
      mma_commit(bar_done);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ weight converters (warps 0-7)
    const int r = tid;  // weight row of the tile owned by this thread
    const bool rowv = n0 + r < a.N;
    const uint8_t* gW = a.packed + (size_t)(rowv ? n0 + r : 0) * (a.K / 4);
    const uint32_t rslot = wraw + (uint32_t)(r * 16);
    auto fetch = [&](int i) {
      if (i < nk && rowv) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(rslot + (uint32_t)(i % kTokARing) * TW_RAW),
                     "l"(gW + (size_t)(kst0 + i) * (BK / 4))
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int i = 0; i < kTokARing; ++i) fetch(i);  // weights never depend on the kernel in front
    for (int j = tid; j < 128; j += kTmaConv) {     // s_x was written two kernels back
      const float sm = j < a.M ? __ldg(a.s_x + j) : 0.0f;
      scale[j] = sm;
      scale[128 + j] = dequant_scale(__ldg(a.w_scale), sm);
    }
    for (int i = 0; i < nk; ++i) {
      const int s = i % kTokNB;
      asm volatile("cp.async.wait_group %0;" ::"n"(kTokARing - 1) : "memory");
      int okw = 1;
      if (lane == 0) okw = i < kTokNB || mbar_wait(b_empty + 8 * s, (uint32_t)(((i / kTokNB) - 1) & 1), abort_flag);
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      uint4 w;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                   : "r"(rslot + (uint32_t)(i % kTokARing) * TW_RAW));
      if (!rowv) w = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
      fetch(i + kTokARing);
      const uint32_t Bs = b0 + (uint32_t)s * TB_STAGE;
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 lo, hi;
        widen_codes(wv[q], lo, hi);
        st_shared_v4(Bs + sw128_off(r, 2 * q), lo);
        st_shared_v4(Bs + sw128_off(r, 2 * q + 1), hi);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_full + 8 * s);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  pdl_wait_all();  // every thread stores outputs: the kernel in front must have finished
  const bool done_ok = mbar_wait(bar_done, 0);
  tc_fence_after();
  __syncthreads();
  const bool failed = !done_ok || *abort_flag != 0 || !ok;
  const int any_fail = __syncthreads_or(failed ? 1 : 0);
  tok_epilogue(a, tmem, reinterpret_cast<float*>(gbase), abort_flag, any_fail, nk, n0, crank, scale);

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}

// x_q [M][K] int8 -> bf16 [M][K], each 16-element group in the MMA K order
// 0,4,1,5,2,6,3,7,8,12,9,13,10,14,11,15 (the order widen_codes gives the weights).
__global__ void __launch_bounds__(256) widen_acts_kernel(const int8_t* __restrict__ x_q, long long groups,
                                                         uint4* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the GEMM behind may start fetching weights
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  uint4 lo, hi;
  widen_acts(__ldg(reinterpret_cast<const uint4*>(x_q) + g), lo, hi);
  out[2 * g] = lo;
  out[2 * g + 1] = hi;
}

}  // namespace gemm
}  // namespace tw

namespace {

struct GemmPlan {
  int BN, nstages, ksplit, kstages_per_split, tiles_n, tiles_m;
  uint32_t tmem_cols, ctrl_off;
  size_t smem;
};

// Tokens per tile: M rounded up to 16, at most 256; K split over a cluster so that
// the grid comes close to one CTA per SM without slicing K below 8 stages.
bool gemm_plan(int M, int N, int K, int num_sms, GemmPlan& p) {
  using namespace tw::gemm;
  p.BN = ((M + 15) / 16) * 16;
  if (p.BN > 256) p.BN = 256;
  p.tiles_n = (N + BM - 1) / BM;
  p.tiles_m = (M + p.BN - 1) / p.BN;
  const int nkst = (K + BK - 1) / BK;
  const long long tiles = (long long)p.tiles_n * p.tiles_m;
  p.ksplit = 1;
  while (p.ksplit < kMaxCluster && tiles * (p.ksplit * 2) <= num_sms && nkst / (p.ksplit * 2) >= 8) p.ksplit *= 2;
  p.kstages_per_split = (nkst + p.ksplit - 1) / p.ksplit;
  const size_t stage = (size_t)A_STAGE_BYTES + (size_t)p.BN * BK * 2;
  const size_t budget = 200 * 1024;
  p.nstages = (int)(budget / stage);
  if (p.nstages > kMaxStages) p.nstages = kMaxStages;
  if (p.nstages > p.kstages_per_split) p.nstages = p.kstages_per_split < 2 ? 2 : p.kstages_per_split;
  if (p.nstages < 2) return false;
  // the partial accumulators of a split reuse the stage memory: BN x 128 fp32
  size_t body = (size_t)p.nstages * stage;
  const size_t partial = (size_t)p.BN * BM * 4;
  if (p.ksplit > 1 && body < partial) body = partial;
  p.ctrl_off = (uint32_t)body;
  p.smem = 1024 + body + kCtrlBytes;
  // at least 114 KB so that one CTA runs per SM: its tensor memory (<= 256 of the 512
  // columns) can then always be allocated, also next to a CTA of a concurrent launch
  if (p.smem < 114 * 1024) p.smem = 114 * 1024;
  p.tmem_cols = 32;
  while ((int)p.tmem_cols < p.BN) p.tmem_cols <<= 1;
  return p.smem <= 227 * 1024;
}

}  // namespace

namespace {

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load(std::memory_order_acquire);
  if (!f) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f) {
      cudaGetLastError();
      return nullptr;
    }
    fn.store(f, std::memory_order_release);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// 2-D byte tensor [rows][cols] (row stride = cols bytes), tiles of box_rows x box_cols,
// no swizzle, zero fill outside the tensor.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, int esize, const void* base, uint64_t cols,
               uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, type, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows][cols] (row stride = cols bytes), no swizzle, zero fill outside.
bool encode_bytes_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                     uint32_t box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, cols, rows, box_cols, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Shared memory of the TMA kernel: NS operand stages + 4 raw stages (or the split-K
// partials, whichever is larger) + barriers; at least 114 KB (one CTA per SM).
bool gemm_tma_plan(GemmPlan& p, bool bpre) {
  using namespace tw::gemm;
  const size_t raw = bpre ? 0 : (size_t)p.BN * BK;
  const size_t op = (size_t)A_STAGE_BYTES + (size_t)p.BN * BK * 2;
  const size_t fixed = (size_t)kARing * A_RAW_BYTES + (bpre ? 0 : (size_t)kRawStages * raw);
  int ns = (int)((200 * 1024 - fixed) / op);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns > p.kstages_per_split) ns = p.kstages_per_split < 2 ? 2 : p.kstages_per_split;
  if (ns < 2) return false;
  p.nstages = ns;
  size_t body = (size_t)ns * op + fixed;
  const size_t partial = (size_t)p.BN * BM * 4;
  if (p.ksplit > 1 && body < partial) body = partial;
  p.ctrl_off = (uint32_t)body;
  p.smem = 1024 + body + kCtrlBytes;
  if (p.smem < 114 * 1024) p.smem = 114 * 1024;
  return p.smem <= 227 * 1024;
}

}  // namespace

size_t tw_gemm_ws_size(long long M, long long K) { return (size_t)(M * K * 2); }

namespace {

// Tokens-on-M plan: ceil(N / 256) weight tiles, K split over a cluster so that the
// grid comes close to one CTA per SM without slicing K below 8 stages.
bool gemm_tok_plan(int M, int N, int K, int num_sms, GemmPlan& p) {
  using namespace tw::gemm;
  if (M > 128 || K % 64 != 0) return false;
  p.BN = 128;
  p.tiles_n = (N + TBN - 1) / TBN;
  p.tiles_m = 1;
  const int nkst = K / BK;
  p.ksplit = 1;
  while (p.ksplit < kMaxCluster && (long long)p.tiles_n * (p.ksplit * 2) <= num_sms && nkst / (p.ksplit * 2) >= 8)
    p.ksplit *= 2;
  p.kstages_per_split = (nkst + p.ksplit - 1) / p.ksplit;
  p.nstages = kTokNA;
  size_t body = (size_t)kTokNA * TA_STAGE + (size_t)kTokNB * TB_STAGE + (size_t)kTokARing * TW_RAW;
  const size_t partial = (size_t)128 * kPartStride * 4;
  if (body < partial) body = partial;
  p.ctrl_off = (uint32_t)body;
  p.smem = 1024 + body + kCtrlBytes;
  if (p.smem < 114 * 1024) p.smem = 114 * 1024;
  p.tmem_cols = 256;
  return p.smem <= 227 * 1024;
}

}  // namespace

cudaError_t tw_launch_gemm(const uint8_t* packed, const float* w_scale, const int8_t* x_q, const float* s_x,
                           int M, int N, int K, float* y, int32_t* acc_out, void* workspace, cudaStream_t stream,
                           int num_sms, int* unsupported) {
  using namespace tw::gemm;
  *unsupported = 0;
  GemmPlan tp;
  if (workspace != nullptr && gemm_tok_plan(M, N, K, num_sms, tp)) {
    CUtensorMap mapX;
    if (encode_2d(&mapX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, workspace, (uint64_t)K, (uint64_t)M, BK, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
      const long long groups = (long long)M * K / 16;
      widen_acts_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, stream>>>(x_q, groups,
                                                                                static_cast<uint4*>(workspace));
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      Args a = {};
      a.packed = packed; a.w_scale = w_scale; a.x_q = x_q; a.s_x = s_x;
      a.M = M; a.N = N; a.K = K; a.BN = tp.BN; a.nstages = tp.nstages; a.ksplit = tp.ksplit;
      a.kstages_per_split = tp.kstages_per_split; a.tmem_cols = tp.tmem_cols; a.ctrl_off = tp.ctrl_off;
      a.y = y; a.acc_out = acc_out;
      e = cudaFuncSetAttribute(gemm_tok_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tp.smem);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(tp.tiles_n * tp.ksplit), 1);
      cfg.blockDim = dim3(kTokThreads);
      cfg.dynamicSmemBytes = tp.smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)tp.ksplit;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      return cudaLaunchKernelEx(&cfg, gemm_tok_kernel, mapX, a);
    }
  }
  if (K % 64 == 0) {
    GemmPlan p;
    CUtensorMap mapA, mapB;
    const bool bpre = workspace != nullptr;
    bool ok = gemm_plan(M, N, K, num_sms, p) && gemm_tma_plan(p, bpre) &&
              encode_bytes_2d(&mapA, packed, (uint64_t)K / 4, (uint64_t)N, BK / 4, BM);
    if (ok && bpre)
      ok = encode_2d(&mapB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, workspace, (uint64_t)K, (uint64_t)M, BK,
                     (uint32_t)p.BN, CU_TENSOR_MAP_SWIZZLE_128B);
    else if (ok)
      ok = encode_bytes_2d(&mapB, x_q, (uint64_t)K, (uint64_t)M, BK, (uint32_t)p.BN);
    if (ok) {
      if (bpre) {
        const long long groups = (long long)M * K / 16;
        widen_acts_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, stream>>>(x_q, groups,
                                                                                  static_cast<uint4*>(workspace));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      Args a = {};
      a.packed = packed; a.w_scale = w_scale; a.x_q = x_q; a.s_x = s_x;
      a.M = M; a.N = N; a.K = K; a.BN = p.BN; a.nstages = p.nstages; a.ksplit = p.ksplit;
      a.kstages_per_split = p.kstages_per_split; a.tmem_cols = p.tmem_cols; a.ctrl_off = p.ctrl_off;
      a.y = y; a.acc_out = acc_out;
      auto kern = bpre ? gemm_tma_kernel<true> : gemm_tma_kernel<false>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(p.tiles_n * p.ksplit), (unsigned)p.tiles_m);
      cfg.blockDim = dim3(kTmaThreads);
      cfg.dynamicSmemBytes = p.smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)p.ksplit;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, kern, mapA, mapB, a);
    }
  }
  GemmPlan p;
  if (K % 16 != 0 || !gemm_plan(M, N, K, num_sms, p)) {
    *unsupported = 1;
    return cudaSuccess;
  }
  Args a = {};
  a.packed = packed; a.w_scale = w_scale; a.x_q = x_q; a.s_x = s_x;
  a.M = M; a.N = N; a.K = K; a.BN = p.BN; a.nstages = p.nstages; a.ksplit = p.ksplit;
  a.kstages_per_split = p.kstages_per_split; a.tmem_cols = p.tmem_cols; a.ctrl_off = p.ctrl_off; a.y = y; a.acc_out = acc_out;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.tiles_n * p.ksplit), (unsigned)p.tiles_m);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.ksplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, a);
}

// Sets the GEMM's abort test switch (synchronous; diagnostics only).
cudaError_t tw_set_gemm_abort_test(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(tw::gemm::g_gemm_abort_test, &v, sizeof(int));
}

// Reads and clears the GEMM's device status word (synchronous; diagnostics only).
cudaError_t tw_read_gemm_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, tw::gemm::g_gemm_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(tw::gemm::g_gemm_status, &zero, sizeof(int));
}
