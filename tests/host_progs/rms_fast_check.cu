// Host driver for the float-float mean-square fast path of tw_common.cuh (the same
// __host__ __device__ code the fused GEMV prologue runs), in the kernel's order:
// 384 threads take 4-element units i = t, t + 384, ...; a 32-lane xor butterfly per
// warp; a 16-lane xor butterfly over the 12 per-warp sums (zeros above), lane 0's result.  Input: per
// case a line "K" then K fp32 bit patterns (decimal).  Output per case: "ok ms_bits".
#include <cstdio>
#include <vector>

#include "../../ternary_weight_quant_b300/csrc/tw_common.cuh"

int main() {
  int K;
  const int kThreads = 384, kWarps = 12;
  while (std::scanf("%d", &K) == 1) {
    std::vector<float> x(K);
    for (int k = 0; k < K; ++k) {
      unsigned b;
      if (std::scanf("%u", &b) != 1) return 1;
      x[k] = tw::f_from_bits(b);
    }
    std::vector<tw::FF> th(kThreads, tw::FF{0.0f, 0.0f});
    for (int t = 0; t < kThreads; ++t)
      for (int i = t; i < K / 4; i += kThreads)
        for (int e = 0; e < 4; ++e) tw::ff_add_square(th[t], x[4 * i + e]);
    std::vector<tw::FF> wsum(32, tw::FF{0.0f, 0.0f});
    for (int w = 0; w < kWarps; ++w) {
      std::vector<tw::FF> l(th.begin() + 32 * w, th.begin() + 32 * w + 32);
      for (int o = 16; o > 0; o >>= 1) {
        std::vector<tw::FF> n(32);
        for (int j = 0; j < 32; ++j) {
          n[j] = l[j];
          tw::ff_add(n[j], l[j ^ o]);
        }
        l = n;
      }
      wsum[w] = l[0];
    }
    for (int o = 8; o > 0; o >>= 1) {  // lanes 0-15; lane 0's value is then broadcast
      std::vector<tw::FF> n(32);
      for (int j = 0; j < 32; ++j) {
        n[j] = wsum[j];
        tw::ff_add(n[j], wsum[j ^ o]);
      }
      wsum = n;
    }
    float ms = 0.0f;
    const bool ok = tw::ff_mean_f32(wsum[0], K, 1.0f / (float)K, ms);
    std::printf("%d %u\n", ok ? 1 : 0, tw::f_bits(ms));
  }
  return 0;
}
