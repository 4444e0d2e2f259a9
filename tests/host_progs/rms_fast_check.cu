// Host driver for the float-float mean-square fast path of tw_common.cuh (the same
// __host__ __device__ code the fused GEMV prologues run), in two of the kernels' orders.
//   C = 0 (one CTA): 384 threads take 4-element units i = t, t + 384, ...; a 32-lane xor
//     butterfly per warp; a 16-lane xor butterfly over the 12 per-warp sums (zeros above),
//     lane 0's result.
//   C > 1 (a cluster of C CTAs sharing the row): rank r takes the 16-element groups
//     [r gw, (r + 1) gw), gw = ceil(K / 16 / C); in it thread t takes units u0 + t, u0 + t +
//     384, ... with one accumulator per vector component, combined as (s0 + s1) + (s2 + s3);
//     a 32-lane xor butterfly per warp; the 12 per-warp sums added in warp order; the C rank
//     sums added in rank order.
// Input: per case a line "K C" then K fp32 bit patterns (decimal).  Output per case:
// "ok ms_bits".
#include <algorithm>
#include <cstdio>
#include <vector>

#include "../../ternary_weight_quant_b300/csrc/tw_common.cuh"

int main() {
  int K;
  const int kThreads = 384, kWarps = 12;
  int C;
  while (std::scanf("%d %d", &K, &C) == 2) {
    std::vector<float> x(K);
    for (int k = 0; k < K; ++k) {
      unsigned b;
      if (std::scanf("%u", &b) != 1) return 1;
      x[k] = tw::f_from_bits(b);
    }
    if (C > 1) {
      const int Kw = K / 16, gw = (Kw + C - 1) / C;
      tw::FF total = {0.0f, 0.0f};
      for (int r = 0; r < C; ++r) {
        const int u0 = 4 * std::min(Kw, r * gw), u1 = 4 * std::min(Kw, (r + 1) * gw);
        std::vector<tw::FF> th(kThreads);
        for (int t = 0; t < kThreads; ++t) {
          tw::FF s4[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
          for (int u = u0 + t; u < u1; u += kThreads)
            for (int e = 0; e < 4; ++e) tw::ff_add_square(s4[e], x[4 * u + e]);
          tw::ff_add(s4[0], s4[1]);
          tw::ff_add(s4[2], s4[3]);
          tw::ff_add(s4[0], s4[2]);
          th[t] = s4[0];
        }
        tw::FF rank_sum = {0.0f, 0.0f};
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
          tw::ff_add(rank_sum, l[0]);
        }
        tw::ff_add(total, rank_sum);
      }
      float ms = 0.0f;
      const bool ok = tw::ff_mean_f32(total, K, 1.0f / (float)K, ms);
      std::printf("%d %u\n", ok ? 1 : 0, tw::f_bits(ms));
      continue;
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
