// Host driver for the integer RMSNorm-scale helpers of tw_common.cuh (the same
// __host__ __device__ code the kernels run).  Reads lines "hi lo E K eps_bits sh"
// (decimal) and prints "m e ms_bits inv_bits shr_hi shr_lo shr_exact": the double
// rounding of (hi:lo) 2^(2E - 364) as m 2^e, fl32(fl64(.) / K) and the RMSNorm scale
// as fp32 bit patterns, and (hi:lo) shifted right by sh with its exactness flag.
#include <cstdio>
#include <cstring>

#include "../../ternary_weight_quant_b300/csrc/tw_common.cuh"

int main() {
  unsigned long long hi, lo, epsb;
  int E, K, sh;
  while (std::scanf("%llu %llu %d %d %llu %d", &hi, &lo, &E, &K, &epsb, &sh) == 6) {
    tw::Sum128 s{lo, hi};
    const tw::KDiv d = tw::make_kdiv(K);
    unsigned long long m = 0;
    int e = 0;
    float ms = 0.0f;
    if (hi | lo) {
      tw::sum128_round53(s, E, m, e);
      ms = tw::div_k_round_f32(m, e, d);
    }
    float eps;
    const uint32_t eb = (uint32_t)epsb;
    std::memcpy(&eps, &eb, 4);
    const float inv = tw::rms_inv_sum128(s, E, d, eps);
    uint32_t msb, invb;
    std::memcpy(&msb, &ms, 4);
    std::memcpy(&invb, &inv, 4);
    tw::Sum128 t = s;
    const bool exact = tw::sum128_shr_exact(t, sh);
    std::printf("%llu %d %u %u %llu %llu %d\n", m, e, msb, invb, t.hi, t.lo, exact ? 1 : 0);
  }
  return 0;
}
