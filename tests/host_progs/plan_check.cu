// Host driver for the launch planning of the streaming GEMV and the GEMMs (the same host
// code the library runs; nothing is launched).  Reads lines "kind M N K sms" and prints the
// plan's fields, or "none" when the kernel does not take the shape.
//   kind: stream (tw_ternary_gemv), fused (tw_quant_gemv), gemm (128-row tiles, no
//   workspace), tma (the same with the workspace), tok (tokens-on-M).
#include <cstdio>
#include <cstring>

#include "../../ternary_weight_quant_b300/csrc/tw_gemv_stream.cu"
#include "../../ternary_weight_quant_b300/csrc/tw_gemm.cu"

int main() {
  char kind[16];
  int M, N, K, sms;
  while (std::scanf("%15s %d %d %d %d", kind, &M, &N, &K, &sms) == 5) {
    if (!std::strcmp(kind, "stream") || !std::strcmp(kind, "fused")) {
      Plan p;
      if (!make_plan(M, N, K, sms, p, !std::strcmp(kind, "fused"))) {
        std::printf("none\n");
        continue;
      }
      std::printf("grid %d rows_base %d rows_rem %d S %d jmax %d xs_off %d acc_off %d xf_off %d cl %d smem %zu\n",
                  p.grid, p.rows_base, p.rows_rem, p.S, p.jmax, p.xs_off, p.acc_off, p.xf_off, p.cl, p.smem);
    } else {
      GemmPlan p;
      bool ok;
      if (!std::strcmp(kind, "tok")) ok = gemm_tok_plan(M, N, K, sms, p);
      else ok = gemm_plan(M, N, K, sms, p) && (std::strcmp(kind, "tma") ? true : gemm_tma_plan(p, true));
      if (!ok) {
        std::printf("none\n");
        continue;
      }
      std::printf("BN %d nstages %d ksplit %d kstages_per_split %d tiles_n %d tiles_m %d tmem_cols %u ctrl_off %u smem %zu\n",
                  p.BN, p.nstages, p.ksplit, p.kstages_per_split, p.tiles_n, p.tiles_m, p.tmem_cols, p.ctrl_off,
                  p.smem);
    }
  }
  return 0;
}
