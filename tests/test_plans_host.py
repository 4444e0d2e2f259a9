"""Launch planning of the streaming GEMV and the GEMMs, checked on the host.

The library's own planning code (compiled here for the host with nvcc; nothing is launched)
is swept over the benchmark's shapes and edge cases, and every plan it accepts must be a
launch the hardware and the kernels take: shared memory within the per-CTA limit, row
blocks that cover N exactly, K slices that cover K, cluster sizes of at most 8 CTAs that
fit the SM count, tensor-memory columns a power of two that holds the tile.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_progs", "plan_check.cu")
SMEM_LIMIT = 227 * 1024          # dynamic shared memory per CTA on this part
SMS = (148, 132)


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("plans") / "plan_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), SRC, "-o", out, "-lcuda"],
                   check=True, capture_output=True)
    return out


def plans(prog, queries):
    text = "".join(f"{k} {M} {N} {K} {s}\n" for k, M, N, K, s in queries)
    out = subprocess.run([prog], input=text, capture_output=True, text=True, check=True).stdout.splitlines()
    assert len(out) == len(queries)
    res = []
    for line in out:
        if line.strip() == "none":
            res.append(None)
        else:
            f = line.split()
            res.append({f[i]: int(f[i + 1]) for i in range(0, len(f), 2)})
    return res


NS = [1, 7, 37, 100, 149, 256, 640, 2560, 3840, 6144, 10240, 13824, 20000, 28672, 57344, 300000]
KS = [64, 128, 256, 2560, 4096, 6912, 8192, 14336, 28672, 65472]


def test_stream_plans(prog):
    q = [(kind, M, N, K, s) for kind in ("stream", "fused") for M in (1, 2, 3, 4, 5) for N in NS for K in KS + [80]
         for s in SMS]
    for (kind, M, N, K, s), p in zip(q, plans(prog, q)):
        if M > 4 or K % 64:
            assert p is None, (kind, M, N, K)
            continue
        if p is None:
            continue  # a shape the streaming kernel declines goes to the dp4a kernel
        MT = 1 if M == 1 else 2 if M == 2 else 4
        Kw = K // 16
        cap = {1: 6, 2: 3, 4: 2}[MT]
        assert 1 <= p["grid"] <= min(N, 2 * s), (kind, M, N, K, p)
        assert p["rows_base"] * p["grid"] + p["rows_rem"] == N and 0 <= p["rows_rem"] < p["grid"]
        assert p["S"] in (1, 2, 3, 4, 6, 12) and 1 <= p["jmax"] <= cap
        assert p["S"] * 32 * p["jmax"] >= Kw  # the K slices cover K
        assert p["acc_off"] == MT * Kw * 16   # byte-transposed x_q of MT tokens
        rows = p["rows_base"] + (1 if p["rows_rem"] else 0)
        sacc_end = p["acc_off"] + (rows * MT * 4 + 15) // 16 * 16
        # the fused prologue (here with RMSNorm) is shared by clusters of 4 CTAs from K = 8192;
        # clusters never stage x
        cl = p["cl"]
        if kind == "stream" or K < 8192 or p["grid"] < 2:
            assert cl == 1
        else:
            assert cl == 4, (kind, M, N, K, s, p)
        if p["xf_off"] >= 0:
            assert kind == "fused" and cl == 1 and (MT + 1) * K * 4 <= 64 * 1024 and p["xf_off"] == sacc_end
            assert p["smem"] == sacc_end + (MT + 1) * K * 4
        else:
            assert p["smem"] == sacc_end
        assert p["smem"] <= 160 * 1024


def test_tokens_on_m_plans(prog):
    q = [("tok", M, N, K, s) for M in (1, 8, 17, 64, 100, 128, 129) for N in NS for K in KS + [80, 2576]
         for s in SMS]
    for (_, M, N, K, s), p in zip(q, plans(prog, q)):
        if M > 128 or K % 64:
            assert p is None, (M, N, K)
            continue
        assert p is not None, (M, N, K)
        assert p["smem"] <= SMEM_LIMIT
        assert p["tiles_n"] == (N + 255) // 256 and p["tiles_m"] == 1
        assert p["ksplit"] in (1, 2, 4, 8)
        if p["ksplit"] > 1:
            assert p["tiles_n"] * p["ksplit"] <= s
        assert p["ksplit"] * p["kstages_per_split"] >= K // 64 >= (p["ksplit"] - 1) * p["kstages_per_split"]
        assert p["tmem_cols"] == 256
        assert p["ctrl_off"] >= 128 * 260 * 4  # the staged split-K partials fit below the barriers


@pytest.mark.parametrize("kind", ["gemm", "tma"])
def test_weight_tile_plans(prog, kind):
    q = [(kind, M, N, K, s) for M in (1, 16, 17, 100, 200, 256, 257, 1000) for N in NS for K in (16, 80, 2560, 6912, 65520)
         for s in SMS]
    for (_, M, N, K, s), p in zip(q, plans(prog, q)):
        if p is None:
            continue
        assert p["smem"] <= SMEM_LIMIT
        assert p["BN"] % 16 == 0 and 16 <= p["BN"] <= 256 and (p["BN"] >= M or p["BN"] == 256)
        assert p["tiles_m"] == (M + p["BN"] - 1) // p["BN"] and p["tiles_n"] == (N + 127) // 128
        assert p["ksplit"] in (1, 2, 4, 8) and p["nstages"] >= 2
        if p["ksplit"] > 1:
            assert p["tiles_n"] * p["tiles_m"] * p["ksplit"] <= s
        nkst = (K + 63) // 64
        assert p["ksplit"] * p["kstages_per_split"] >= nkst
        t = p["tmem_cols"]
        assert t & (t - 1) == 0 and p["BN"] <= t <= 512
