"""The bench's byte and FLOP models, pinned to the DeepGEMM article's Table 1 (CPU only).

Table 1 prints TFLOPS and GB/s for three dense shapes; its GB/s equals the
bytes of FP8 A and B plus BF16 C over the time the TFLOPS figure implies.
"""
import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "deepgemm_table1.txt")


def _rows():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            M, N, K, tf, gbs = line.split()
            yield int(M), int(N), int(K), float(tf), float(gbs)


def test_table1_byte_model_reproduces_printed_bandwidth():
    rows = list(_rows())
    assert len(rows) == 3
    for M, N, K, tf, gbs in rows:
        assert abs(bench.table1_gbs(M, N, K, tf) - gbs) / gbs < 0.005


def test_algorithmic_bytes_add_scales_to_table1_model():
    M, N, K = 4096, 4096, 7168
    base = M * K + N * K + 2 * M * N
    scales = M * (K // 128) * 4 + (N // 128) * (K // 128) * 4
    assert bench.gemm_bytes(M, N, K) == base + scales
    assert bench.gemm_flops(M, N, K) == 2 * M * N * K
    assert bench.quant_1x128_bytes(M, K) == M * K * 3 + M * (K // 128) * 4
