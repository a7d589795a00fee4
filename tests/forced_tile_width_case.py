"""Child process of test_gpu_forced_tile_width.py: GEMM parity against the
oracle with the tile width forced by FP8FG_BN (read once per process, so the
parent sets it in this process's environment).

The shapes are chosen for 192-column tiles: a tile starting in the middle of
a 128-column scale block (n0 = 192, 576), a last tile whose second block
lies past N (N = 584: zero-filled block scale), one inside N (N = 712), and
more tiles than SMs (5120 x 584: 160 tiles), in the dense, grouped-
contiguous and grouped-masked layouts, BF16 and FP32 output.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import fp8_fine_grained_24_b300 as fg  # noqa: E402
import test_gpu_gemm as t  # noqa: E402


def main():
    bn = os.environ.get("FP8FG_BN", "")
    t._dense_case(fg, 300, 584, 640, seed=701)
    t._dense_case(fg, 256, 712, 384, seed=702)
    t._dense_case(fg, 5120, 584, 512, seed=703)
    t._dense_case(fg, 200, 584, 384, seed=704, out_dtype=torch.float32)
    t.test_dense_fp32_out_and_accumulate(fg)
    t._contig_case(fg, np.array([130, 0, 61, 256, 1]), 584, 384, 705)
    t._masked_case(fg, 4, 256, 584, 384, np.array([0, 256, 17, 129], np.int32), 706)
    # the launched kernel is the forced width's
    qa, sa = fg.fp8_quant_1x128(torch.randn(512, 512, device="cuda", dtype=torch.bfloat16))
    qb, sb = fg.fp8_quant_128x128(torch.randn(584, 512, device="cuda", dtype=torch.bfloat16))
    with torch.profiler.profile(activities=[torch.profiler.ProfilerActivity.CUDA]) as prof:
        fg.fp8_gemm_dense(qa, sa, qb, sb)
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if "fp8_gemm_kernel" in e.name]
    assert names and all(f"fp8_gemm_kernel<{bn}," in n for n in names), names
    print(f"tile width {bn}: ok")


if __name__ == "__main__":
    main()
