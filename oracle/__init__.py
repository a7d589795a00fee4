"""CPU oracle for the fine-grained FP8 GEMM path.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it. It shares no code,
header, table or constant generator with the CUDA library.

It is written for clarity, not speed: NumPy in float32 where the method
fixes float32 arithmetic (the scale ``amax/448`` and the quotient ``x/s``),
float64 for the GEMM reference, and exact rationals in the pins.

Sources (page titles as extracted):

* "DeepSeek-V3" report excerpt (page 1): fine-grained quantization with 1x128
  activation tiles, FP8 activations cached for backward and retiled from 1x128
  to 128x1, FP8 GEMMs taking FP8 inputs and producing BF16 or FP32, promotion
  of partial sums to FP32 on CUDA cores; limited (about 14-bit) accumulation on
  H800 with a relative error near 2% at K=4096.
* same report excerpt (page 2): fixed-point accumulation with sign-fill right
  shift and truncation; power-of-2 scaling factors for selected activations
  and activation gradients; decode batches of at most 256 tokens per expert.
* "DeepGEMM" article (page 4): dense and two MoE layouts; FP8 formats E4M3 and
  E5M2; Table 1 shapes.

Modules:

* :mod:`oracle.e4m3`   -- E4M3 codec from the OCP FP8 definition.
* :mod:`oracle.quant`  -- 1x128, 128x128 and 1x128->128x1 quantizers.
* :mod:`oracle.gemm`   -- FP64 reference products of dequantized operands for
  the dense, grouped-contiguous and grouped-masked layouts and Wgrad.
* :mod:`oracle.accum`  -- emulator of limited-precision fixed-point
  accumulation with optional FP32 promotion.
* :mod:`oracle.bf16`   -- round-to-nearest-even to BF16 for output comparison.
"""
from . import e4m3, quant, gemm, accum, bf16  # noqa: F401
