"""GB300-native FP8 quantization and scaled FP8 GEMM (sm_103a CUDA kernels behind a C ABI).

The compute path is libfp8bs.so (built from csrc/ by build.py); ``binding``
marshals torch tensors into its C entry points. ``synth`` draws the seeded
synthetic inputs the tests and the bench share.
"""
from .binding import (BLOCK_128x128, E4M3, E5M2, MX32, SF_LINEAR, SF_TCGEN05, TENSOR, TILE_1x128, TOKEN,  # noqa: F401
                      Fp8Error, dequantize, gemm_blockscaled, gemm_mx, quantize)
