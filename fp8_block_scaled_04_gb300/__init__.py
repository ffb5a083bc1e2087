"""GB300-native FP8 quantization and scaled FP8 GEMM (sm_103a CUDA kernels behind a C ABI)."""
