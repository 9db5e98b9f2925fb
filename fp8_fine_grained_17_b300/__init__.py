"""Fine-grained FP8 (1x128 / 128x128 block-scaled) GEMM library for B300."""
