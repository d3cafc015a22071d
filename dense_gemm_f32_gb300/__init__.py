"""GB300-native dense GEMM: C = A x B, row-major, on sm_103a."""
