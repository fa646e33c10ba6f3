"""GB300-native tiled dense GEMM, C = A x B^T (placeholder; the binding lands with the C ABI)."""
