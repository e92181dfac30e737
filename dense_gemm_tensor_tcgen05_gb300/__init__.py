"""GB300-native dense GEMM (placeholder; binding follows)."""
