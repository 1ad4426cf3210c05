"""GB300-native ragged-M grouped GEMM (placeholder; the binding follows)."""
