"""GB300 TN GEMM library (placeholder until the binding lands)."""
