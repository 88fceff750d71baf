// Grouped GEMM for prefill (filled in with the tcgen05 kernel).
