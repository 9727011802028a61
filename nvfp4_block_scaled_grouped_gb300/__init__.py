"""NVFP4 block-scaled grouped GEMM for GB300 (sm_103a)."""
