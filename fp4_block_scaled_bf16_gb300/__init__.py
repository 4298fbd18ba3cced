"""UE5M3-scaled FP4 quantisation and block-scaled GEMM for GB300 (sm_103a).

The compute path is the C-ABI library libfp4q.so (CUDA kernels); the Python
binding in :mod:`fp4_block_scaled_bf16_gb300.fp4q` marshals torch tensors and
streams to it.  Importing this package does not load the library, so that the
seeded input generators (:mod:`.workloads`) are usable without a GPU.
"""
__all__ = ["fp4q", "workloads"]
