"""Shapes, byte accounting and seeded synthetic inputs shared by the CUDA
decode path and the CPU oracle.  Holds none of the decode arithmetic."""
from .configs import (  # noqa: F401
    FORMAT_BF16, FORMAT_INT4, FORMAT_INT8, FORMAT_CODE, FORMATS, INT4_GROUP,
    ModelConfig, Workload, WORKLOADS, workload, matrix_bytes, weight_bytes_per_token,
    kv_bytes_per_position, kv_read_bytes, step_bytes, step_flops, mean_step_bytes,
    with_format, TINY, LLAMA_1B, LLAMA_8B_BF16, LLAMA_8B_INT8, LLAMA_8B_INT4,
)
