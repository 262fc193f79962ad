"""GB300-native exact DeBERTa-v2/v3 disentangled self-attention.

The compute lives in ``libdfattn.so`` (C ABI in ``include/df_attn.h``,
tcgen05/TMA kernels for bf16/fp16 and CUDA-core kernels for strict fp32);
this package holds its build script, a ctypes binding and the seeded input
recipes of the workloads.
"""
from .binding import (Geometry, DfError, attn_bwd, attn_fwd, device_error, load, rel_index_table,  # noqa: F401
                      step_host, step_host_arena_size, workspace_size)

__version__ = "0.1.0"
