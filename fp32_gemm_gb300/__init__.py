"""GB300 (sm_103a) gx_gemm: the deterministic FP32 per-step d_u update of a chunked backward pass.

d_u[n, i, c] = d_u[n, i, c] + acc, acc = fmaf(x[n, j, i], d_dv[n, j, c], acc) for j = 0..C-1 from +0, for every chunk
n = ti*P + p of step ti (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula).

The compute runs in the CUDA library libsdm_gx_gemm.so (C ABI: include/sdm_gx_gemm.h); this package is its thin
ctypes binding. PyTorch provides device memory and streams only.
"""

from ._binding import (FLAG_CONFIG_MASK, FLAG_CTAS_SHIFT, FLAG_GENERIC, FLAG_NO_PREFETCH, Geom, Graph, GxGemmError, Plan,  # noqa: F401,E501
                       Strides, abi_version, device_error, geometry, kernel_attrs, launch_counts, lib, num_configs,
                       producer_step, step, step_ex, strerror)
from ._binding import (ERR_FATAL_MASK, ERR_HANDOFF_RECOMPUTED, FLAG_NOALLOC, FLAG_TEST_NO_HANDOFF, FLAG_TEST_STALL, FLAG_X_TRANSPOSED, LIB_PATH, autotune, choose_config, config_info,  # noqa: F401
                       noalloc_geometry, step_noalloc, stream_pieces, workspace_size)


def config_flag(config: int, ctas_per_sm: int = 0) -> int:
    """Flags forcing tile configuration `config` (and optionally the resident CTAs per SM)."""
    return ((int(config) + 1) & FLAG_CONFIG_MASK) | ((int(ctas_per_sm) & 0xF) << FLAG_CTAS_SHIFT)
