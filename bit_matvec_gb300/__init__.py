"""Ternary pq2_0 x q8_K matrix product on GB300 (sm_103a).

The computation lives in libtq.so (C ABI in include/tq.h, CUDA kernels in
csrc/); this package is its Python binding, with the same function names.
"""
from .binding import (  # noqa: F401
    GROUP,
    PQ2_0_BYTES,
    Q8K_BYTES,
    QK_K,
    TILE_BYTES,
    TILE_ROWS,
    TQ_ERR_ALIAS,
    TQ_ERR_ALIGN,
    TQ_ERR_CUDA,
    TQ_ERR_NULL,
    TQ_ERR_SHAPE,
    TQ_ERR_TIMEOUT,
    TQ_OK,
    TQError,
    header_functions,
    library,
    q8K_empty,
    q8K_nbytes,
    repacked_empty,
    tq_device_status,
    tq_last_cuda_error,
    tq_matmul,
    tq_matmul_groupsums,
    tq_quantize_q8K,
    tq_repack,
    tq_repacked_bytes,
    tq_strerror,
    tq_unrepack,
    tq_version,
)
