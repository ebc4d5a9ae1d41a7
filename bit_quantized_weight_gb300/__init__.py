"""bit_quantized_weight_gb300 -- decode-step quantised GEMV on NVIDIA GB300.

A thin Python binding over the C-ABI library libqgemv.so (include/qgemv.h).
Every computation runs in the library's CUDA kernels; this module only checks
tensor shapes, passes device pointers and the current CUDA stream, and turns a
non-zero status into an exception. PyTorch supplies memory and streams.
"""
from .qgemv import (  # noqa: F401
    QG_OK, QG_ERR_INVALID_ARG, QG_ERR_UNSUPPORTED, QG_ERR_MISALIGNED, QG_ERR_WORKSPACE,
    QG_ERR_CUDA, QG_ERR_DEVICE_TIMEOUT, QGemvError, lib, lib_path,
    qgemv_nvfp4, qgemv_q45, qgemv_swiglu_nvfp4, moe_route_topk, moe_qgemv_nvfp4, moe_qgemv_nvfp4_noalloc,
    moe_qgemv_nvfp4_workspace_size, qdequant_nvfp4, qdequant_q45, qg_last_device_status,
    qg_status_string, qg_debug_set_wait, read_probe, GemvChain, qgemv_chain, QgGemvOp, qgemv_swiglu_q45,
    QG_FMT_NVFP4, QG_FMT_Q4, QG_FMT_Q5, QG_EPI_NONE, QG_EPI_RESIDUAL, QG_EPI_SWIGLU,
)
