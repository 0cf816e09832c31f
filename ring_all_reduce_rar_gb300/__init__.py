"""Ring all-reduce over p virtual ranks held in one GB300's HBM.

A thin Python binding over the C-ABI library ``librar.so`` (include/rar.h);
all work runs in that library's CUDA kernels.  PyTorch is only used to hand
over device pointers and streams.

    import ring_all_reduce_rar_gb300 as rar
    with rar.Handle(device=0, engine="fused") as h:
        h.allreduce(tensors, op="sum")     # tensors: p CUDA tensors of n elements
"""
from ._abi import (DTYPE_CODES, ENGINE_CODES, FAULT_CODES, OP_CODES, RAR_MAX_P, STATUS_NAMES, Handle, Options,
                   RarError, library_path, load_library, make_options, rar_all_gather, rar_allreduce,
                   rar_allreduce_host, rar_allreduce_noalloc, rar_allreduce_ptrs, rar_allreduce_range, rar_debug_set_epoch,
                   rar_destroy,
                   rar_init, rar_last_error, rar_reduce_scatter, rar_send_counts, rar_set_options, rar_status,
                   rar_trace, rar_version)
from ._build import build

__all__ = [
    "DTYPE_CODES", "ENGINE_CODES", "FAULT_CODES", "OP_CODES", "RAR_MAX_P", "STATUS_NAMES", "Handle", "Options",
    "RarError", "build", "library_path", "load_library", "make_options", "rar_all_gather", "rar_allreduce",
    "rar_allreduce_host", "rar_allreduce_noalloc", "rar_allreduce_ptrs", "rar_allreduce_range", "rar_debug_set_epoch",
    "rar_destroy",
    "rar_init", "rar_last_error", "rar_reduce_scatter", "rar_send_counts", "rar_set_options", "rar_status",
    "rar_trace", "rar_version",
]
