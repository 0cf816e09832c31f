"""ctypes binding of the C-ABI in include/rar.h (argument marshalling only).

Every function named ``rar_*`` here calls the C function of the same name in
``librar.so``; the library must have been built (``__graft_entry__.build()``
or ``python -m ring_all_reduce_rar_gb300._build``).  There is no fallback:
if the library is missing the import of the call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

DTYPE_CODES = {"int32": 0, "float32": 1, "bfloat16": 2, "float16": 3}
OP_CODES = {"sum": 0, "max": 1, "avg": 2, "avg_prediv": 3}
ENGINE_CODES = {"fused": 0, "ring": 1, "ring_bidir": 2, "fused_tree": 3, "tree": 4}
FAULT_CODES = {"none": 0, "mute": 1, "delay": 2}
FUSED_PATHS = {"auto": 0, "registers": 1, "stream": 2}
PROTOCOLS = {"auto": 0, "simple": 1, "ll": 2}
STATUS_NAMES = {0: "RAR_OK", 1: "RAR_EINVAL", 2: "RAR_EUNSUPPORTED", 3: "RAR_ENOMEM",
                4: "RAR_ECUDA", 5: "RAR_ETIMEOUT", 6: "RAR_EABORTED"}
RAR_MAX_P = 1024


class RarError(RuntimeError):
    """A non-OK status from the library; .code is the rar_status_code."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


class Options(ctypes.Structure):
    """rar_options (all zero = defaults)."""
    _fields_ = [
        ("engine", ctypes.c_int),
        ("channels", ctypes.c_int),
        ("slice_elems", ctypes.c_int),
        ("block_threads", ctypes.c_int),
        ("timeout_ns", ctypes.c_ulonglong),
        ("skip_pointer_check", ctypes.c_int),
        ("fault_mode", ctypes.c_int),
        ("fault_rank", ctypes.c_int),
        ("fault_delay_ns", ctypes.c_uint),
        ("fused_path", ctypes.c_int),
        ("hier_group", ctypes.c_int),
        ("protocol", ctypes.c_int),
        ("slice_block", ctypes.c_int),
        ("trace", ctypes.c_int),
    ]


def make_options(engine="fused", channels=0, slice_elems=0, block_threads=0, timeout_ns=0,
                 skip_pointer_check=False, fault_mode="none", fault_rank=0, fault_delay_ns=0,
                 fused_path="auto", hier_group=0, protocol="auto", slice_block=0, trace=False) -> Options:
    o = Options()
    o.engine = ENGINE_CODES[engine] if isinstance(engine, str) else int(engine)
    o.channels = channels
    o.slice_elems = slice_elems
    o.block_threads = block_threads
    o.timeout_ns = timeout_ns
    o.skip_pointer_check = 1 if skip_pointer_check else 0
    o.fault_mode = FAULT_CODES[fault_mode] if isinstance(fault_mode, str) else int(fault_mode)
    o.fault_rank = fault_rank
    o.fault_delay_ns = fault_delay_ns
    o.fused_path = FUSED_PATHS[fused_path] if isinstance(fused_path, str) else int(fused_path)
    o.hier_group = hier_group
    o.protocol = PROTOCOLS[protocol] if isinstance(protocol, str) else int(protocol)
    o.slice_block = slice_block
    o.trace = 1 if trace else 0
    return o


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load librar.so (built in-tree).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.rar_init.argtypes = [ctypes.POINTER(vp), i32, ctypes.POINTER(Options)]
        lib.rar_set_options.argtypes = [vp, ctypes.POINTER(Options)]
        for name in ("rar_allreduce", "rar_reduce_scatter"):
            getattr(lib, name).argtypes = [vp, ctypes.POINTER(vp), i32, sz, i32, i32, vp]
        lib.rar_all_gather.argtypes = [vp, ctypes.POINTER(vp), i32, sz, i32, vp]
        lib.rar_allreduce_range.argtypes = [vp, ctypes.POINTER(vp), i32, sz, sz, sz, i32, i32, vp]
        lib.rar_allreduce_host.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, sz, i32, i32, vp]
        lib.rar_allreduce_noalloc.argtypes = [ctypes.POINTER(vp), i32, sz, i32, i32, vp]
        lib.rar_status.argtypes = [vp]
        lib.rar_send_counts.argtypes = [vp, ctypes.POINTER(ctypes.c_ulonglong), i32]
        lib.rar_last_error.argtypes = [vp]
        lib.rar_last_error.restype = ctypes.c_char_p
        lib.rar_destroy.argtypes = [vp]
        lib.rar_version.argtypes = []
        lib.rar_debug_set_epoch.argtypes = [vp, ctypes.c_uint]
        u64p = ctypes.POINTER(ctypes.c_ulonglong)
        lib.rar_trace.argtypes = [vp, u64p, u64p, i32, i32, ctypes.POINTER(i32)]
        for name in ("rar_init", "rar_set_options", "rar_allreduce", "rar_reduce_scatter",
                     "rar_all_gather", "rar_allreduce_range", "rar_allreduce_host", "rar_debug_set_epoch",
                     "rar_allreduce_noalloc", "rar_status", "rar_send_counts", "rar_destroy", "rar_version",
                     "rar_trace"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def _check(handle, rc: int):
    if rc != 0:
        msg = load_library().rar_last_error(handle).decode(errors="replace")
        raise RarError(rc, msg)


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _marshal(tensors):
    """(pointer array, p, n, dtype code, device) from a list of tensors."""
    import torch
    if len(tensors) < 1:
        raise ValueError("need at least one rank buffer")
    t0 = tensors[0]
    names = {torch.int32: "int32", torch.float32: "float32", torch.bfloat16: "bfloat16",
             torch.float16: "float16"}
    if t0.dtype not in names:
        raise ValueError(f"unsupported dtype {t0.dtype}")
    for t in tensors:
        if t.dtype != t0.dtype or t.numel() != t0.numel() or t.device != t0.device:
            raise ValueError("rank buffers must share dtype, length and device")
        if not t.is_contiguous():
            raise ValueError("rank buffers must be contiguous")
        if t.device.type != "cuda":
            raise ValueError("rank buffers must be CUDA tensors")
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr, len(tensors), t0.numel(), DTYPE_CODES[names[t0.dtype]], t0.device


# ----------------------------------------------------------- same-name calls

def rar_version() -> int:
    return load_library().rar_version()


def rar_init(device: int = 0, options: Options | None = None) -> int:
    lib = load_library()
    h = ctypes.c_void_p()
    rc = lib.rar_init(ctypes.byref(h), device, ctypes.byref(options) if options is not None else None)
    _check(None, rc)
    return h.value


def rar_set_options(handle: int, options: Options) -> None:
    _check(handle, load_library().rar_set_options(handle, ctypes.byref(options)))


def rar_allreduce(handle: int, tensors, op: str = "sum", stream=None) -> None:
    arr, p, n, dt, dev = _marshal(tensors)
    _check(handle, load_library().rar_allreduce(handle, arr, p, n, dt, OP_CODES[op], _stream_ptr(stream, dev)))


def rar_reduce_scatter(handle: int, tensors, op: str = "sum", stream=None) -> None:
    arr, p, n, dt, dev = _marshal(tensors)
    _check(handle, load_library().rar_reduce_scatter(handle, arr, p, n, dt, OP_CODES[op],
                                                       _stream_ptr(stream, dev)))


def rar_all_gather(handle: int, tensors, stream=None) -> None:
    arr, p, n, dt, dev = _marshal(tensors)
    _check(handle, load_library().rar_all_gather(handle, arr, p, n, dt, _stream_ptr(stream, dev)))


def rar_allreduce_range(handle: int, tensors, n_total: int, lo: int, op: str = "sum", stream=None) -> None:
    """All-reduce of indices [lo, lo + numel) of rank buffers of n_total
    elements (see rar_allreduce_range in rar.h): `tensors` are the pieces,
    element 0 of each being global index lo."""
    arr, p, n, dt, dev = _marshal(tensors)
    _check(handle, load_library().rar_allreduce_range(handle, arr, p, n_total, lo, lo + n, dt, OP_CODES[op],
                                                        _stream_ptr(stream, dev)))


def rar_allreduce_host(handle: int, host_tensors, dev_tensors=None, op: str = "sum", stream=None) -> None:
    """All-reduce host-resident buffers (see rar_allreduce_host in rar.h):
    pinned host tensors are reduced in place by the GPU over the host link;
    pageable ones are staged through dev_tensors."""
    import torch
    names = {torch.int32: "int32", torch.float32: "float32", torch.bfloat16: "bfloat16", torch.float16: "float16"}
    p = len(host_tensors)
    if p < 1:
        raise ValueError("need at least one rank buffer")
    t0 = host_tensors[0]
    if t0.dtype not in names:
        raise ValueError(f"unsupported dtype {t0.dtype}")
    for t in host_tensors:
        if t.device.type != "cpu" or not t.is_contiguous() or t.numel() != t0.numel() or t.dtype != t0.dtype:
            raise ValueError("host buffers must be contiguous CPU tensors of one dtype and length")
    harr = (ctypes.c_void_p * p)(*[t.data_ptr() for t in host_tensors])
    if dev_tensors is not None:
        darr, dp, dn, dt, dev = _marshal(dev_tensors)
        if dp != p or dn != t0.numel() or dev_tensors[0].dtype != t0.dtype:
            raise ValueError("device staging buffers must match the host buffers")
    else:
        darr, dev = None, torch.device("cuda", torch.cuda.current_device())
    _check(handle, load_library().rar_allreduce_host(handle, harr, darr, p, t0.numel(), DTYPE_CODES[names[t0.dtype]],
                                                       OP_CODES[op], _stream_ptr(stream, dev)))


def rar_allreduce_noalloc(tensors, op: str = "sum", stream=None) -> None:
    """Handle-free ring all-reduce that allocates no device memory (see
    rar_allreduce_noalloc in rar.h); tensors on the current device."""
    arr, p, n, dt, dev = _marshal(tensors)
    _check(None, load_library().rar_allreduce_noalloc(arr, p, n, dt, OP_CODES[op], _stream_ptr(stream, dev)))


def rar_allreduce_ptrs(handle: int, ptrs, n: int, dtype: str, op: str = "sum", stream: int = 0) -> int:
    """Raw form: device pointers as ints; returns the status code (no raise)."""
    arr = (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)
    return load_library().rar_allreduce(handle, arr, len(ptrs), n, DTYPE_CODES[dtype], OP_CODES[op], stream)


def rar_status(handle: int) -> int:
    """Device-side status of the last call (waits for it); does not raise."""
    return load_library().rar_status(handle)


def rar_send_counts(handle: int, p: int) -> list[int]:
    out = (ctypes.c_ulonglong * p)()
    _check(handle, load_library().rar_send_counts(handle, out, p))
    return list(out)


def rar_trace(handle: int, p: int) -> tuple[list[list[int]], list[list[int]]]:
    """Per-rank step times of the last traced call (see rar_trace in
    rar.h): (work_ns, wait_ns), each p lists of one entry per schedule step."""
    max_steps = 2046
    work = (ctypes.c_ulonglong * (p * max_steps))()
    wait = (ctypes.c_ulonglong * (p * max_steps))()
    steps = ctypes.c_int()
    _check(handle, load_library().rar_trace(handle, work, wait, p, max_steps, ctypes.byref(steps)))
    s = steps.value
    return ([list(work[r * max_steps:r * max_steps + s]) for r in range(p)],
            [list(wait[r * max_steps:r * max_steps + s]) for r in range(p)])


def rar_last_error(handle: int | None) -> str:
    return load_library().rar_last_error(handle).decode(errors="replace")


def rar_debug_set_epoch(handle: int, epoch: int) -> None:
    """Test hook (see rar_debug_set_epoch in rar.h)."""
    _check(handle, load_library().rar_debug_set_epoch(handle, epoch))


def rar_destroy(handle: int) -> None:
    load_library().rar_destroy(handle)


class Handle:
    """A library handle with its options; usable as a context manager.

        with Handle(device=0, engine="ring") as h:
            h.allreduce(list_of_tensors, op="sum")
            h.check()
    """

    def __init__(self, device: int = 0, **opts):
        self.device = device
        self.options = make_options(**opts)
        self.h = rar_init(device, self.options)

    def set_options(self, **opts):
        options = make_options(**opts)
        rar_set_options(self.h, options)  # raises, keeping the old options, if refused
        self.options = options

    def allreduce(self, tensors, op="sum", stream=None):
        rar_allreduce(self.h, tensors, op, stream)

    def allreduce_range(self, tensors, n_total, lo, op="sum", stream=None):
        rar_allreduce_range(self.h, tensors, n_total, lo, op, stream)

    def allreduce_host(self, host_tensors, dev_tensors=None, op="sum", stream=None):
        rar_allreduce_host(self.h, host_tensors, dev_tensors, op, stream)

    def reduce_scatter(self, tensors, op="sum", stream=None):
        rar_reduce_scatter(self.h, tensors, op, stream)

    def all_gather(self, tensors, stream=None):
        rar_all_gather(self.h, tensors, stream)

    def status(self) -> int:
        return rar_status(self.h)

    def check(self):
        rc = rar_status(self.h)
        _check(self.h, rc)

    def send_counts(self, p: int) -> list[int]:
        return rar_send_counts(self.h, p)

    def trace(self, p: int):
        return rar_trace(self.h, p)

    def close(self):
        if self.h:
            rar_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
