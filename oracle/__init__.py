"""Plain, slow CPU oracle for the ring all-reduce -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (``bench.py --impl reference`` and its ``cpu_baseline`` object) may import
this package.  The product path (``ring_all_reduce_rar_gb300``) never does,
and the two share no code: this wrapper loads ``rar_oracle.c`` (plain C,
compiled here with gcc) through ctypes.

The C file restates the pages' method:
  * "Ring All-Reduce, in depth" -- "The schedule" (reduce-scatter and
    all-gather step rules, ownership of chunk (r + 1) mod p), "An
    implementation" (chunk_bounds, the snapshot-then-apply simulator),
    "What real libraries add" / "Bidirectional rings" (the mirrored ring).
  * "AllReduce 与 Ring 通信算法详解" -- "AllReduce 语义" (sum / avg / max).
  * "Derive the cost of a ring all-reduce" -- last probe (reduction in the
    buffer's dtype).

Parity pins (tests/test_oracle_*.py) tie it to the pages' worked examples,
to brute-force sums, to exact rational rounding and to closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rar_oracle.c")
_HDR = os.path.join(_HERE, "rar_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "librar_oracle.so")

DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2, "float16": 3}
OPS = {"sum": 0, "max": 1, "avg": 2, "avg_prediv": 3}
MODES = {"ring": 0, "bidir": 1, "tree": 2}
_STORAGE = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16, "float16": np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile rar_oracle.c into a shared library (gcc, plain C11).

    IEEE behaviour is kept: no fast-math, no FMA contraction, no FTZ."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH):
        newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if os.path.getmtime(_LIB_PATH) >= newest:
            return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-fno-strict-aliasing", "-Wall", "-Wextra",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.orc_chunk_bounds.argtypes = [i64, i32, ctypes.POINTER(i64)]
        lib.orc_chunk_bounds.restype = None
        lib.orc_elem_size.argtypes = [i32]
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f32.restype = ctypes.c_float
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f32.restype = ctypes.c_float
        lib.orc_combine.argtypes = [i32, i32, vp, vp, vp]
        lib.orc_combine.restype = None
        lib.orc_ring_simulate.argtypes = [ctypes.POINTER(vp), i32, i64, i32, i32, i32, i32, i32,
                                          ctypes.POINTER(i64)]
        lib.orc_ring_simulate_bidir.argtypes = [ctypes.POINTER(vp), i32, i64, i32, i32, i32,
                                                ctypes.POINTER(i64)]
        lib.orc_fold_sampled.argtypes = [vp, ctypes.POINTER(i64), i64, i32, i64, i32, i32, i32, vp]
        lib.orc_tree_fold.argtypes = [ctypes.POINTER(vp), i32, i64, i32, i32]
        lib.orc_hier_simulate.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i32, i32,
                                          ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.orc_hier_fold_sampled.argtypes = [vp, ctypes.POINTER(i64), i64, i32, i32, i64, i32, i32, vp]
        lib.orc_f64_sum.argtypes = [ctypes.POINTER(vp), i32, i64, i32,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        _lib = lib
        return lib


def _check_bufs(bufs, dtype):
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    st = _STORAGE[dtype]
    n = None
    for b in bufs:
        if not isinstance(b, np.ndarray) or b.ndim != 1 or not b.flags.c_contiguous:
            raise ValueError("oracle buffers must be 1-D contiguous numpy arrays")
        if b.dtype != st and not (dtype == "float16" and b.dtype == np.float16):
            raise ValueError(f"{dtype} buffers are stored as {np.dtype(st).name}, got {b.dtype}")
        if n is None:
            n = b.shape[0]
        elif b.shape[0] != n:
            raise ValueError("all rank buffers must have the same length")
    return 0 if n is None else n


def _ptr_array(bufs):
    arr = (ctypes.c_void_p * max(1, len(bufs)))()
    for r, b in enumerate(bufs):
        arr[r] = b.ctypes.data
    return arr


def chunk_bounds(n: int, p: int) -> list[tuple[int, int]]:
    """chunk_bounds(n, p) as [(start, end)] * p."""
    lib = _load()
    starts = (ctypes.c_int64 * (p + 1))()
    lib.orc_chunk_bounds(n, p, starts)
    return [(starts[i], starts[i + 1]) for i in range(p)]


def simulate(bufs, dtype: str, op: str = "sum", direction: str = "forward",
             first_step: int = 0, n_steps: int | None = None) -> np.ndarray:
    """Run schedule steps [first_step, first_step + n_steps) in place.

    Steps 0..p-2 are reduce-scatter, p-1..2p-3 all-gather.  Returns the
    per-rank count of elements sent (int64[p])."""
    lib = _load()
    n = _check_bufs(bufs, dtype)
    p = len(bufs)
    if n_steps is None:
        n_steps = 2 * (p - 1) - first_step
    sends = (ctypes.c_int64 * max(1, p))()
    d = {"forward": 0, "mirrored": 1}[direction]
    rc = lib.orc_ring_simulate(_ptr_array(bufs), p, n, DTYPES[dtype], OPS[op], d,
                               first_step, n_steps, sends)
    if rc != 0:
        raise ValueError("orc_ring_simulate rejected its arguments")
    return np.array(sends[:p], dtype=np.int64)


def simulate_bidir(bufs, dtype: str, op: str = "sum", rs_only: bool = False) -> np.ndarray:
    """Bidirectional half-data ring, in place; returns per-rank sends."""
    lib = _load()
    n = _check_bufs(bufs, dtype)
    p = len(bufs)
    sends = (ctypes.c_int64 * max(1, p))()
    rc = lib.orc_ring_simulate_bidir(_ptr_array(bufs), p, n, DTYPES[dtype], OPS[op],
                                     1 if rs_only else 0, sends)
    if rc != 0:
        raise ValueError("orc_ring_simulate_bidir rejected its arguments")
    return np.array(sends[:p], dtype=np.int64)


def fold_sampled(vals: np.ndarray, idx: np.ndarray, n: int, dtype: str, op: str = "sum",
                 mode: str = "ring") -> np.ndarray:
    """All-reduced value at sampled indices.

    vals: (p, m) array of rank inputs at idx (storage dtype as the buffers)."""
    lib = _load()
    vals = np.ascontiguousarray(vals)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    p, m = vals.shape
    if idx.shape != (m,):
        raise ValueError("idx must have one entry per sampled column")
    out = np.empty(m, dtype=vals.dtype)
    rc = lib.orc_fold_sampled(vals.ctypes.data, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                              m, p, n, DTYPES[dtype], OPS[op], MODES[mode], out.ctypes.data)
    if rc != 0:
        raise ValueError("orc_fold_sampled rejected its arguments")
    return out


def hier_simulate(bufs, g: int, dtype: str, op: str = "sum"):
    """Hierarchical 2D all-reduce with nodes of g ranks, in place; returns
    (intra-node sends, cross-node sends) per rank."""
    lib = _load()
    n = _check_bufs(bufs, dtype)
    p = len(bufs)
    si = (ctypes.c_int64 * max(1, p))()
    sx = (ctypes.c_int64 * max(1, p))()
    rc = lib.orc_hier_simulate(_ptr_array(bufs), p, g, n, DTYPES[dtype], OPS[op], si, sx)
    if rc != 0:
        raise ValueError("orc_hier_simulate rejected its arguments")
    return np.array(si[:p], dtype=np.int64), np.array(sx[:p], dtype=np.int64)


def hier_fold_sampled(vals: np.ndarray, idx: np.ndarray, n: int, g: int, dtype: str, op: str = "sum"):
    """Hierarchical all-reduced value at sampled indices (vals: (p, m))."""
    lib = _load()
    vals = np.ascontiguousarray(vals)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    p, m = vals.shape
    out = np.empty(m, dtype=vals.dtype)
    rc = lib.orc_hier_fold_sampled(vals.ctypes.data, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), m, p, g,
                                   n, DTYPES[dtype], OPS[op], out.ctypes.data)
    if rc != 0:
        raise ValueError("orc_hier_fold_sampled rejected its arguments")
    return out


def tree_fold(bufs, dtype: str, op: str = "sum") -> None:
    """Tree-order fold over the rank index, in place on every rank."""
    lib = _load()
    n = _check_bufs(bufs, dtype)
    rc = lib.orc_tree_fold(_ptr_array(bufs), len(bufs), n, DTYPES[dtype], OPS[op])
    if rc != 0:
        raise ValueError("orc_tree_fold rejected its arguments")


def f64_sum(bufs, dtype: str):
    """(sum, sum of magnitudes) per element in float64."""
    lib = _load()
    n = _check_bufs(bufs, dtype)
    ref = np.empty(n, dtype=np.float64)
    mag = np.empty(n, dtype=np.float64)
    rc = lib.orc_f64_sum(_ptr_array(bufs), len(bufs), n, DTYPES[dtype],
                         ref.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         mag.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("orc_f64_sum rejected its arguments")
    return ref, mag


def combine(dtype: str, op: str, acc, own):
    """One hop on single elements given in storage form; returns storage form."""
    lib = _load()
    st = _STORAGE[dtype]
    a = np.array([acc], dtype=st)
    b = np.array([own], dtype=st)
    out = np.zeros(1, dtype=st)
    lib.orc_combine(DTYPES[dtype], OPS[op], a.ctypes.data, b.ctypes.data, out.ctypes.data)
    return out[0]


def f32_to_bf16(x: float) -> int:
    return int(_load().orc_f32_to_bf16(ctypes.c_float(x)))


def bf16_to_f32(h: int) -> float:
    return float(_load().orc_bf16_to_f32(ctypes.c_uint16(h)))


def f32_to_f16(x: float) -> int:
    return int(_load().orc_f32_to_f16(ctypes.c_float(x)))


def f16_to_f32(h: int) -> float:
    return float(_load().orc_f16_to_f32(ctypes.c_uint16(h)))
