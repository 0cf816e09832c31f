"""rar_allreduce_noalloc: the all-reduce for callers that may not allocate
device memory (their memory belongs to another allocator, or they cannot
pay for cudaMalloc at call time).  Called through the C-ABI, its results
must equal the handle-based rar_allreduce bit for bit -- the tolerance every
ring-order test here uses -- on two calls in a row, since every call reuses
the same fixed scratch array.

This file is collected last on purpose, so that a run that stops at the
first failure has already run every other test; it also passes on its own in
a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as w

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import ring_all_reduce_rar_gb300 as rar
    rar.build()
    assert torch.cuda.is_available()
    return rar.load_library()


NAMES = {torch.float32: "float32", torch.bfloat16: "bfloat16", torch.int32: "int32", torch.float16: "float16"}


def _rows(host, dev):
    big, rows = w.alloc_ranks(len(host), host[0].numel(), NAMES[host[0].dtype], dev)
    for r, t in enumerate(host):
        rows[r].copy_(t)
    return big, rows


def _bits(t):
    return w.to_storage_numpy(t).view(np.uint8)


@pytest.mark.parametrize("p,n,dtype,op,dist", [
    (8, 8 * 100003 + 5, "bfloat16", "sum", ("normal", 1e-2)),
    (4, 4099, "float32", "avg", ("uniform", -1.0, 1.0)),
    (16, 16 * 4096, "int32", "sum", ("uniform_int", -(1 << 20), 21)),
])
def test_noalloc_matches_allreduce_on_two_calls(lib, p, n, dtype, op, dist):
    import ring_all_reduce_rar_gb300 as rar
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    _, host = w.make_inputs(p, n, dtype, dist, 4242 + p)
    # the existing entry point (handle-based ring executor)
    _, ref = _rows(host, dev)
    with rar.Handle(0, engine="ring") as h:
        h.allreduce(ref, op=op)
        h.check()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        _, rows = _rows(host, dev)
        arr = (ctypes.c_void_p * p)(*[t.data_ptr() for t in rows])
        rc = lib.rar_allreduce_noalloc(arr, p, n, rar.DTYPE_CODES[dtype], rar.OP_CODES[op], stream)
        assert rc == 0, lib.rar_last_error(None)
        torch.cuda.synchronize()
        for r in range(p):
            assert np.array_equal(_bits(rows[r]), _bits(ref[r])), f"call {call}, rank {r}"


def test_noalloc_rejects_p_above_its_limit(lib):
    dev = torch.device("cuda:0")
    p, n = 65, 100
    big = torch.zeros(p, 128, device=dev)
    arr = (ctypes.c_void_p * p)(*[big[r].data_ptr() for r in range(p)])
    rc = lib.rar_allreduce_noalloc(arr, p, n, 1, 0, None)
    assert rc == 1  # RAR_EINVAL
    assert b"p must be in [1, 64]" in lib.rar_last_error(None)
