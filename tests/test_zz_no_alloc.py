"""rar_allreduce_noalloc: the all-reduce for callers that may not allocate
device memory (their memory belongs to another allocator, or they cannot
pay for cudaMalloc at call time).  Called through the C-ABI, its results
must equal the oracle's schedule simulation bit for bit -- the tolerance
every ring-order test here uses -- and the handle-based rar_allreduce, on
two calls in a row, since every call reuses the same fixed scratch array.
Calls with different p in a row (64, then 4, then 16) reuse progress words
left by another channel layout; p = 64 is the documented limit, where
p * channels meets the 1024-CTA cap of the array.

This file is collected last on purpose, so that a run that stops at the
first failure has already run every other test; it also passes on its own in
a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import ring_all_reduce_rar_gb300 as rar
    rar.build()
    assert torch.cuda.is_available()
    return rar.load_library()


NAMES = {torch.float32: "float32", torch.bfloat16: "bfloat16", torch.int32: "int32", torch.float16: "float16"}


def _rows(host, dev, offset=0):
    """Upload host rows into one padded allocation; `offset` elements into
    each row (offset 1 breaks 16-byte alignment)."""
    big, _ = w.alloc_ranks(len(host), host[0].numel() + offset, NAMES[host[0].dtype], dev)
    rows = [big[r, offset:offset + host[0].numel()] for r in range(len(host))]
    for r, t in enumerate(host):
        rows[r].copy_(t)
    return big, rows


def _bits(t):
    return w.to_storage_numpy(t).view(np.uint8)


def _oracle(host, dtype, op):
    ref = [w.to_storage_numpy(t).copy() for t in host]
    oracle.simulate(ref, dtype, op)
    return ref


def _noalloc(lib, rows, dtype, op):
    import ring_all_reduce_rar_gb300 as rar
    p, n = len(rows), rows[0].numel()
    arr = (ctypes.c_void_p * p)(*[t.data_ptr() for t in rows])
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.rar_allreduce_noalloc(arr, p, n, rar.DTYPE_CODES[dtype], rar.OP_CODES[op], stream)
    assert rc == 0, lib.rar_last_error(None)
    torch.cuda.synchronize()


def _assert_equal(rows, ref, what):
    for r in range(len(rows)):
        got = _bits(rows[r])
        exp = ref[r].view(np.uint8)
        assert np.array_equal(got, exp), f"{what}, rank {r}"


@pytest.mark.parametrize("p,n,dtype,op,dist", [
    (8, 8 * 100003 + 5, "bfloat16", "sum", ("normal", 1e-2)),
    (4, 4099, "float32", "avg", ("uniform", -1.0, 1.0)),
    (16, 16 * 4096, "int32", "sum", ("uniform_int", -(1 << 20), 21)),
])
def test_noalloc_matches_oracle_and_allreduce_on_two_calls(lib, p, n, dtype, op, dist):
    import ring_all_reduce_rar_gb300 as rar
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    _, host = w.make_inputs(p, n, dtype, dist, 4242 + p)
    expect = _oracle(host, dtype, op)
    # the existing entry point (handle-based ring executor)
    _, ref = _rows(host, dev)
    with rar.Handle(0, engine="ring") as h:
        h.allreduce(ref, op=op)
        h.check()
    torch.cuda.synchronize()
    _assert_equal(ref, expect, "rar_allreduce against the oracle")
    for call in range(2):
        _, rows = _rows(host, dev)
        _noalloc(lib, rows, dtype, op)
        _assert_equal(rows, expect, f"call {call}")


def test_noalloc_sequence_of_p_limit_misaligned_and_prediv(lib):
    """Back-to-back calls that change p and the channel layout between them,
    the largest p the entry point takes, rank pointers off the 16-byte
    grid, and the pre-divided fp16 average: every call against the oracle."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cases = [
        (64, 64 * 2048 + 33, "bfloat16", "sum", ("normal", 1e-2), 0),   # p = 64: 1024 CTAs
        (4, 4099, "float32", "sum", ("uniform", -1.0, 1.0), 0),         # chunks 1025/1025/1025/1024
        (16, 16 * 3000 + 7, "float32", "max", ("uniform", -1e3, 1e3), 0),
        (8, 8 * 5000 + 3, "bfloat16", "sum", ("normal", 1e-2), 1),      # misaligned rank pointers
        (16, 16 * 4096, "float16", "avg_prediv", ("normal", 1.0), 0),
        (64, 64 * 1000 + 5, "float32", "avg", ("normal", 1.0), 1),
    ]
    for k, (p, n, dtype, op, dist, offset) in enumerate(cases):
        _, host = w.make_inputs(p, n, dtype, dist, 777 + k)
        expect = _oracle(host, dtype, op)
        for call in range(2):
            _, rows = _rows(host, dev, offset)
            _noalloc(lib, rows, dtype, op)
            _assert_equal(rows, expect, f"case {k} (p={p}, {dtype} {op}, offset {offset}), call {call}")


def test_noalloc_rejects_p_above_its_limit(lib):
    dev = torch.device("cuda:0")
    p, n = 65, 100
    big = torch.zeros(p, 128, device=dev)
    arr = (ctypes.c_void_p * p)(*[big[r].data_ptr() for r in range(p)])
    rc = lib.rar_allreduce_noalloc(arr, p, n, 1, 0, None)
    assert rc == 1  # RAR_EINVAL
    assert b"p must be in [1, 64]" in lib.rar_last_error(None)
