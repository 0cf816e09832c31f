"""The oracle against the values the pages print (tests/golden/)."""
import numpy as np
import pytest

import oracle
from tests.conftest import read_golden


def _inputs(g, dtype):
    st = np.int32 if dtype == "int32" else np.float32
    return [np.array(row[1:], dtype=st) for row in g["input"]]


@pytest.mark.parametrize("dtype", ["int32", "float32"])
def test_page_trace_result_and_sends(dtype):
    """"Ring All-Reduce, in depth", "Tracing four GPUs": result on every rank
    and six elements sent per rank."""
    g = read_golden("ring_trace_p4_n4.txt")
    bufs = _inputs(g, dtype)
    sends = oracle.simulate(bufs, dtype, "sum")
    expect = np.array(g["expect"][0], dtype=bufs[0].dtype)
    for b in bufs:
        np.testing.assert_array_equal(b, expect)
    np.testing.assert_array_equal(sends, np.array(g["sends"][0], dtype=np.int64))


def test_page_trace_chunk0_path():
    """Same section: chunk 0's value at each rank after each step (1 -> 3 ->
    6 -> 10 in the reduce-scatter, then copied 3 -> 0 -> 1 -> 2)."""
    g = read_golden("ring_trace_p4_n4.txt")
    for step, rank, value in g["chunk0"]:
        bufs = _inputs(g, "float32")
        oracle.simulate(bufs, "float32", "sum", first_step=0, n_steps=int(step) + 1)
        assert bufs[int(rank)][0] == value


def test_page_trace_bf16():
    """The page's example is exact in bf16 too (all values need <= 8 bits)."""
    g = read_golden("ring_trace_p4_n4.txt")
    bufs = [np.array([oracle.f32_to_bf16(v) for v in row[1:]], dtype=np.uint16) for row in g["input"]]
    oracle.simulate(bufs, "bfloat16", "sum")
    expect = [oracle.f32_to_bf16(v) for v in g["expect"][0]]
    for b in bufs:
        assert list(b) == expect


def test_semantics_example_p4_n1():
    """"AllReduce 与 Ring 通信算法详解", "AllReduce 语义": [1,2,3,4] -> 10 on
    every rank.  N = 1 < p, so three of the four chunks are empty."""
    g = read_golden("allreduce_semantics_p4_n1.txt")
    bufs = _inputs(g, "float32")
    sends = oracle.simulate(bufs, "float32", "sum")
    for b in bufs:
        assert b[0] == g["expect"][0][0]
    # only chunk 0 is non-empty: rank r sends it in reduce-scatter unless it
    # is the owner's predecessor's ... by the law 2N - |C_(r+1)| - |C_(r+2)|
    np.testing.assert_array_equal(sends, [2, 2, 1, 1])
