"""The oracle against the values the pages print (tests/golden/)."""
from fractions import Fraction

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


def _bf16_rne(x: Fraction) -> Fraction:
    """x rounded to the nearest bfloat16 (8 significant bits, ties to even),
    written from the format's definition for the normal range these values
    lie in; independent of the oracle's conversion."""
    if x == 0:
        return Fraction(0)
    sign, a = (-1 if x < 0 else 1), abs(x)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)  # spacing of 8-bit significands in [2^e, 2^(e+1))
    lo = int(a / q)
    rem = a / q - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * q


def test_page_trace_bf16_rounded_inputs():
    """The page's example with its inputs rounded to bf16 (3000 -> 3008 and
    5000, an intermediate, -> 4992: the page prints exact values only, so
    the expected results here are derived, not printed).  Each element of
    chunk c is folded in hop order x_c, x_(c+1), ... with one bf16 rounding
    per hop, computed with exact rationals; the oracle must match every
    element on every rank.  Chunk 3's path, 4000 + 1000 = 5000 -> 4992,
    + 2000 = 6992 -> 6976 (a tie, to even), + 3008 = 9984, differs from a
    single rounding of the exact sum only by luck of the last step, so a
    wrong order or a missing per-hop rounding shows in the intermediate
    values checked below."""
    g = read_golden("ring_trace_p4_n4.txt")
    rows = [[_bf16_rne(Fraction(v)) for v in row[1:]] for row in g["input"]]
    p, n = len(rows), len(rows[0])
    bufs = [np.array([oracle.f32_to_bf16(float(v)) for v in row], dtype=np.uint16) for row in rows]
    oracle.simulate(bufs, "bfloat16", "sum")
    expect = []
    for i in range(n):  # n = p: element i is chunk i
        acc = rows[i][i]
        for k in range(1, p):
            acc = _bf16_rne(acc + rows[(i + k) % p][i])
        expect.append(acc)
    assert rows[2][3] == 3008 and expect[3] == 9984
    for b in bufs:
        assert [Fraction(oracle.bf16_to_f32(int(h))) for h in b] == expect
    # the per-hop intermediates of chunk 3 after each reduce-scatter step
    bufs = [np.array([oracle.f32_to_bf16(float(v)) for v in row], dtype=np.uint16) for row in rows]
    path = []
    for s in range(p - 1):
        step = [b.copy() for b in bufs]
        oracle.simulate(step, "bfloat16", "sum", first_step=0, n_steps=s + 1)
        owner = (3 + s + 1) % p  # chunk 3 starts at rank 3 and moves one rank per step
        path.append(oracle.bf16_to_f32(int(step[owner][3])))
    assert path == [4992.0, 6976.0, 9984.0]


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
