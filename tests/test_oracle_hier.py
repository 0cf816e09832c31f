"""Pins of the oracle's hierarchical 2D ring ("Ring All-Reduce, in depth",
"Hierarchy" and "Worked example: flat versus hierarchical")."""
import numpy as np
import pytest

import oracle
from tests.conftest import read_golden

rng = np.random.default_rng(777)


def _naive_i32(bufs):
    s = np.zeros(bufs[0].shape, dtype=np.int64)
    for b in bufs:
        s += b.astype(np.int64)
    return (s & 0xFFFFFFFF).astype(np.uint32).view(np.int32)


def test_worked_example_phase_times():
    """The page's three phase times follow from the oracle's send counts:
    per GPU, the intra-node reduce-scatter and all-gather each send 7/8 of
    the buffer, and the cross-node all-reduce sends 2 x 7/8 of the 1/8
    shard."""
    gold = {k: v[0][0] for k, v in read_golden("hierarchical_worked_example.txt").items()}
    g, m = int(gold["gpus_per_node"]), int(gold["nodes"])
    p = g * m
    n = p * 16  # elements; each stands for buffer_bytes / n bytes
    bytes_per_elem = gold["buffer_bytes"] / n
    bufs = [rng.integers(-9, 9, size=n).astype(np.int32) for _ in range(p)]
    intra, inter = oracle.hier_simulate(bufs, g, "int32", "sum")
    assert np.all(intra == intra[0]) and np.all(inter == inter[0])
    # the shard each GPU all-reduces across nodes
    assert n // g * bytes_per_elem == pytest.approx(gold["shard_bytes"])
    t_intra = intra[0] * bytes_per_elem / gold["intra_bytes_per_s"]
    t_inter = inter[0] * bytes_per_elem / gold["inter_bytes_per_s"]
    assert t_intra == pytest.approx(gold["seconds_intra_reduce_scatter"] + gold["seconds_intra_all_gather"])
    assert t_inter == pytest.approx(gold["seconds_cross_node_allreduce"])


@pytest.mark.parametrize("p,g", [(4, 2), (6, 3), (6, 2), (8, 4), (8, 2), (12, 3), (16, 4), (9, 3)])
def test_int32_brute_force(p, g):
    for n in [0, 1, p - 1, p, 3 * p + 1, 100, 257]:
        bufs = [rng.integers(-(2 ** 31), 2 ** 31, size=n, dtype=np.int64).astype(np.int32) for _ in range(p)]
        expect = _naive_i32(bufs)
        oracle.hier_simulate(bufs, g, "int32", "sum")
        for b in bufs:
            np.testing.assert_array_equal(b, expect)


def _rand(p, n, dtype, seed):
    g_ = np.random.default_rng(seed)
    vals = [g_.normal(0, 1, size=n).astype(np.float32) for _ in range(p)]
    if dtype == "float32":
        return vals
    return [np.array([oracle.f32_to_bf16(float(x)) for x in v], dtype=np.uint16) for v in vals]


@pytest.mark.parametrize("op", ["sum", "avg", "max", "avg_prediv"])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_degenerate_groups_are_the_flat_ring(op, dtype):
    """Nodes of p ranks (one node) or of 1 rank (p nodes) leave only one
    ring: the result equals the flat ring bit for bit."""
    for p in [4, 6, 8]:
        n = 5 * p + 3
        for g in [p, 1]:
            base = _rand(p, n, dtype, p * 10 + g)
            flat = [b.copy() for b in base]
            hier = [b.copy() for b in base]
            oracle.simulate(flat, dtype, op)
            oracle.hier_simulate(hier, g, dtype, op)
            for a, b in zip(flat, hier):
                np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("op", ["sum", "avg", "max", "avg_prediv"])
def test_closed_form_equals_simulator(op):
    for p, g in [(4, 2), (8, 2), (8, 4), (6, 3), (16, 4)]:
        for n in [p, 7 * p + 5, 333]:
            bufs = _rand(p, n, "float32", p * 100 + n)
            folded = oracle.hier_fold_sampled(np.stack(bufs), np.arange(n), n, g, "float32", op)
            oracle.hier_simulate(bufs, g, "float32", op)
            for b in bufs:
                np.testing.assert_array_equal(b, folded)


def test_two_level_order_closed_form():
    """p = 4 in 2 nodes of 2, N = 4: element 0 is in intra-node chunk 0 and
    shard sub-chunk 0.  Node 0's partial is 2^24 + 1, a tie that rounds to
    2^24; node 1's partial is 1 + 1 = 2; across nodes 2^24 + 2 (exact).  The
    flat ring folds 2^24 + 1 + 1 + 1 and stays at 2^24."""
    vals = [2.0 ** 24, 1.0, 1.0, 1.0]
    hier = [np.array([v, 0, 0, 0], dtype=np.float32) for v in vals]
    oracle.hier_simulate(hier, 2, "float32", "sum")
    assert hier[0][0] == np.float32(2.0 ** 24 + 2)
    flat = [np.array([v, 0, 0, 0], dtype=np.float32) for v in vals]
    oracle.simulate(flat, "float32", "sum")
    assert flat[0][0] == np.float32(2.0 ** 24)


def test_send_counts():
    """Across nodes each GPU sends 2(m-1)/m of its 1/g shard (the cross-node
    traffic shrinks by the factor g); in total 2(m-1)N cross-node and
    2m(g-1)N intra-node elements."""
    for p, g in [(8, 2), (8, 4), (16, 4), (12, 3)]:
        m = p // g
        for n in [p * 6, p * 6 + 5]:
            bufs = [rng.integers(-5, 5, size=n).astype(np.int32) for _ in range(p)]
            intra, inter = oracle.hier_simulate(bufs, g, "int32", "sum")
            assert inter.sum() == 2 * (m - 1) * n
            assert intra.sum() == 2 * m * (g - 1) * n
            if n % p == 0:
                assert all(x * m * g == 2 * (m - 1) * n for x in inter)
