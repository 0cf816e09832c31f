"""GPU: rar_allreduce_range.  Pieces [lo, hi) of the rank buffers, reduced
by separate calls, must leave the buffers exactly as one whole-buffer call
does -- the oracle's result for the whole buffers, bit for bit -- because
every element keeps its chunk (cut from n_total) and with it its fold
order.  Send counts of the pieces add up to the whole call's."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

ENGINE_OPTS = {"fused_regs": dict(engine="fused", fused_path="registers"),
               "fused_stream": dict(engine="fused", fused_path="stream")}
ENGINES = ["fused", "fused_regs", "fused_stream", "ring", "ring_bidir", "fused_tree", "tree"]


@pytest.fixture(scope="module")
def rar():
    import ring_all_reduce_rar_gb300 as rar
    rar.build()
    rar.load_library()
    assert torch.cuda.is_available()
    return rar


@pytest.fixture(scope="module")
def dev():
    return torch.device("cuda:0")


def expect(host, dtype, op, engine, hier_group=0):
    ref = [w.to_storage_numpy(t).copy() for t in host]
    if hier_group:
        intra, inter = oracle.hier_simulate(ref, hier_group, dtype, op)
        return ref, list(intra + inter)
    if engine == "ring_bidir":
        return ref, list(oracle.simulate_bidir(ref, dtype, op))
    if engine in ("fused_tree", "tree"):
        oracle.tree_fold(ref, dtype, op)
        return ref, None
    return ref, list(oracle.simulate(ref, dtype, op))


def run_pieces(rar, dev, host, cuts, op, opts):
    """Reduce [cuts[k], cuts[k+1]) one call each; returns (rows, summed sends)."""
    p, n = len(host), host[0].numel()
    dtype = {torch.int32: "int32", torch.float32: "float32", torch.bfloat16: "bfloat16",
             torch.float16: "float16"}[host[0].dtype]
    _, rows = w.alloc_ranks(p, n, dtype, dev)
    for r in range(p):
        rows[r].copy_(host[r])
    sends = [0] * p
    with rar.Handle(0, **opts) as h:
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            h.allreduce_range([rows[r][lo:hi] for r in range(p)], n, lo, op=op)
            h.check()
            sends = [a + b for a, b in zip(sends, h.send_counts(p))]
    torch.cuda.synchronize()
    return rows, sends


def assert_rows(rows, ref, what):
    for r, (t, e) in enumerate(zip(rows, ref)):
        got = w.to_storage_numpy(t)
        if not np.array_equal(got.view(np.uint8), e.view(np.uint8)):
            bad = np.nonzero(got.view(e.dtype) != e)[0]
            raise AssertionError(f"{what}: rank {r} differs at {len(bad)} elements, first {bad[:8]}")


def check_sends(engine, sends, ref_sends, p, n):
    if engine in ("ring", "ring_bidir"):
        assert sends == ref_sends
    elif engine == "tree":
        assert sum(sends) == 2 * (p - 1) * n
    else:
        assert sends == [0] * p


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("bfloat16", "avg"),
                                      ("int32", "max"), ("float16", "avg_prediv")])
def test_pieces_equal_the_whole_buffer_result(rar, dev, engine, dtype, op):
    """p = 8, n = 10,007 (chunks 1,251 x 7 and 1,250): pieces that start and
    end inside chunks, an empty piece, single elements.  The streaming path
    takes 16-byte aligned pieces only, so it gets cuts on 16-byte bounds."""
    if engine == "tree" and op == "avg_prediv":
        pytest.skip("the tree executor does not offer the pre-divided average")
    p, n = 8, 10007
    dist = ("uniform_int", -(1 << 20), 21) if dtype == "int32" else ("normal", 1.0)
    host = w.make_inputs(p, n, dtype, dist, w.seed_of(0) + 71)[1]
    ref, ref_sends = expect(host, dtype, op, engine)
    if engine == "fused_stream":
        cuts = [0, 2496, 2496, 5000, 9984, n]
    else:
        cuts = [0, 1, 1250, 1251, 3001, 3001, 7777, n - 1, n]
    rows, sends = run_pieces(rar, dev, host, cuts, op, ENGINE_OPTS.get(engine, dict(engine=engine)))
    assert_rows(rows, ref, f"{engine} {dtype} {op} cuts {cuts}")
    check_sends(engine, sends, ref_sends, p, n)


@pytest.mark.parametrize("engine", ["fused", "ring"])
def test_hierarchical_pieces(rar, dev, engine):
    """The two-level order of "Ring All-Reduce, in depth", "Hierarchy" on
    pieces: intra-node chunks and cross-node sub-chunks are cut from n_total."""
    for p, g in [(8, 2), (16, 4)]:
        n = p * 300 + 7
        host = w.make_inputs(p, n, "bfloat16", ("normal", 1e-2), 300 + p)[1]
        ref, ref_sends = expect(host, "bfloat16", "sum", engine, hier_group=g)
        cuts = [0, 5, n // 3, n // 3 + 1, n - 9, n]
        rows, sends = run_pieces(rar, dev, host, cuts, "sum", dict(engine=engine, hier_group=g))
        assert_rows(rows, ref, f"{engine} hier p={p} g={g}")
        if engine == "ring":
            assert sends == ref_sends


def test_many_pieces_large_p(rar, dev):
    """p = 64 (pointer table path is p > 64; here the inline pointers),
    n < p (empty chunks), then p = 100 through the pointer table."""
    for p, n in [(64, 50), (100, 3 * 100 + 17)]:
        host = w.make_inputs(p, n, "float32", ("normal", 1.0), 400 + p)[1]
        for engine in ["fused", "ring"]:
            ref, ref_sends = expect(host, "float32", "sum", engine)
            cuts = sorted(set([0, n] + list(range(0, n, 7))))
            rows, sends = run_pieces(rar, dev, host, cuts, "sum", dict(engine=engine))
            assert_rows(rows, ref, f"{engine} p={p} n={n}")
            check_sends(engine, sends, ref_sends, p, n)


def test_pieces_on_two_streams(rar, dev):
    """Disjoint pieces reduced concurrently on two streams (fused engine,
    one handle per stream) give the whole-buffer result."""
    p, n = 8, 1 << 20
    host = w.make_inputs(p, n, "bfloat16", ("normal", 1e-2), 500)[1]
    ref, _ = expect(host, "bfloat16", "sum", "fused")
    _, rows = w.alloc_ranks(p, n, "bfloat16", dev)
    for r in range(p):
        rows[r].copy_(host[r])
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    cut = 333_336  # 16-byte aligned
    with rar.Handle(0, engine="fused") as h1, rar.Handle(0, engine="fused") as h2:
        h1.allreduce_range([rows[r][:cut] for r in range(p)], n, 0, stream=s1)
        h2.allreduce_range([rows[r][cut:] for r in range(p)], n, cut, stream=s2)
        torch.cuda.synchronize()
        h1.check()
        h2.check()
    assert_rows(rows, ref, "two streams")


def test_range_argument_errors(rar, dev):
    p, n = 4, 64
    _, rows = w.alloc_ranks(p, n, "float32", dev)
    lib = rar.load_library()
    import ctypes
    with rar.Handle(0) as h:
        arr = (ctypes.c_void_p * p)(*[t.data_ptr() for t in rows])
        s = torch.cuda.current_stream().cuda_stream
        assert lib.rar_allreduce_range(h.h, arr, p, n, 10, 5, 1, 0, s) == 1   # lo > hi
        assert lib.rar_allreduce_range(h.h, arr, p, n, 0, n + 1, 1, 0, s) == 1   # hi > n_total
        assert lib.rar_allreduce_range(h.h, arr, p, n, 7, 7, 1, 0, s) == 0   # empty range
        assert lib.rar_allreduce_range(None, arr, p, n, 0, n, 1, 0, s) == 1
        with pytest.raises(rar.RarError):
            h.allreduce_range(rows, n - 1, 0)  # pieces longer than the buffers
