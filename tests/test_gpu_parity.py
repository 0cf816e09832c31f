"""GPU parity: every engine against the oracle, through the C-ABI.

Bit-exact for every ring-order path (int32, fp32, bf16, f16, sum/max/avg);
the tree-order engine is bit-exact against the oracle's tree fold and within
4 p 2^-24 sum|x| of the fp64 sum.  Inputs come from workloads/ (seeded),
generated on the CPU and uploaded, except the 16 GiB workload, which is
generated on the GPU by the same generator and checked against a CPU
regeneration at the sampled indices."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

RING_ENGINES = ["fused", "fused_regs", "fused_stream", "ring", "ring_bidir"]
# "fused_regs" / "fused_stream" force the fused engine's per-thread or
# streaming (bulk-copy) data path; "fused" lets the library choose.  "ring"
# is the ring executor with progress words; "ring_ll" the same schedule with
# the low-latency hand-off (tests/test_gpu_ll.py).
def _mailbox_bytes():
    import os
    import re
    from tests.conftest import ROOT
    text = open(os.path.join(ROOT, "include", "rar.h")).read()
    m = re.search(r"#define RAR_LL_MAILBOX_BYTES \((\d+)u << (\d+)\)", text)
    return int(m.group(1)) << int(m.group(2))


MAILBOX_BYTES = _mailbox_bytes()
# small-buffer tests also run the low-latency ring
SMALL_ENGINES = RING_ENGINES + ["ring_ll"]
ENGINE_OPTS = {"fused_regs": dict(engine="fused", fused_path="registers"),
               "fused_stream": dict(engine="fused", fused_path="stream"),
               "ring": dict(engine="ring", protocol="simple"),
               "ring_ll": dict(engine="ring", protocol="ll"),
               "tree": dict(engine="tree", protocol="simple"),
               "tree_ll": dict(engine="tree", protocol="ll")}


def handle_opts(engine, **opts):
    o = dict(ENGINE_OPTS.get(engine, dict(engine=engine)))
    o.update(opts)
    return o


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


def upload(host_rows, dev, offset_elems=0):
    """Copy CPU rows into one padded device allocation (optionally offset to
    break 16-byte alignment); returns (storage, rows)."""
    p, n = len(host_rows), host_rows[0].numel()
    dtype = {torch.int32: "int32", torch.float32: "float32", torch.bfloat16: "bfloat16",
             torch.float16: "float16"}[host_rows[0].dtype]
    big, _ = w.alloc_ranks(p, n + offset_elems, dtype, dev)
    rows = [big[r, offset_elems:offset_elems + n] for r in range(p)]
    for r in range(p):
        rows[r].copy_(host_rows[r])
    return big, rows


def oracle_expect(host_rows, dtype, op, engine):
    ref = [w.to_storage_numpy(t).copy() for t in host_rows]
    if engine == "ring_bidir":
        sends = oracle.simulate_bidir(ref, dtype, op)
    elif engine in ("fused_tree", "tree", "tree_ll"):
        oracle.tree_fold(ref, dtype, op)
        sends = None
    else:
        sends = oracle.simulate(ref, dtype, op)
    return ref, sends


def assert_bits_equal(rows, ref, what=""):
    for r, (t, e) in enumerate(zip(rows, ref)):
        got = w.to_storage_numpy(t)
        if not np.array_equal(got.view(np.uint8), e.view(np.uint8)):
            bad = np.nonzero(got.view(e.dtype) != e)[0]
            raise AssertionError(f"{what}: rank {r} differs at {len(bad)} elements, first {bad[:8]}")


def run_case(rar, dev, host_rows, dtype, op, engine, offset=0, **opts):
    ref, sends = oracle_expect(host_rows, dtype, op, engine)
    _, rows = upload(host_rows, dev, offset)
    if engine == "fused_stream" and offset:
        engine = "fused"  # the streaming path needs 16-byte aligned ranks
    with rar.Handle(0, **handle_opts(engine, **opts)) as h:
        h.allreduce(rows, op=op)
        h.check()
        got_sends = h.send_counts(len(rows))
    torch.cuda.synchronize()
    assert_bits_equal(rows, ref, f"{engine} {dtype} {op} p={len(rows)} n={rows[0].numel()}")
    p, n = len(rows), rows[0].numel()
    if engine in ("ring", "ring_ll", "ring_bidir"):
        assert list(got_sends) == list(sends)
    elif engine in ("tree", "tree_ll"):
        assert sum(got_sends) == 2 * (p - 1) * n
    else:
        assert list(got_sends) == [0] * p


def gen(p, n, dtype, dist, seed):
    _, rows = w.make_inputs(p, n, dtype, dist, seed)
    return rows


# ----------------------------------------------------------------- page cases

@pytest.mark.parametrize("engine", SMALL_ENGINES + ["fused_tree"])
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
def test_page_trace_p4_n4(rar, dev, engine, dtype):
    """"Ring All-Reduce, in depth", "Tracing four GPUs": [10, 100, 1000, 10000]
    on every rank, six elements sent per rank."""
    vals = w.page_trace_inputs()
    host = [torch.tensor(v, dtype=torch.float32).to(w.TORCH_DTYPES[dtype]) for v in vals]
    _, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce(rows)
        h.check()
        sends = h.send_counts(4)
    if dtype == "bfloat16":
        # 3000 and 10000 are not bf16 values (they round to 3008 and 9984):
        # compare with the oracle on the same bf16 inputs instead
        ref, _ = oracle_expect(host, dtype, "sum", engine)
        assert_bits_equal(rows, ref, "page trace bf16")
    else:
        for t in rows:
            assert t.float().tolist() == [10.0, 100.0, 1000.0, 10000.0]
    if engine in ("ring", "ring_ll"):
        assert sends == [6, 6, 6, 6]


@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_semantics_example_p4_n1(rar, dev, engine):
    """"AllReduce 与 Ring 通信算法详解": [1, 2, 3, 4] -> 10 everywhere (N < p)."""
    host = [torch.tensor([float(r + 1)]) for r in range(4)]
    _, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce(rows)
        h.check()
        sends = h.send_counts(4)
    assert [t.item() for t in rows] == [10.0] * 4
    if engine in ("ring", "ring_ll"):
        assert sends == [2, 2, 1, 1]


# ----------------------------------------------------------------- workloads

@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_p4_n4099_f32_uniform_sum(rar, dev, engine):
    cfg = w.WORKLOADS["p4_n4099_f32"]
    host = gen(cfg["p"], cfg["n"], cfg["dtype"], cfg["dist"], w.seed_of(cfg["index"]))
    run_case(rar, dev, host, "float32", "sum", engine)


@pytest.mark.parametrize("engine", RING_ENGINES)
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_p8_n6553600_f32_normal(rar, dev, engine, op):
    cfg = w.WORKLOADS["p8_n6553600_f32"]
    host = gen(cfg["p"], cfg["n"], cfg["dtype"], cfg["dist"], w.seed_of(cfg["index"]))
    run_case(rar, dev, host, "float32", op, engine)


@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_p64_bf16_full_compare_reduced_n(rar, dev, engine):
    """p = 64 bf16 (large-p case) at a size the oracle runs element by
    element: 64 chunks of ~1000 elements plus a ragged tail."""
    host = gen(64, 64 * 1000 + 13, "bfloat16", ("normal", 1e-2), w.seed_of(3))
    run_case(rar, dev, host, "bfloat16", "sum", engine)


def sampled_indices(n, p, m, seed, halves=False):
    g = np.random.default_rng(seed)
    idx = set(g.integers(0, n, size=m).tolist())
    segs = [(0, n)]
    if halves:
        h = n - n // 2
        segs = [(0, h), (h, n)]
    for lo, hi in segs:
        for c, (s, e) in enumerate(oracle.chunk_bounds(hi - lo, p)):
            for i in (s - 1, s, s + 1, e - 2, e - 1):
                if lo <= lo + i < hi:
                    idx.add(lo + i)
    idx.update([0, n - 1])
    return np.array(sorted(i for i in idx if 0 <= i < n), dtype=np.int64)


def check_sampled(rows, p, n, dtype, dist, seed, op, engine, m=200_000):
    """Sampled parity at full size: the oracle's per-element fold on inputs
    regenerated on the CPU at the sampled indices."""
    mode = {"ring_bidir": "bidir", "fused_tree": "tree"}.get(engine, "ring")
    idx = sampled_indices(n, p, m, seed, halves=(engine == "ring_bidir"))
    vals = w.sample_inputs(seed, p, torch.from_numpy(idx), dist, dtype)
    vals_np = np.stack([w.to_storage_numpy(vals[r]) for r in range(p)])
    expect = oracle.fold_sampled(vals_np, idx, n, dtype, op, mode)
    ti = torch.from_numpy(idx).to(rows[0].device)
    for r in range(p):
        got = w.to_storage_numpy(rows[r][ti])
        assert np.array_equal(got.view(np.uint8), expect.view(np.uint8)), f"{engine} rank {r}"
    for r in range(1, p):
        assert torch.equal(rows[r], rows[0]), f"{engine}: rank {r} differs from rank 0"


@pytest.mark.parametrize("engine", RING_ENGINES)
def test_p64_n16777216_bf16_full_size_sampled(rar, dev, engine):
    cfg = w.WORKLOADS["p64_n16777216_bf16"]
    p, n, seed = cfg["p"], cfg["n"], w.seed_of(cfg["index"])
    big, rows = w.make_inputs(p, n, cfg["dtype"], cfg["dist"], seed, device=dev)
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce(rows)
        h.check()
    check_sampled(rows, p, n, cfg["dtype"], cfg["dist"], seed, "sum", engine)


@pytest.mark.parametrize("engine", RING_ENGINES)
def test_p8_n2pow30_bf16_full_size_sampled(rar, dev, engine):
    """The 16 GiB workload, in the launch configuration the benchmark times."""
    cfg = w.WORKLOADS["p8_n1073741824_bf16"]
    p, n, seed = cfg["p"], cfg["n"], w.seed_of(cfg["index"])
    big, rows = w.make_inputs(p, n, cfg["dtype"], cfg["dist"], seed, device=dev)
    # the GPU-side generation equals the CPU generator at sampled indices
    idx = torch.from_numpy(sampled_indices(n, p, 10_000, 1))
    cpu = w.sample_inputs(seed, p, idx, cfg["dist"], cfg["dtype"])
    for r in range(p):
        assert torch.equal(rows[r][idx.to(dev)].cpu(), cpu[r])
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce(rows)
        h.check()
    check_sampled(rows, p, n, cfg["dtype"], cfg["dist"], seed, "sum", engine)
    del big
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", SMALL_ENGINES)
@pytest.mark.parametrize("pair", range(3))
def test_p16_sweep(rar, dev, engine, pair):
    """p = 16, N = 4^5 .. 4^13: int32 sum, fp32 max, fp32 avg.  Element by
    element up to 4^10, sampled above."""
    dtype, op, dist = w.SWEEP_PAIRS[pair]
    seed = w.seed_of(w.SWEEP_INDEX) + 16 * pair
    p = w.SWEEP_P
    for n in w.SWEEP_SIZES:
        if engine == "ring_ll" and n > 4 ** 8:
            break  # larger buffers do not fit the low-latency mailbox
        if n <= 4 ** 10:
            host = gen(p, n, dtype, dist, seed)
            run_case(rar, dev, host, dtype, op, engine)
        else:
            big, rows = w.make_inputs(p, n, dtype, dist, seed, device=dev)
            with rar.Handle(0, **handle_opts(engine)) as h:
                h.allreduce(rows, op=op)
                h.check()
            check_sampled(rows, p, n, dtype, dist, seed, op, engine, m=50_000)


# ----------------------------------------------------------------- edge cases

@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_odd_p_ragged_n_and_small_n(rar, dev, engine):
    """Runtime-p paths (p not 4/8/16), N < p (empty chunks), ragged tails."""
    for p in [2, 3, 5, 7, 13, 31]:
        for n in [1, 2, p - 1, p, p + 1, 8 * p + 3, 1000 + p]:
            if n < 1:
                continue
            host = gen(p, n, "float32", ("normal", 1.0), 1000 * p + n)
            run_case(rar, dev, host, "float32", "sum", engine)


@pytest.mark.parametrize("engine", SMALL_ENGINES)
@pytest.mark.parametrize("dtype,op", [("int32", "max"), ("bfloat16", "max"), ("bfloat16", "avg"),
                                      ("float16", "sum"), ("float16", "avg"), ("float16", "max"),
                                      ("int32", "sum"), ("float32", "max"), ("float32", "avg_prediv"),
                                      ("bfloat16", "avg_prediv"), ("float16", "avg_prediv")])
def test_dtype_op_matrix(rar, dev, engine, dtype, op):
    dist = ("uniform_int", -(1 << 20), 21) if dtype == "int32" else ("normal", 1.0)
    for p, n in [(4, 4099), (8, 8 * 777 + 5), (6, 1001)]:
        host = gen(p, n, dtype, dist, 7 * p + n)
        run_case(rar, dev, host, dtype, op, engine)


@pytest.mark.parametrize("dtype,op", [("bfloat16", "sum"), ("bfloat16", "max"), ("float16", "avg"),
                                      ("float16", "avg_prediv"), ("int32", "sum"), ("float32", "avg")])
def test_vectors_across_chunk_starts_beyond_p8(rar, dev, dtype, op):
    """Fused per-thread path, p > 8: the vectors that hold an unaligned
    chunk start are folded by a warp each in a launch of their own, every
    element in its own chunk's hop order.  Chunks longer than a vector, and
    shorter ones, so that one vector holds several chunk starts (and empty
    chunks when N < p)."""
    dist = ("uniform_int", -(1 << 20), 21) if dtype == "int32" else ("normal", 1.0)
    for p in [12, 24, 40]:
        for n in [37 * p + 5, 3 * p + 1, p + 3, p - 5]:
            host = gen(p, n, dtype, dist, 31 * p + n)
            run_case(rar, dev, host, dtype, op, "fused_regs")


@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_misaligned_pointers_take_element_path(rar, dev, engine):
    """Rank pointers offset by one element (not 16-byte aligned): same bits."""
    for dtype in ["float32", "bfloat16"]:
        host = gen(8, 8 * 513 + 3, dtype, ("normal", 1.0), 5)
        run_case(rar, dev, host, dtype, "sum", engine, offset=1)


@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_large_p_uses_pointer_table(rar, dev, engine):
    """p > 64: rank pointers travel through the device-side table."""
    p = 96 if engine == "fused" else 72
    host = gen(p, p * 50 + 7, "float32", ("normal", 1.0), 11)
    run_case(rar, dev, host, "float32", "sum", engine)


@pytest.mark.parametrize("engine", ["fused_regs", "fused_stream", "fused_tree", "tree", "tree_ll"])
def test_largest_p(rar, dev, engine):
    """p at the top of the range: 1024 ranks (the fused engines: pointer
    table, runtime p); 200 ranks for the tree executors (one CTA per rank)."""
    p = 200 if engine in ("tree", "tree_ll") else 1024
    host = gen(p, 2 * p + 37, "float32", ("normal", 1.0), 13)
    run_case(rar, dev, host, "float32", "sum", engine)


@pytest.mark.parametrize("engine", SMALL_ENGINES)
def test_trivial_calls(rar, dev, engine):
    one = [torch.arange(10, dtype=torch.float32, device=dev)]
    empty = [torch.zeros(0, device=dev) for _ in range(4)]
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce(one)
        h.allreduce(empty)
        h.check()
    assert one[0].tolist() == list(map(float, range(10)))


def test_fp32_special_values(rar, dev):
    """Subnormals survive (no flush to zero), overflow goes to inf, -0 kept."""
    tiny = np.float32(1e-45)
    host = [torch.tensor([tiny, 3e38, -0.0, 1.0] * 8, dtype=torch.float32) for _ in range(4)]
    for engine in SMALL_ENGINES:
        run_case(rar, dev, host, "float32", "sum", engine)


def test_bf16_subnormals_and_ties(rar, dev):
    vals = np.array([0x0001, 0x0080, 0x8001, 0x3F80, 0x3B80, 0x4380, 0x7F7F] * 9, dtype=np.uint16)
    host = [torch.from_numpy(np.roll(vals, r).astype(np.int16)).view(torch.bfloat16) for r in range(5)]
    for engine in SMALL_ENGINES:
        run_case(rar, dev, host, "bfloat16", "sum", engine)


@pytest.mark.parametrize("engine", SMALL_ENGINES + ["fused_tree"])
def test_prediv_fp16_no_overflow(rar, dev, engine):
    """16 ranks of fp16 4096: the post-divided average overflows to inf (the
    sum 65536 exceeds 65504), the pre-divided one is exactly 4096."""
    p, n = 16, 16 * 64 + 3
    host = [torch.full((n,), 4096.0, dtype=torch.float16) for _ in range(p)]
    for op, expect in [("avg", float("inf")), ("avg_prediv", 4096.0)]:
        _, rows = upload(host, dev)
        with rar.Handle(0, **handle_opts(engine)) as h:
            h.allreduce(rows, op=op)
            h.check()
        torch.cuda.synchronize()
        for t in rows:
            assert torch.all(t.float() == expect), (engine, op)


# ----------------------------------------------------------------- ring engine specifics

def test_ring_race_check_slices_and_channels(rar, dev):
    """Results must not depend on slice size, channel count or block size."""
    host = gen(8, 8 * 10000 + 5, "bfloat16", ("normal", 1e-2), 21)
    ref, _ = oracle_expect(host, "bfloat16", "sum", "ring")
    for engine in ["ring", "ring_bidir"]:
        r2 = oracle_expect(host, "bfloat16", "sum", engine)[0]
        for ch, sl, bt in [(1, 16, 128), (2, 64, 256), (3, 1024, 512), (7, 4096, 512), (16, 160, 64)]:
            _, rows = upload(host, dev)
            with rar.Handle(0, **handle_opts(engine, channels=ch, slice_elems=sl, block_threads=bt)) as h:
                h.allreduce(rows)
                h.check()
            assert_bits_equal(rows, r2 if engine == "ring_bidir" else ref, f"{engine} ch={ch} sl={sl}")


@pytest.mark.parametrize("engine,extra", [("ring", {}), ("ring_bidir", {}), ("ring", dict(hier_group=2)),
                                          ("tree", {})])
def test_slice_order_does_not_change_results(rar, dev, engine, extra):
    """slice_block (slice positions per block of the processing order) only
    reorders the hand-offs: any block size, with several slices per channel
    and step, gives the same bits and send counts."""
    p, n = 8, 8 * 30000 + 13
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 23)
    if extra.get("hier_group"):
        ref = [w.to_storage_numpy(t).copy() for t in host]
        intra, inter = oracle.hier_simulate(ref, extra["hier_group"], "bfloat16", "sum")
        sends = list(intra + inter)
    else:
        ref, sends = oracle_expect(host, "bfloat16", "sum", engine)
    for blk in [1, 2, 3, 7, 1 << 20]:
        _, rows = upload(host, dev)
        with rar.Handle(0, **handle_opts(engine, channels=3, slice_elems=1024, slice_block=blk, **extra)) as h:
            h.allreduce(rows)
            h.check()
            got = h.send_counts(p)
        assert_bits_equal(rows, ref, f"{engine} {extra} slice_block={blk}")
        if engine == "tree":
            assert sum(got) == 2 * (p - 1) * n
        else:
            assert got == list(sends)


def test_tree_weighted_ctas_any_group_size(rar, dev):
    """The tree executor's default grid gives rank r a CTA count in proportion
    to the steps it takes part in, and walks slice groups as a wavefront.
    Any slice size and group size, odd and even p, gives the tree order's
    bits and sends n up plus n per child."""
    for p, n in [(3, 3 * 7000 + 1), (8, 8 * 30000 + 13), (13, 13 * 5000 + 6), (64, 64 * 600 + 3)]:
        host = gen(p, n, "bfloat16", ("normal", 1e-2), 40 + p)
        ref, _ = oracle_expect(host, "bfloat16", "sum", "tree")
        for sl, blk in [(16, 1), (1024, 1), (1024, 2), (1024, 5), (4096, 3), (0, 0)]:
            _, rows = upload(host, dev)
            with rar.Handle(0, **handle_opts("tree", slice_elems=sl, slice_block=blk)) as h:
                h.allreduce(rows)
                h.check()
                got = h.send_counts(p)
            assert_bits_equal(rows, ref, f"tree p={p} slice={sl} block={blk}")
            assert got == [(n if r else 0) + n * len(_tree_children(r, p)) for r in range(p)]


def test_stream_order_with_programmatic_launches(rar, dev):
    """The fused kernels are launched so that they may be scheduled while
    the previous kernel of the stream drains; each waits for it before it
    touches a rank buffer.  A chain on one stream, with no synchronisation
    in between -- fused all-reduce, a torch kernel that rewrites the
    buffers, fused again, the ring executor, the tree executor, fused --
    must give the oracle's result for every step of the chain."""
    p, n = 8, 8 * 50000 + 3
    host = gen(p, n, "float32", ("uniform", -1.0, 1.0), 81)
    _, rows = upload(host, dev)
    big = torch.stack([t for t in host]).clone()  # (p, n) CPU copy of the inputs
    stream = torch.cuda.current_stream()

    def expect(x, order):
        bufs = [w.to_storage_numpy(x[r]).copy() for r in range(p)]
        if order == "tree":
            oracle.tree_fold(bufs, "float32", "sum")
        else:
            oracle.simulate(bufs, "float32", "sum")
        return torch.from_numpy(np.stack(bufs))

    with rar.Handle(0, engine="fused") as hf, rar.Handle(0, engine="ring", protocol="simple") as hr, \
            rar.Handle(0, engine="tree", protocol="simple") as ht:
        hf.allreduce(rows, stream=stream)
        ref = expect(big, "ring")
        for r in range(p):  # a kernel of another library between two calls
            rows[r].mul_(0.5).add_(float(r))
        ref = ref * 0.5 + torch.arange(p, dtype=torch.float32)[:, None]
        hf.allreduce(rows, stream=stream)
        ref = expect(ref, "ring")
        for r in range(p):
            rows[r].sub_(float(r))
        ref = ref - torch.arange(p, dtype=torch.float32)[:, None]
        hr.allreduce(rows, stream=stream)
        ref = expect(ref, "ring")
        for r in range(p):
            rows[r].mul_(0.25)
        ref = ref * 0.25
        ht.allreduce(rows, stream=stream)
        ref = expect(ref, "tree")
        hf.allreduce(rows, stream=stream)
        ref = expect(ref, "ring")
        for h in (hf, hr, ht):
            h.check()
    torch.cuda.synchronize()
    got = torch.stack([t.cpu() for t in rows])
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))


def test_ring_back_to_back_calls_reuse_flags(rar, dev):
    host = gen(4, 4099, "float32", ("uniform", -1.0, 1.0), 3)
    ref, _ = oracle_expect(host, "float32", "sum", "ring")
    with rar.Handle(0, **handle_opts("ring")) as h:
        for _ in range(5):
            _, rows = upload(host, dev)
            h.allreduce(rows)
            h.check()
            assert_bits_equal(rows, ref, "repeat")


@pytest.mark.parametrize("engine", ["ring", "ring_bidir"])
def test_ring_muted_rank_times_out_and_handle_recovers(rar, dev, engine):
    """A rank that never publishes: its neighbour's bounded wait runs out,
    the call reports RAR_ETIMEOUT, and the next call on the same handle
    succeeds (the context stays usable)."""
    host = gen(4, 4 * 4096, "float32", ("normal", 1.0), 9)
    _, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine, timeout_ns=50_000_000, fault_mode="mute", fault_rank=2,
                                     slice_elems=512)) as h:
        h.allreduce(rows)
        assert h.status() == 5  # RAR_ETIMEOUT
        assert "timed out" in rar.rar_last_error(h.h)
        h.set_options(**handle_opts(engine))
        ref, _ = oracle_expect(host, "float32", "sum", engine)
        _, rows = upload(host, dev)
        h.allreduce(rows)
        h.check()
        assert_bits_equal(rows, ref, "after timeout")


@pytest.mark.parametrize("p,n", [(4, 4 * 65536 + 12), (8, 8 * 40000 + 8)])
def test_fused_stream_muted_rank_times_out_and_handle_recovers(rar, dev, p, n):
    """The fused streaming path with a dead rank (RAR_FAULT_MUTE: its bulk
    loads are never issued): the consumers' bounded waits run out, the call
    reports RAR_ETIMEOUT naming that rank, every CTA finishes (the producer
    waits for the loads it did issue), and the next call on the same handle
    is exact ("Ring All-Reduce, in depth", "Failure modes": a dead rank must
    end in an error, not a hang)."""
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 31 + p)
    ref, _ = oracle_expect(host, "bfloat16", "sum", "fused")
    _, rows = upload(host, dev)
    with rar.Handle(0, engine="fused", fused_path="stream", timeout_ns=50_000_000, fault_mode="mute",
                    fault_rank=p - 2) as h:
        h.allreduce(rows)
        assert h.status() == 5  # RAR_ETIMEOUT
        msg = rar.rar_last_error(h.h)
        assert "bulk-copy wait timed out" in msg and f"waiting for rank {p - 2}'s tile" in msg, msg
        assert h.status() == 0  # each failure is reported once
        h.set_options(engine="fused", fused_path="stream", timeout_ns=50_000_000)
        for _ in range(2):
            _, rows = upload(host, dev)
            h.allreduce(rows)
            h.check()
            assert_bits_equal(rows, ref, "fused stream after timeout")


@pytest.mark.parametrize("engine", ["ring", "ring_ll", "ring_bidir", "tree", "tree_ll"])
def test_epoch_wrap_after_a_timeout(rar, dev, engine):
    """A timed-out launch at epoch E raises the abort word to E.  The launch
    that wraps the 32-bit epoch clears it, so that the launch that reaches
    epoch E again after the wrap runs normally instead of taking itself for
    aborted."""
    E = 3
    host = gen(8, 8 * 3000 + 5, "bfloat16", ("normal", 1e-2), 91)
    ref, _ = oracle_expect(host, "bfloat16", "sum", engine)
    with rar.Handle(0, **handle_opts(engine, timeout_ns=50_000_000, fault_mode="mute", fault_rank=2)) as h:
        rar.rar_debug_set_epoch(h.h, E - 1)
        _, rows = upload(host, dev)
        h.allreduce(rows)  # runs with epoch E, times out
        assert h.status() == 5
        h.set_options(**handle_opts(engine, timeout_ns=50_000_000))
        rar.rar_debug_set_epoch(h.h, 0xFFFFFFFE)
        for k in range(E + 1):  # epochs 0xFFFFFFFF (the wrap), 1, ..., E
            _, rows = upload(host, dev)
            h.allreduce(rows)
            h.check()
            assert_bits_equal(rows, ref, f"{engine}: call {k} after the wrap")


@pytest.mark.parametrize("engine", ["ring", "ring_ll", "ring_bidir", "tree", "tree_ll"])
def test_epoch_wrap_around(rar, dev, engine):
    """Progress and mailbox words carry a 32-bit launch epoch.  The launch
    that runs with epoch 0xFFFFFFFF clears them and restarts the count, so
    calls on either side of the wrap stay exact (without the clearing, the
    old high tags would satisfy every wait after the wrap)."""
    host = gen(8, 8 * 3000 + 5, "bfloat16", ("normal", 1e-2), 90)
    ref, _ = oracle_expect(host, "bfloat16", "sum", engine)
    with rar.Handle(0, **handle_opts(engine)) as h:
        for start, calls in [(0xFFFFFFF0, 2), (0xFFFFFFFD, 5)]:
            rar.rar_debug_set_epoch(h.h, start)
            for k in range(calls):
                _, rows = upload(host, dev)
                h.allreduce(rows)
                h.check()
                assert_bits_equal(rows, ref, f"{engine}: epoch {start + k + 1:#x}")


@pytest.mark.parametrize("engine", ["ring", "ring_bidir", "tree"])
def test_step_trace_finds_the_straggler(rar, dev, engine):
    """"Ring All-Reduce, in depth", "Failure modes": a straggler is found by
    comparing per-rank step times.  With a pause injected before every slice
    of one rank, the step trace shows that rank with by far the most work
    time (and, on the one-way ring, its right neighbour with the most wait
    time); the results stay exact."""
    p, n, slow = 8, 8 * 40000 + 3, 3
    host = gen(p, n, "float32", ("normal", 1.0), 77)
    ref, _ = oracle_expect(host, "float32", "sum", engine)
    _, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine, trace=True, fault_mode="delay", fault_rank=slow,
                                     fault_delay_ns=20_000, slice_elems=2048)) as h:
        h.allreduce(rows)
        h.check()
        work, wait = h.trace(p)
    assert_bits_equal(rows, ref, f"{engine} traced straggler")
    steps = 2 * (p - 1) if engine != "tree" else 2 * 3
    assert all(len(w) == steps for w in work + wait)
    total = [sum(w) for w in work]
    order = sorted(range(p), key=total.__getitem__)
    assert order[-1] == slow and total[slow] > 3 * total[order[-2]], total
    if engine == "ring":
        waited = [sum(w) for w in wait]
        assert max(range(p), key=waited.__getitem__) == (slow + 1) % p, waited
        # every rank works at every step of the ring
        assert all(x > 0 for w in work for x in w)


def test_step_trace_refusals(rar, dev):
    """rar_trace reports only a traced call of an executor with progress
    words: not an untraced call, nor the fused engine, nor another p."""
    host = gen(4, 4 * 3000, "float32", ("normal", 1.0), 78)
    _, rows = upload(host, dev)
    with rar.Handle(0, engine="ring", protocol="simple") as h:
        h.allreduce(rows)
        with pytest.raises(rar.RarError):
            h.trace(4)
    with rar.Handle(0, engine="fused", trace=True) as h:
        h.allreduce(rows)
        with pytest.raises(rar.RarError):
            h.trace(4)
    with rar.Handle(0, engine="ring", protocol="simple", trace=True) as h:
        h.allreduce(rows)
        work, wait = h.trace(4)
        assert len(work) == 4 and len(work[0]) == 6
        with pytest.raises(rar.RarError):
            h.trace(5)


def test_ring_straggler_keeps_results(rar, dev):
    """An injected slow rank (pause before every slice) changes timing only."""
    host = gen(4, 4 * 3000 + 1, "float32", ("normal", 1.0), 10)
    run_case(rar, dev, host, "float32", "sum", "ring", fault_mode="delay", fault_rank=1,
             fault_delay_ns=20_000, slice_elems=1024)


@pytest.mark.parametrize("engine", ["fused", "ring", "ring_bidir"])
def test_reduce_scatter_then_all_gather(rar, dev, engine):
    """The two halves alone: after reduce-scatter rank r owns chunk (r + 1);
    all-gather then completes the all-reduce."""
    p, n = 8, 8 * 999 + 5
    host = gen(p, n, "float32", ("normal", 1.0), 12)
    full, _ = oracle_expect(host, "float32", "sum", engine)
    _, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.reduce_scatter(rows)
        h.check()
        if engine == "ring":
            rs = [w.to_storage_numpy(t).copy() for t in host]
            oracle.simulate(rs, "float32", "sum", first_step=0, n_steps=p - 1)
            assert_bits_equal(rows, rs, "ring reduce-scatter state")
            assert h.send_counts(p) == [n - (e - s) for s, e in
                                        [oracle.chunk_bounds(n, p)[(r + 1) % p] for r in range(p)]]
        else:
            segs = [(0, n, +1)] if engine == "fused" else [(0, n - n // 2, +1), (n - n // 2, n, -1)]
            for lo, hi, d in segs:
                for r in range(p):
                    s, e = oracle.chunk_bounds(hi - lo, p)[(r + d) % p]
                    got = w.to_storage_numpy(rows[r][lo + s:lo + e])
                    assert np.array_equal(got, full[r][lo + s:lo + e])
        h.all_gather(rows, )
        h.check()
    assert_bits_equal(rows, full, f"{engine} rs+ag")


# ----------------------------------------------------------------- tree order

def test_tree_order_bit_exact_and_bound(rar, dev):
    for p in [2, 3, 4, 8, 16, 64]:
        n = p * 300 + 7
        host = gen(p, n, "float32", ("normal", 1.0), 100 + p)
        run_case(rar, dev, host, "float32", "sum", "fused_tree")
        _, rows = upload(host, dev)
        with rar.Handle(0, engine="fused_tree") as h:
            h.allreduce(rows)
            h.check()
        ref, mag = oracle.f64_sum([w.to_storage_numpy(t).copy() for t in host], "float32")
        got = rows[0].cpu().double().numpy()
        assert np.all(np.abs(got - ref) <= 4 * p * 2.0 ** -24 * mag)


# ----------------------------------------------------------------- hierarchical

@pytest.mark.parametrize("engine", ["fused", "ring"])
@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("bfloat16", "avg"),
                                      ("float32", "max"), ("float16", "avg_prediv"), ("int32", "sum")])
def test_hierarchical_matches_oracle(rar, dev, engine, dtype, op):
    """"Ring All-Reduce, in depth", "Hierarchy": the two-level schedule
    (reduce-scatter in nodes, all-reduce of shards across nodes, all-gather
    in nodes) against the oracle's composition of rings, bit for bit; the
    ring engine's per-rank sends equal the oracle's intra + cross-node."""
    dist = ("uniform_int", -(1 << 20), 21) if dtype == "int32" else ("normal", 1.0)
    for p, g in [(4, 2), (8, 2), (8, 4), (16, 4), (64, 8)]:
        n = p * 300 + 7
        host = gen(p, n, dtype, dist, 1000 + p * g)
        ref = [w.to_storage_numpy(t).copy() for t in host]
        intra, inter = oracle.hier_simulate(ref, g, dtype, op)
        _, rows = upload(host, dev)
        with rar.Handle(0, engine=engine, hier_group=g) as h:
            h.allreduce(rows, op=op)
            h.check()
            sends = h.send_counts(p)
        torch.cuda.synchronize()
        assert_bits_equal(rows, ref, f"{engine} hier p={p} g={g} {dtype} {op}")
        if engine == "ring":
            assert list(sends) == list(intra + inter)


def test_hierarchical_degenerate_groups_are_flat(rar, dev):
    p, n = 8, 8 * 123 + 5
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 5)
    ref, _ = oracle_expect(host, "bfloat16", "sum", "ring")
    for engine in ["fused", "ring"]:
        for g in [1, p]:
            _, rows = upload(host, dev)
            with rar.Handle(0, engine=engine, hier_group=g) as h:
                h.allreduce(rows)
                h.check()
            assert_bits_equal(rows, ref, f"{engine} g={g}")


def test_hierarchical_rejections(rar, dev):
    host = gen(8, 800, "float32", ("normal", 1.0), 6)
    _, rows = upload(host, dev)
    for opts, code in [(dict(engine="ring_bidir", hier_group=2), 2), (dict(engine="fused_tree", hier_group=2), 2),
                       (dict(engine="fused", fused_path="stream", hier_group=2), 2),
                       (dict(engine="ring", hier_group=3), 1)]:
        with rar.Handle(0, **opts) as h:
            with pytest.raises(rar.RarError) as e:
                h.allreduce(rows)
            assert e.value.code == code, opts
    with rar.Handle(0, engine="ring", hier_group=2) as h:
        with pytest.raises(rar.RarError) as e:
            h.reduce_scatter(rows)
        assert e.value.code == 2


# ----------------------------------------------------------------- tree executor

def _tree_children(r, p):
    L = max(1, (p - 1).bit_length())
    kids = []
    for l in range(L):
        span = 1 << l
        if r % (2 * span) == 0 and r + span < p:
            kids.append(r + span)
    return kids


@pytest.mark.parametrize("protocol", ["simple", "ll"])
@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("float16", "avg"),
                                      ("float32", "max"), ("int32", "sum"), ("bfloat16", "avg")])
def test_tree_executor_matches_tree_order(rar, dev, dtype, op, protocol):
    """"Derive the cost of a ring all-reduce": reduce up a binary tree,
    broadcast down.  The executor folds in the oracle's tree order bit for
    bit, with either hand-off; every non-root rank sends n up once and n to
    each child."""
    dist = ("uniform_int", -(1 << 20), 21) if dtype == "int32" else ("normal", 1.0)
    e = 2 if dtype in ("bfloat16", "float16") else 4
    for p in [2, 3, 4, 5, 7, 8, 13, 16, 64]:
        for n in [1, p + 3, 4099, 64 * 1000 + 5]:
            levels = max(1, (p - 1).bit_length())
            if protocol == "ll" and p * (levels + 1) * -(-n * e // 4) * 8 > MAILBOX_BYTES:
                continue  # does not fit the low-latency mailbox
            host = gen(p, n, dtype, dist, 300 + p * 7 + n)
            ref = [w.to_storage_numpy(t).copy() for t in host]
            oracle.tree_fold(ref, dtype, op)
            _, rows = upload(host, dev)
            with rar.Handle(0, engine="tree", protocol=protocol) as h:
                h.allreduce(rows, op=op)
                h.check()
                sends = h.send_counts(p)
            torch.cuda.synchronize()
            assert_bits_equal(rows, ref, f"tree p={p} n={n} {dtype} {op}")
            expect = [(n if r else 0) + n * len(_tree_children(r, p)) for r in range(p)]
            assert list(sends) == expect
            assert sum(sends) == 2 * (p - 1) * n


@pytest.mark.parametrize("protocol", ["simple", "ll"])
def test_tree_executor_fault_and_rejections(rar, dev, protocol):
    host = gen(8, 8 * 4096, "float32", ("normal", 1.0), 8)
    _, rows = upload(host, dev)
    with rar.Handle(0, engine="tree", protocol=protocol, timeout_ns=50_000_000, fault_mode="mute",
                    fault_rank=2) as h:
        # rank 2 is waited on by rank 0 at level 1 (a muted leaf such as rank 1
        # stalls nobody: its data is only read at step 0, which has no wait)
        h.allreduce(rows)
        assert h.status() == 5
    for fn, kw in [("reduce_scatter", {}), ("allreduce", dict(op="avg_prediv"))]:
        with rar.Handle(0, engine="tree") as h:
            with pytest.raises(rar.RarError) as e:
                getattr(h, fn)(rows, **kw)
            assert e.value.code == 2
    with rar.Handle(0, engine="tree", hier_group=2) as h:
        with pytest.raises(rar.RarError) as e:
            h.allreduce(rows)
        assert e.value.code == 2


# ----------------------------------------------------------------- CUDA graphs

@pytest.mark.parametrize("engine,opts", [("fused_regs", {}), ("fused_stream", {}), ("ring", {}), ("ring_ll", {}),
                                         ("ring_bidir", {}), ("tree", {}), ("tree_ll", {}),
                                         ("ring", dict(hier_group=2)), ("fused_tree", {})])
def test_captured_call_replays(rar, dev, engine, opts):
    """A call recorded with stream capture replays correctly again and again:
    the ring and tree executors take their epoch from device memory."""
    p, n = 8, 8 * 3000 + 5
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 60)
    if opts.get("hier_group"):
        ref = [w.to_storage_numpy(t).copy() for t in host]
        oracle.hier_simulate(ref, opts["hier_group"], "bfloat16", "sum")
    else:
        ref, _ = oracle_expect(host, "bfloat16", "sum", engine)
    big, rows = upload(host, dev)
    with rar.Handle(0, **handle_opts(engine, **opts)) as h:
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                h.allreduce(rows, stream=stream)
        torch.cuda.synchronize()
        for replay in range(3):
            for r in range(p):
                rows[r].copy_(host[r])
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            assert h.status() == 0
            assert_bits_equal(rows, ref, f"{engine} {opts} replay {replay}")


# ----------------------------------------------------------------- host buffers

@pytest.mark.parametrize("engine", ["fused", "fused_stream", "ring", "ring_ll"])
def test_allreduce_host_pinned_and_pageable(rar, dev, engine):
    """rar_allreduce_host: pinned host buffers are reduced in place by the GPU
    (zero copy); pageable ones are staged through device buffers.  Both equal
    the oracle bit for bit."""
    p, n = 8, 8 * 5000 + 5
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 77)
    ref, _ = oracle_expect(host, "bfloat16", "sum", "ring")
    pinned = [t.clone().pin_memory() for t in host]
    with rar.Handle(0, **handle_opts(engine)) as h:
        h.allreduce_host(pinned)
        h.check()
        torch.cuda.synchronize()
        assert_bits_equal(pinned, ref, f"{engine} pinned")
        pageable = [t.clone() for t in host]
        _, staging = upload(host, dev)
        h.allreduce_host(pageable, staging)
        h.check()
        torch.cuda.synchronize()
        assert_bits_equal(pageable, ref, f"{engine} pageable")
        assert_bits_equal(staging, ref, f"{engine} staging")
        with pytest.raises(rar.RarError) as e:
            h.allreduce_host([t.clone() for t in host])
        assert e.value.code == 1


# ----------------------------------------------------------------- argument errors

def test_argument_errors(rar, dev):
    a = torch.zeros(4 * 100, device=dev)
    with rar.Handle(0) as h:
        # overlapping rank buffers
        assert rar.rar_allreduce_ptrs(h.h, [a.data_ptr(), a.data_ptr() + 8], 100, "float32") == 1
        # host pointer
        c = torch.zeros(100)
        assert rar.rar_allreduce_ptrs(h.h, [a.data_ptr(), c.data_ptr()], 100, "float32") == 1
        # NULL rank pointer, p out of range
        assert rar.rar_allreduce_ptrs(h.h, [a.data_ptr(), 0], 100, "float32") == 1
        assert rar.rar_allreduce_ptrs(h.h, [], 100, "float32") == 1
        # avg on int32 is not offered
        i = torch.zeros(2, 10, dtype=torch.int32, device=dev)
        with pytest.raises(rar.RarError) as e:
            h.allreduce([i[0], i[1]], op="avg")
        assert e.value.code == 2


def test_option_errors(rar, dev):
    """Out-of-range options are refused by rar_init and rar_set_options
    (RAR_EINVAL), and the handle keeps its previous options."""
    bad = [dict(engine=7), dict(protocol=3), dict(fused_path=5), dict(block_threads=100), dict(channels=-1),
           dict(fault_mode=9), dict(hier_group=-2)]
    for opts in bad:
        with pytest.raises(rar.RarError) as e:
            rar.Handle(0, **opts)
        assert e.value.code == 1, opts
    host = gen(4, 4099, "float32", ("uniform", -1.0, 1.0), 3)
    ref, _ = oracle_expect(host, "float32", "sum", "ring")
    with rar.Handle(0, engine="ring", protocol="ll") as h:
        for opts in bad:
            with pytest.raises(rar.RarError) as e:
                h.set_options(**opts)
            assert e.value.code == 1, opts
        _, rows = upload(host, dev)
        h.allreduce(rows)
        h.check()
        assert_bits_equal(rows, ref, "after refused options")
