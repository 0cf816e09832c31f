"""GPU: the low-latency hand-off (rar_options.protocol) of the ring and tree
engines.  They run the schedules of "Ring All-Reduce, in depth", "The
schedule" and of the tree in "Derive the cost of a ring all-reduce" with
every message word tagged by the launch, so results and send counts must
equal the oracle's exactly, like the progress-word executors'.  The parity
cases shared with the other engines run them as "ring_ll" / "tree_ll" in
test_gpu_parity.py; this file covers what is particular to them."""
import pytest
import torch

from tests.test_gpu_parity import (MAILBOX_BYTES, assert_bits_equal, dev, gen, oracle_expect, rar,  # noqa: F401
                                   run_case, upload)

pytestmark = pytest.mark.gpu


def test_channel_counts_do_not_change_results(rar, dev):
    """The words of a chunk are spread over channels x 128 threads per rank;
    one thread may poll several words per step.  Results do not depend on it."""
    host = gen(8, 8 * 20000 + 5, "bfloat16", ("normal", 1e-2), 31)
    ref, sends = oracle_expect(host, "bfloat16", "sum", "ring")
    for ch in [1, 2, 3, 8, 40]:
        _, rows = upload(host, dev)
        with rar.Handle(0, engine="ring", protocol="ll", channels=ch) as h:
            h.allreduce(rows)
            h.check()
            got = h.send_counts(8)
        assert_bits_equal(rows, ref, f"channels={ch}")
        assert got == list(sends)


def test_back_to_back_and_alternating_protocols(rar, dev):
    """Mailbox words carry the launch's epoch, shared with the progress-word
    executor on the same handle: calls in any order, with stale words from
    earlier launches in the mailbox, stay exact."""
    host = gen(4, 4099, "float32", ("uniform", -1.0, 1.0), 3)
    ref, _ = oracle_expect(host, "float32", "sum", "ring")
    with rar.Handle(0, engine="ring", protocol="ll") as h:
        for k in range(6):
            h.set_options(engine="ring", protocol="ll" if k % 3 != 2 else "simple")
            _, rows = upload(host, dev)
            h.allreduce(rows)
            h.check()
            assert_bits_equal(rows, ref, f"call {k}")


def test_largest_p_one_cta_per_rank(rar, dev):
    """p = 1024: one 128-thread CTA per rank, all co-resident; N < p, so
    chunks of one element and empty ones (p * 2 (p - 1) one-word slots fit
    the mailbox; longer chunks at this p do not)."""
    p = 1024
    host = gen(p, 1000, "float32", ("normal", 1.0), 13)
    run_case(rar, dev, host, "float32", "sum", "ring_ll")


def test_muted_rank_times_out_and_handle_recovers(rar, dev):
    """A rank that never sends: its neighbour's bounded wait runs out, the
    call reports RAR_ETIMEOUT naming the ranks, and the next call succeeds."""
    host = gen(4, 4 * 4096, "float32", ("normal", 1.0), 9)
    _, rows = upload(host, dev)
    with rar.Handle(0, engine="ring", protocol="ll", timeout_ns=50_000_000, fault_mode="mute", fault_rank=2) as h:
        h.allreduce(rows)
        assert h.status() == 5  # RAR_ETIMEOUT
        msg = rar.rar_last_error(h.h)
        assert "timed out" in msg and "waiting on rank" in msg, msg
        h.set_options(engine="ring", protocol="ll")
        ref, _ = oracle_expect(host, "float32", "sum", "ring")
        _, rows = upload(host, dev)
        h.allreduce(rows)
        h.check()
        assert_bits_equal(rows, ref, "after timeout")


def test_straggler_keeps_results(rar, dev):
    host = gen(4, 4 * 3000 + 1, "float32", ("normal", 1.0), 10)
    run_case(rar, dev, host, "float32", "sum", "ring_ll", fault_mode="delay", fault_rank=1, fault_delay_ns=20_000)


def test_mailbox_limit_and_rejections(rar, dev):
    """protocol=ll runs while p * 2 (p - 1) chunk-sized slots fit in the
    mailbox; beyond that, and for the bidirectional ring, the hierarchical
    schedule and the reduce-scatter / all-gather halves, it is refused
    (RAR_EUNSUPPORTED)."""
    p = 16
    words_fit = MAILBOX_BYTES // (8 * p * 2 * (p - 1))
    n_fit = p * words_fit  # fp32: one element per word
    for n, ok in [(n_fit, True), (n_fit + p, False)]:
        host = gen(p, n, "float32", ("normal", 1.0), 17)
        _, rows = upload(host, dev)
        with rar.Handle(0, engine="ring", protocol="ll") as h:
            if ok:
                h.allreduce(rows)
                h.check()
                ref, _ = oracle_expect(host, "float32", "sum", "ring")
                assert_bits_equal(rows, ref, f"n={n}")
            else:
                with pytest.raises(rar.RarError) as e:
                    h.allreduce(rows)
                assert e.value.code == 2
    host = gen(8, 800, "float32", ("normal", 1.0), 6)
    _, rows = upload(host, dev)
    for opts in [dict(engine="ring_bidir", protocol="ll"), dict(engine="ring", protocol="ll", hier_group=2)]:
        with rar.Handle(0, **opts) as h:
            with pytest.raises(rar.RarError) as e:
                h.allreduce(rows)
            assert e.value.code == 2, opts
    with rar.Handle(0, engine="ring", protocol="ll") as h:
        for call in (h.reduce_scatter, h.all_gather):
            with pytest.raises(rar.RarError) as e:
                call(rows)
            assert e.value.code == 2


@pytest.mark.parametrize("n", [4096, 65536, 262144, 1 << 20])
def test_auto_protocol_is_exact_on_both_sides_of_the_switch(rar, dev, n):
    """protocol=auto takes the low-latency hand-off for small buffers and the
    progress words for large ones; either way the result is the oracle's."""
    p = 8
    host = gen(p, n, "bfloat16", ("normal", 1e-2), 41)
    run_case(rar, dev, host, "bfloat16", "sum", "ring", protocol="auto")


def test_ranges_on_the_low_latency_ring(rar, dev):
    """rar_allreduce_range with protocol=ll: chunks cut from n_total."""
    p, n = 8, 10007
    host = gen(p, n, "float32", ("normal", 1.0), 71)
    ref, sends = oracle_expect(host, "float32", "sum", "ring")
    _, rows = upload(host, dev)
    total = [0] * p
    cuts = [0, 1, 1250, 1251, 3001, 3001, 7777, n - 1, n]
    with rar.Handle(0, engine="ring", protocol="ll") as h:
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            h.allreduce_range([rows[r][lo:hi] for r in range(p)], n, lo)
            h.check()
            total = [a + b for a, b in zip(total, h.send_counts(p))]
    torch.cuda.synchronize()
    assert_bits_equal(rows, ref, "ranges")
    assert total == list(sends)


def test_tree_channel_counts_do_not_change_results(rar, dev):
    """Low-latency tree: with few channels a thread carries several batches
    of words through the whole tree, one batch after the other."""
    p, n = 13, 3000 * 13 + 7
    host = gen(p, n, "float32", ("normal", 1.0), 51)
    ref, _ = oracle_expect(host, "float32", "sum", "tree")
    for ch in [1, 3, 50]:
        _, rows = upload(host, dev)
        with rar.Handle(0, engine="tree", protocol="ll", channels=ch) as h:
            h.allreduce(rows)
            h.check()
            sends = h.send_counts(p)
        assert_bits_equal(rows, ref, f"channels={ch}")
        assert sum(sends) == 2 * (p - 1) * n


def test_tree_mailbox_limit(rar, dev):
    """The low-latency tree needs p * (ceil(log2 p) + 1) buffer-sized slots."""
    p = 16
    n_fit = MAILBOX_BYTES // (8 * p * 5)  # fp32: one element per word, 5 slots at p = 16
    for n, ok in [(n_fit, True), (n_fit + 1, False)]:
        host = gen(p, n, "float32", ("normal", 1.0), 57)
        _, rows = upload(host, dev)
        with rar.Handle(0, engine="tree", protocol="ll") as h:
            if ok:
                h.allreduce(rows)
                h.check()
                ref, _ = oracle_expect(host, "float32", "sum", "tree")
                assert_bits_equal(rows, ref, f"n={n}")
            else:
                with pytest.raises(rar.RarError) as e:
                    h.allreduce(rows)
                assert e.value.code == 2
