"""GPU: the large workloads checked against the oracle at every element, on
every engine the benchmark times, in the launch configuration it times:
p = 8, N = 2^30 bf16 (16 GiB, the benchmark's workload) and p = 64,
N = 2^24 bf16 on the fused engine, the ring executor, the bidirectional ring
and the tree executor; p = 8, N = 6,553,600 fp32 on the fused engine; and
the p = 16 sweep at N = 4^11 ... 4^13 (int32 sum, fp32 max, fp32 avg) on
the fused engine, the ring and the bidirectional ring.

The oracle's per-element fold runs on inputs regenerated on the CPU by the
seeded generator, window by window; the GPU result comes back once.  Ring
order ("Ring All-Reduce, in depth", "The schedule": element i of chunk c is
x_c[i] (+) x_(c+1)[i] (+) ..., rounded to the dtype after every hop); the
mirrored order on the second half for the bidirectional ring ("What real
libraries add", "Bidirectional rings"); adjacent pairs level by level for
the tree ("Derive the cost of a ring all-reduce", tree all-reduce).  All
ranks must hold the same bits."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from tests.test_gpu_parity import dev, rar  # noqa: F401

pytestmark = pytest.mark.gpu

WINDOW = 1 << 24  # largest CPU window: elements per rank (32 MiB of bf16)


# (name, engine, p, n, dtype, dist, seed, op, oracle order)
CASES = [(name, "fused", cfg["p"], cfg["n"], cfg["dtype"], cfg["dist"], w.seed_of(cfg["index"]), "sum", "ring")
         for name, cfg in w.WORKLOADS.items() if cfg["n"] > 4 ** 10]
# the executors on the two largest workloads, as the benchmark times them
for _eng, _mode in [("ring", "ring"), ("ring_bidir", "bidir"), ("tree", "tree")]:
    CASES += [(f"{name}_{_eng}", _eng, cfg["p"], cfg["n"], cfg["dtype"], cfg["dist"], w.seed_of(cfg["index"]), "sum",
               _mode) for name, cfg in w.WORKLOADS.items() if cfg["n"] >= 1 << 24]
# the p = 16 sweep above the sizes the other tests check element by element
for _eng, _mode in [("fused", "ring"), ("ring", "ring"), ("ring_bidir", "bidir")]:
    CASES += [(f"p16_n{n}_{w.SWEEP_PAIRS[k][0]}_{w.SWEEP_PAIRS[k][1]}_{_eng}", _eng, w.SWEEP_P, n,
               w.SWEEP_PAIRS[k][0], w.SWEEP_PAIRS[k][2], w.seed_of(w.SWEEP_INDEX) + 16 * k, w.SWEEP_PAIRS[k][1], _mode)
              for k in range(len(w.SWEEP_PAIRS)) for n in w.SWEEP_SIZES if n > 4 ** 10]


@pytest.mark.parametrize("name,engine,p,n,dtype,dist,seed,op,mode", CASES, ids=[c[0] for c in CASES])
def test_full_size_every_element(rar, dev, name, engine, p, n, dtype, dist, seed, op, mode):
    big, rows = w.make_inputs(p, n, dtype, dist, seed, device=dev)
    with rar.Handle(0, engine=engine) as h:
        h.allreduce(rows, op=op)
        h.check()
    for r in range(1, p):
        assert torch.equal(rows[r], rows[0]), f"rank {r} differs from rank 0"
    got = w.to_storage_numpy(rows[0])
    del big, rows
    torch.cuda.empty_cache()

    window = min(WINDOW, max(1 << 20, n // 16))  # at least 16 windows for the threads

    def check(i0):
        idx = torch.arange(i0, min(n, i0 + window), dtype=torch.int64)
        vals = w.sample_inputs(seed, p, idx, dist, dtype)
        vals_np = np.stack([w.to_storage_numpy(vals[r]) for r in range(p)])
        expect = oracle.fold_sampled(vals_np, idx.numpy(), n, dtype, op, mode)
        bad = np.nonzero(got[i0:i0 + idx.numel()] != expect)[0]
        return i0, int(bad.size), (bad[:5] + i0).tolist()

    with ThreadPoolExecutor(max_workers=8) as ex:
        results = list(ex.map(check, range(0, n, window)))
    assert len(results) * window >= n
    failures = [(i0, cnt, first) for i0, cnt, first in results if cnt]
    assert not failures, f"{sum(c for _, c, _ in failures)} elements differ; first windows: {failures[:3]}"
