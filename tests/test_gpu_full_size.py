"""GPU: the two large workloads -- p = 8, N = 2^30 bf16 (16 GiB, the
benchmark's) and p = 64, N = 2^24 bf16 (2 GiB), N(0, 1e-2), sum -- checked
against the oracle at every element, on the fused engine in the launch
configuration the benchmark times (the streaming path).

The oracle's per-element fold ("Ring All-Reduce, in depth", "The
schedule": element i of chunk c is x_c[i] (+) x_(c+1)[i] (+) ..., rounded
to bf16 after every hop) runs on inputs regenerated on the CPU by the seeded
generator, window by window; the GPU result comes back once.  All ranks must
hold the same bits.  test_gpu_parity.py checks the other engines on these
workloads at sampled indices."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from tests.test_gpu_parity import dev, rar  # noqa: F401

pytestmark = pytest.mark.gpu

WINDOW = 1 << 24  # largest CPU window: elements per rank (32 MiB of bf16)


@pytest.mark.parametrize("workload", ["p8_n1073741824_bf16", "p64_n16777216_bf16"])
def test_full_size_every_element(rar, dev, workload):
    cfg = w.WORKLOADS[workload]
    p, n, dtype, dist, seed = cfg["p"], cfg["n"], cfg["dtype"], cfg["dist"], w.seed_of(cfg["index"])
    big, rows = w.make_inputs(p, n, dtype, dist, seed, device=dev)
    with rar.Handle(0, engine="fused") as h:
        h.allreduce(rows)
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
        expect = oracle.fold_sampled(vals_np, idx.numpy(), n, dtype, "sum", "ring")
        bad = np.nonzero(got[i0:i0 + idx.numel()] != expect)[0]
        return i0, int(bad.size), (bad[:5] + i0).tolist()

    with ThreadPoolExecutor(max_workers=8) as ex:
        results = list(ex.map(check, range(0, n, window)))
    assert len(results) * window >= n
    failures = [(i0, cnt, first) for i0, cnt, first in results if cnt]
    assert not failures, f"{sum(c for _, c, _ in failures)} elements differ; first windows: {failures[:3]}"
