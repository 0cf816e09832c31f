"""The seeded input generator: published splitmix64 outputs, torch/int
agreement, per-index regeneration, distribution shape."""
import numpy as np
import torch

import workloads as w


def test_splitmix64_published_sequence():
    """splitmix64 with state 1234567: the first five outputs of the reference
    generator (state += 0x9E3779B97F4A7C15, output = finaliser(state))."""
    s = 1234567
    out = []
    for _ in range(5):
        s = (s + w.GAMMA) & w.MASK64
        out.append(w.mix_int(s))
    assert out == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_torch_bits_match_python_ints():
    idx = torch.tensor([0, 1, 2, 1000, 2 ** 31 - 1, 2 ** 33 + 5], dtype=torch.int64)
    for seed, rank in [(w.seed_of(0), 0), (w.seed_of(3), 63)]:
        got = w.element_bits(seed, rank, idx)
        k = w.stream_key(seed, rank)
        for j, i in enumerate(idx.tolist()):
            ref = w.mix_int(k + (i + 1) * w.GAMMA)
            assert (int(got[j]) & w.MASK64) == ref


def test_sampled_regeneration_matches_fill():
    for dist, dtype in [(("uniform", -1.0, 1.0), "float32"), (("normal", 1e-2), "bfloat16"),
                        (("uniform_int", -(1 << 20), 21), "int32"), (("normal", 1.0), "float32"),
                        (("uniform", -1e3, 1e3), "float32")]:
        _, rows = w.make_inputs(3, 5000, dtype, dist, 77)
        idx = torch.tensor([0, 1, 17, 4095, 4999])
        s = w.sample_inputs(77, 3, idx, dist, dtype)
        for r in range(3):
            assert torch.equal(rows[r][idx], s[r])


def test_distribution_shapes():
    idx = torch.arange(200000)
    z = w.rank_values(1, 0, idx, ("normal", 1.0), "float32").double()
    assert abs(z.mean().item()) < 0.01 and abs(z.std().item() - 1.0) < 0.01
    u = w.rank_values(1, 1, idx, ("uniform", -1.0, 1.0), "float32")
    assert u.min().item() >= -1.0 and u.max().item() < 1.0
    assert abs(u.double().mean().item()) < 0.01
    i = w.rank_values(1, 2, idx, ("uniform_int", -(1 << 20), 21), "int32")
    assert i.min().item() >= -(1 << 20) and i.max().item() < (1 << 20)
    b = w.rank_values(1, 3, idx, ("normal", 1e-2), "bfloat16").double()
    assert abs(b.std().item() - 1e-2) < 2e-4


def test_rows_aligned_for_vector_access():
    big, rows = w.alloc_ranks(4, 4099, "float32", "cpu")
    assert big.shape[1] % 64 == 0
    assert all(r.numel() == 4099 for r in rows)
