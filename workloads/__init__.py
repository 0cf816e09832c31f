"""Seeded synthetic workloads for the ring all-reduce.

This module is the one piece shared by the CUDA side and the oracle side: it
makes the input buffers and nothing else (none of the method's arithmetic
lives here).  Every value is a pure function of (seed, rank, element index),
computed with integer operations and single IEEE binary32 operations in
torch, so the same call gives the same bits on the CPU and on a GPU, and any
sampled element can be regenerated on its own.

Generator (all arithmetic modulo 2^64):
  * splitmix64 finaliser (S. Vigna, "splitmix64.c"): z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
    z ^= z >> 31.
  * stream key  K = mix(seed * 2^16 + rank + 1)
  * element bits  B(i) = mix(K + (i + 1) * 0x9E3779B97F4A7C15)
Distributions:
  * uniform[lo, hi) binary32: u = (B >> 40) * 2^-24 (exact), value =
    lo + u * (hi - lo), two binary32 operations;
  * uniform integers [lo, lo + 2^k): lo + (B >> (64 - k));
  * normal N(0, sigma) (sigma is the standard deviation): inverse-CDF table
    of 2^16 + 1 binary32 knots of the standard normal, q_k = Phi^-1(k / 2^16)
    for 0 < k < 2^16 with the end knots at Phi^-1(2^-17) and
    Phi^-1(1 - 2^-17); k = B >> 48, f = ((B >> 24) & (2^24 - 1)) * 2^-24,
    value = (q_k + (q_(k+1) - q_k) * f) * sigma, each step one binary32
    operation; 16-bit types are then rounded to nearest even by torch.
"""
from __future__ import annotations

import functools
import statistics

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

SEED_BASE = 0x5241520000

TORCH_DTYPES = {"int32": torch.int32, "float32": torch.float32,
                "bfloat16": torch.bfloat16, "float16": torch.float16}


def _s64(v: int) -> int:
    """A 64-bit pattern as the signed int64 torch stores."""
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(M1)
    z = (z ^ _lsr(z, 27)) * _s64(M2)
    return z ^ _lsr(z, 31)


def mix_int(v: int) -> int:
    """The splitmix64 finaliser on a Python int (reference for tests)."""
    z = v & MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, rank: int) -> int:
    return mix_int((seed << 16) + rank + 1)


def element_bits(seed: int, rank: int, idx: torch.Tensor) -> torch.Tensor:
    """64 random bits per element index (int64 tensor, any device)."""
    k = _s64(stream_key(seed, rank))
    z = (idx.to(torch.int64) + 1) * _s64(GAMMA) + k
    return _mix(z)


@functools.lru_cache(maxsize=None)
def _normal_knots_cpu():
    nd = statistics.NormalDist()
    K = 1 << 16
    q = [nd.inv_cdf(2.0 ** -17)]
    q += [nd.inv_cdf(k / K) for k in range(1, K)]
    q.append(nd.inv_cdf(1.0 - 2.0 ** -17))
    t = torch.tensor(q, dtype=torch.float64).to(torch.float32)
    d = t[1:] - t[:-1]           # binary32 differences
    return t[:-1].contiguous(), d.contiguous()


_knot_cache: dict = {}


def _normal_knots(device):
    key = str(device)
    if key not in _knot_cache:
        t, d = _normal_knots_cpu()
        _knot_cache[key] = (t.to(device), d.to(device))
    return _knot_cache[key]


def values_from_bits(bits: torch.Tensor, dist: tuple, dtype: str) -> torch.Tensor:
    """Map 64-bit patterns to values of `dist` in `dtype` (same device)."""
    kind = dist[0]
    if kind == "uniform_int":
        lo, log2_range = dist[1], dist[2]
        v = _lsr(bits, 64 - log2_range) + lo
        return v.to(torch.int32)
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        u = _lsr(bits, 40).to(torch.float32) * (2.0 ** -24)
        v = u * torch.tensor(hi - lo, dtype=torch.float32) + torch.tensor(lo, dtype=torch.float32)
    elif kind == "normal":
        sigma = dist[1]
        t, d = _normal_knots(bits.device)
        k = _lsr(bits, 48)
        f = (_lsr(bits, 24) & ((1 << 24) - 1)).to(torch.float32) * (2.0 ** -24)
        z = t[k] + d[k] * f
        v = z * torch.tensor(sigma, dtype=torch.float32)
    elif kind == "const":
        v = torch.full(bits.shape, float(dist[1]), dtype=torch.float32, device=bits.device)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return v.to(TORCH_DTYPES[dtype])


def rank_values(seed: int, rank: int, idx: torch.Tensor, dist: tuple, dtype: str) -> torch.Tensor:
    """Rank `rank`'s input at element indices idx."""
    return values_from_bits(element_bits(seed, rank, idx), dist, dtype)


def fill_rank(out: torch.Tensor, seed: int, rank: int, dist: tuple, dtype: str,
              block: int = 1 << 26) -> None:
    """Fill a 1-D tensor with rank `rank`'s inputs, in blocks (any device)."""
    n = out.numel()
    for lo in range(0, n, block):
        hi = min(n, lo + block)
        idx = torch.arange(lo, hi, dtype=torch.int64, device=out.device)
        out[lo:hi] = rank_values(seed, rank, idx, dist, dtype)


def sample_inputs(seed: int, p: int, idx: torch.Tensor, dist: tuple, dtype: str) -> torch.Tensor:
    """(p, m) CPU tensor of every rank's input at the sampled indices."""
    idx = idx.to("cpu", torch.int64)
    return torch.stack([rank_values(seed, r, idx, dist, dtype) for r in range(p)])


# --------------------------------------------------------------- workloads
#
# The pages' workloads, as seeded synthetic buffers (seed = SEED_BASE + the
# workload's index below).  "N(0, s)" is read with s as the standard
# deviation.

def page_trace_inputs(p: int = 4, n: int = 4):
    """"Ring All-Reduce, in depth", "Tracing four GPUs": rank r holds
    (r + 1) * [1, 10, 100, 1000]."""
    base = [1.0, 10.0, 100.0, 1000.0][:n]
    return [[(r + 1) * v for v in base] for r in range(p)]


WORKLOADS = {
    # p = 4, N = 4,099 fp32 (chunks 1025/1025/1025/1024), uniform[-1, 1), sum
    "p4_n4099_f32": dict(index=0, p=4, n=4099, dtype="float32",
                         dist=("uniform", -1.0, 1.0), ops=("sum",)),
    # p = 8, N = 6,553,600 fp32 (one 25 MB gradient bucket), N(0, 1e-3), sum and avg
    "p8_n6553600_f32": dict(index=1, p=8, n=6553600, dtype="float32",
                            dist=("normal", 1e-3), ops=("sum", "avg")),
    # p = 8, N = 2^30 bf16 (2 GiB per rank, 16 GiB total), N(0, 1e-2), sum
    "p8_n1073741824_bf16": dict(index=2, p=8, n=1 << 30, dtype="bfloat16",
                                dist=("normal", 1e-2), ops=("sum",)),
    # p = 64, N = 2^24 bf16 (32 MiB per rank, 2 GiB total), N(0, 1e-2), sum
    "p64_n16777216_bf16": dict(index=3, p=64, n=1 << 24, dtype="bfloat16",
                               dist=("normal", 1e-2), ops=("sum",)),
}

# p = 16 message-size sweep, N = 4^5 .. 4^13, three dtype/op pairs
SWEEP_P = 16
SWEEP_SIZES = tuple(4 ** k for k in range(5, 14))
SWEEP_PAIRS = (
    ("int32", "sum", ("uniform_int", -(1 << 20), 21)),
    ("float32", "max", ("uniform", -1e3, 1e3)),
    ("float32", "avg", ("normal", 1.0)),
)
SWEEP_INDEX = 4


def seed_of(index: int) -> int:
    return SEED_BASE + index


def alloc_ranks(p: int, n: int, dtype: str, device, align_elems: int = 64) -> tuple:
    """One [p, n_pad] tensor (rows 256-byte aligned when n_pad*e allows) and
    its p row views of length n."""
    n_pad = max(align_elems, ((n + align_elems - 1) // align_elems) * align_elems)
    big = torch.empty((p, n_pad), dtype=TORCH_DTYPES[dtype], device=device)
    return big, [big[r, :n] for r in range(p)]


def make_inputs(p: int, n: int, dtype: str, dist: tuple, seed: int, device="cpu") -> tuple:
    """Allocate and fill p rank buffers; returns (storage, row views)."""
    big, rows = alloc_ranks(p, n, dtype, device)
    for r in range(p):
        fill_rank(rows[r], seed, r, dist, dtype)
    return big, rows


def to_storage_numpy(t: torch.Tensor):
    """A CPU tensor as the numpy storage form the oracle takes (bf16/f16 as
    raw uint16 patterns)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
