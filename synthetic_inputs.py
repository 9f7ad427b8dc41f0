"""Seeded synthetic inputs for the virtual-rank collectives.

This module only makes input buffers; it holds none of the reduction
arithmetic, and both the oracle's tests and the CUDA path's tests and bench
draw their inputs from it.

Host generator: counter-based.  Element i of rank r is a function of
(seed, r, i) alone -- the splitmix64 output function (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) applied to a
per-rank key plus (i + 1) times the golden-ratio increment -- so any slice of
any rank can be regenerated without the rest.

Device generator (for buffers too large to build on the host): torch's own
seeded CUDA generator.  Its values differ from the host generator's; every
check reads the device bytes back, so that difference never matters.

Distributions (the shapes of the workloads the pages and the configurations
describe):
  rank_linear   x^(r)_i = 100 r + i  (the pages' four-rank worked example)
  uniform_pm1   k * 2^-23 - 1 with k uniform in [0, 2^24): uniform on [-1, 1),
                every value a multiple of 2^-23 (so exact sums are integers
                after scaling by 2^23)
  normal        Box-Muller in double, sigma given, rounded to the dtype
  uniform_int   integers uniform in [lo, hi]
No generator produces NaN, infinities or negative zero.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

NP_STORAGE = {"int32": np.int32, "int64": np.int64, "float32": np.float32,
              "bfloat16": np.uint16}


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _key(seed: int, rank: int) -> np.uint64:
    base = np.array([(seed * 0x2545F4914F6CDD1D + rank * 0xD1B54A32D192ED03 + 1)
                     & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(base)[0]


def random_bits(seed: int, rank: int, start: int, count: int, stream: int = 0) -> np.ndarray:
    """64 random bits for elements start .. start+count-1 of one rank."""
    key = _key(seed + 7919 * stream, rank)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + ctr * GOLDEN)


def _f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 bits, nearest-even (finite inputs only)."""
    u = f.astype(np.float32).view(np.uint32).astype(np.uint64)
    lower = u & np.uint64(0xFFFF)
    upper = u >> np.uint64(16)
    up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    return (upper + up.astype(np.uint64)).astype(np.uint16)


def _no_negative_zero(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "float32":
        a[a == 0] = np.float32(0.0)
    elif dtype == "bfloat16":
        a[a == 0x8000] = 0
    return a


def generate_rank(dtype: str, dist: str, seed: int, rank: int, M: int, start: int = 0,
                  **params) -> np.ndarray:
    """Elements start .. start+M-1 of rank ``rank`` (numpy storage array;
    bfloat16 as raw uint16 bits)."""
    if dist == "rank_linear":
        vals = 100 * rank + np.arange(start, start + M, dtype=np.int64)
        return _cast_exact(vals, dtype)
    if dist == "uniform_pm1":
        k = (random_bits(seed, rank, start, M) >> np.uint64(40)).astype(np.int64)
        f = (k.astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)
        if dtype == "float32":
            return _no_negative_zero(f, dtype)
        if dtype == "bfloat16":
            return _no_negative_zero(_f32_to_bf16_bits(f), dtype)
        raise ValueError("uniform_pm1 is a float distribution")
    if dist == "normal":
        sigma = float(params.get("sigma", 1.0))
        b1 = random_bits(seed, rank, start, M, stream=1)
        b2 = random_bits(seed, rank, start, M, stream=2)
        u1 = ((b1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (b2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * sigma
        f = z.astype(np.float32)
        if dtype == "float32":
            return _no_negative_zero(f, dtype)
        if dtype == "bfloat16":
            return _no_negative_zero(_f32_to_bf16_bits(f), dtype)
        raise ValueError("normal is a float distribution")
    if dist == "uniform_int":
        lo, hi = int(params["lo"]), int(params["hi"])
        span = np.uint64(hi - lo + 1)
        v = (random_bits(seed, rank, start, M) % span).astype(np.int64) + lo
        if dtype in ("float32", "bfloat16"):
            return _cast_exact(v, dtype)
        return v.astype(NP_STORAGE[dtype])
    raise ValueError(dist)


def _cast_exact(vals: np.ndarray, dtype: str) -> np.ndarray:
    if dtype in ("int32", "int64"):
        return vals.astype(NP_STORAGE[dtype])
    f = vals.astype(np.float32)
    if dtype == "float32":
        return _no_negative_zero(f, dtype)
    return _no_negative_zero(_f32_to_bf16_bits(f), dtype)


def generate(dtype: str, dist: str, n: int, M: int, seed: int, **params) -> list:
    """N host buffers of M elements each."""
    return [generate_rank(dtype, dist, seed, r, M, **params) for r in range(n)]


def generate_device(torch, dtype: str, dist: str, n: int, M: int, seed: int, device,
                    **params) -> list:
    """N device buffers of M elements each, made by torch's seeded generator on
    the device (for sizes the host generator would take too long on)."""
    tdt = {"int32": torch.int32, "int64": torch.int64, "float32": torch.float32,
           "bfloat16": torch.bfloat16}[dtype]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for r in range(n):
        if dist == "rank_linear":
            t = (100 * r + torch.arange(M, device=device, dtype=torch.int64)).to(tdt)
        elif dist == "uniform_pm1":
            k = torch.randint(0, 1 << 24, (M,), generator=g, device=device, dtype=torch.int32)
            t = (k.to(torch.float32) * (2.0 ** -23) - 1.0).to(tdt)
        elif dist == "normal":
            sigma = float(params.get("sigma", 1.0))
            t = (torch.randn(M, generator=g, device=device, dtype=torch.float32) * sigma).to(tdt)
        elif dist == "uniform_int":
            lo, hi = int(params["lo"]), int(params["hi"])
            t = torch.randint(lo, hi + 1, (M,), generator=g, device=device,
                              dtype=torch.int64).to(tdt)
        else:
            raise ValueError(dist)
        if tdt in (torch.float32, torch.bfloat16):
            t = t + 0.0  # -0 + 0 = +0: no negative zeros
        out.append(t.contiguous())
    return out


# Seeds: one per workload, 20261202 + its index in the workload list below.
SEED_BASE = 20261202

WORKLOADS = {
    # four ranks, twenty int64, x = 100 r + i (the pages' worked example)
    "worked_example_n4_m20_int64": dict(n=4, M=20, dtype="int64", dist="rank_linear",
                                        seed=SEED_BASE + 0),
    # eight ranks, 1,000,003 fp32 uniform[-1,1) (q = 125,001, five padding slots)
    "n8_m1000003_f32_uniform": dict(n=8, M=1_000_003, dtype="float32", dist="uniform_pm1",
                                    seed=SEED_BASE + 1),
    # eight ranks, one 25 MiB gradient bucket of bf16 normal(0, 1e-3)
    "n8_bucket25mib_bf16_normal": dict(n=8, M=13_107_200, dtype="bfloat16", dist="normal",
                                       sigma=1e-3, seed=SEED_BASE + 2),
    # four ranks, 256 MiB fp32 normal(0, 1) each
    "n4_256mib_f32_normal": dict(n=4, M=67_108_864, dtype="float32", dist="normal",
                                 sigma=1.0, seed=SEED_BASE + 3),
    # four ranks, the same element count in int64 uniform[-2^20, 2^20)
    "n4_m67108864_i64_uniform": dict(n=4, M=67_108_864, dtype="int64", dist="uniform_int",
                                     lo=-(1 << 20), hi=(1 << 20) - 1, seed=SEED_BASE + 3),
}


# The smallest per-rank size at which the fused AllReduce and the
# ReduceScatter are to hold 80 % of the copy peak; the sweep measures it too,
# although 8 KiB * 4^k steps over it.
TARGET_BYTES_PER_RANK = 64 << 20


def sweep_points(max_total_bytes: int = 64 << 30):
    """The size x rank-count sweep: per-rank bytes 8 KiB * 4^k (k = 0..8) and
    1 GiB, plus the 64 MiB target point, N in {2, 4, 8, 16, 64}, keeping
    N * bytes <= 64 GiB."""
    sizes = sorted([8192 * 4 ** k for k in range(9)] + [TARGET_BYTES_PER_RANK, 1 << 30])
    pts = []
    for nbytes in sizes:
        for n in (2, 4, 8, 16, 64):
            if n * nbytes <= max_total_bytes:
                pts.append((n, nbytes))
    return pts
