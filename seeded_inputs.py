"""Seeded synthetic inputs for the scan and compaction workloads.

This module only draws random numbers.  It holds none of the scan or
compaction arithmetic, so both the CPU oracle's tests and the GPU parity
tests / benchmark can use it without sharing any of the method's code.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: element i of stream
`seed` is ``mix(key + (i + 1) * GAMMA)`` with ``key = mix(seed + GAMMA)``.
Every value depends only on (seed, i), so any index range can be drawn on its
own and a sample of a large workload is the prefix of the full one.

Distributions (all derived from the 64-bit word ``x`` with integer steps, so
the same bits come out on every machine):

* uniform integers in [lo, hi]:  ``lo + ((x >> 32) * (hi - lo + 1)) >> 32``
* uniform fp32 in [0, 1):        ``(x >> 40) * 2**-24`` (exact in fp32)
* uniform uint32 (full range):   ``x >> 32``
* Bernoulli(p) keep flags:       ``(x >> 32) < round(p * 2**32)`` as uint8 0/1
* Poisson(lam) counts:           inversion of the 53-bit uniform ``x >> 11``
  against the CDF table ``floor(F(k) * 2**53)``, F built by the
  recurrence p_0 = exp(-lam), p_k = p_{k-1} * lam / k in float64.

The workloads (sizes and value ranges) follow the pages: uniform integers in
[0, 9] at ten million elements ("Prefix sum and other parallel patterns",
scan.cu harness), fp32 at 1M / 10M / 100M elements ("Parallel Prefix Sum
(Scan) for NVIDIA T4 (sm_75)", Performance), structured exact floats ("The
CUDA scan algorithm: the tree and the three kernels", Measuring three scans;
"CUDA prefix sum, the Hillis-Steele scan", What the program checks).
"""

from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30 = np.uint64(30)
_S27 = np.uint64(27)
_S31 = np.uint64(31)

# Elements drawn per numpy pass; bounds the temporary uint64 arrays.
_CHUNK = 1 << 24


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, in place on a uint64 array."""
    z ^= z >> _S30
    z *= _M1
    z ^= z >> _S27
    z *= _M2
    z ^= z >> _S31
    return z


def _mix_scalar(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_key(seed: int) -> int:
    return _mix_scalar(int(seed) + int(GAMMA))


def raw_u64(seed: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of stream ``seed`` (uint64)."""
    key = np.uint64(stream_key(seed))
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + idx * GAMMA
    return _mix(z)


def _chunked(n: int, dtype, seed: int, fn) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(raw_u64(seed, s, c))
    return out


def uniform_int32(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Uniform integers in [lo, hi] (inclusive) as int32."""
    r = np.uint64(hi - lo + 1)
    assert 0 < int(r) <= 1 << 32

    def f(x):
        v = ((x >> np.uint64(32)) * r) >> np.uint64(32)
        return (v.astype(np.int64) + lo).astype(np.int32)

    return _chunked(n, np.int32, seed, f)


def uniform_f32(n: int, seed: int) -> np.ndarray:
    """Uniform fp32 in [0, 1): 24 random bits times 2**-24 (exact)."""

    def f(x):
        return ((x >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)).astype(np.float32)

    return _chunked(n, np.float32, seed, f)


def uniform_u32(n: int, seed: int) -> np.ndarray:
    """Uniform uint32 over the full range."""

    def f(x):
        return (x >> np.uint64(32)).astype(np.uint32)

    return _chunked(n, np.uint32, seed, f)


def bernoulli_flags(n: int, p: float, seed: int) -> np.ndarray:
    """uint8 keep flags, 1 with probability p (threshold round(p * 2**32))."""
    thr = np.uint64(min(int(round(p * 2.0 ** 32)), 1 << 32))

    def f(x):
        return ((x >> np.uint64(32)) < thr).astype(np.uint8)

    return _chunked(n, np.uint8, seed, f)


def poisson_cdf_table(lam: float, kmax: int | None = None) -> np.ndarray:
    """Thresholds floor(F(k) * 2**53) for k = 0..kmax (uint64)."""
    if kmax is None:
        kmax = int(lam + 20.0 * math.sqrt(lam) + 20.0)
    p = math.exp(-lam)
    f = p
    out = []
    for k in range(kmax + 1):
        if k > 0:
            p = p * lam / k
            f = f + p
        out.append(min(int(math.floor(f * 2.0 ** 53)), (1 << 53)))
    out[-1] = 1 << 53  # every draw lands at or below kmax
    return np.array(out, dtype=np.uint64)


def poisson_u32(n: int, lam: float, seed: int) -> np.ndarray:
    """Poisson(lam) counts as uint32, by inversion of the 53-bit uniform."""
    table = poisson_cdf_table(lam)

    def f(x):
        u = x >> np.uint64(11)
        # k = number of thresholds <= u  (first k with u < C_k)
        return np.searchsorted(table, u, side="right").astype(np.uint32)

    return _chunked(n, np.uint32, seed, f)


# The five workloads, by what they are.  Sizes are element counts.
def workload_int_0_100(n: int = 4096, seed: int = 0) -> np.ndarray:
    """Single-tile int32 case: uniform integers in [0, 100)."""
    return uniform_int32(n, 0, 99, seed)


def workload_f32_unit(n: int, seed: int = 1) -> np.ndarray:
    """fp32 uniform in [0, 1) at the pages' 1M / 10M / 100M sizes."""
    return uniform_f32(n, seed)


def workload_int_pm1000(n: int, seed: int = 2) -> np.ndarray:
    """int32 uniform in [-1000, 1000] for the size sweep (wraps at large n)."""
    return uniform_int32(n, -1000, 1000, seed)


def workload_compaction(n: int, p: float, seed: int = 3):
    """uint32 keys over the full range and Bernoulli(p) uint8 keep flags.

    Keys and flags come from two disjoint streams of the same seed
    (stream ``2*seed`` and ``2*seed+1``) so they are independent.
    """
    keys = uniform_u32(n, 2 * seed)
    flags = bernoulli_flags(n, p, 2 * seed + 1)
    return keys, flags


def workload_positive_f32(n: int, p: float, seed: int = 5) -> np.ndarray:
    """fp32 uniform in [-(1 - p), p) for the predicate compaction (keep v > 0):
    a fraction of about p is positive.  The [0, 1) draw is shifted by the
    fp32 value nearest 1 - p, in fp32."""
    return (uniform_f32(n, seed) - np.float32(1.0 - p)).astype(np.float32)


def topk_ids(num_tokens: int, top_k: int, num_experts: int, seed: int = 6) -> np.ndarray:
    """Router choices for an MoE layer: int32 [num_tokens, top_k], each row
    top_k distinct experts drawn uniformly from [0, num_experts).

    Column j of every row is drawn as ``((x >> 32) * E) >> 32`` from counter
    range ``[(r * top_k + j) * num_tokens, ...)`` of the stream, redrawing
    (r = 1, 2, ...) the rows where it repeats an earlier column of the row.
    """
    assert 1 <= top_k <= num_experts
    E = np.uint64(num_experts)
    out = np.empty((num_tokens, top_k), dtype=np.int32)
    for j in range(top_k):
        todo = np.arange(num_tokens)
        r = 0
        while todo.size:
            x = raw_u64(seed, (r * top_k + j) * num_tokens, num_tokens)[todo]
            out[todo, j] = (((x >> np.uint64(32)) * E) >> np.uint64(32)).astype(np.int32)
            dup = np.zeros(todo.size, dtype=bool)
            for q in range(j):
                dup |= out[todo, q] == out[todo, j]
            todo = todo[dup]
            r += 1
    return out


def segment_offsets(n: int, mean_len: float, seed: int = 90, empty_frac: float = 0.0) -> np.ndarray:
    """Offsets (uint64, from 0 to n) of segments with lengths uniform in
    [1, 2 * mean_len - 1] (mean mean_len; all 1 when mean_len <= 1), a
    fraction empty_frac of them set to 0.  The last segment ends at n."""
    hi = int(min(max(2.0 * mean_len - 1.0, 1.0), 2.0 ** 31 - 1))
    m = int(n / max(mean_len, 1.0)) + 16
    lens = uniform_int32(m, 1, hi, seed).astype(np.int64)
    if empty_frac > 0.0:
        lens[bernoulli_flags(m, empty_frac, seed + 1) != 0] = 0
    ends = np.cumsum(lens)
    while ends[-1] < n:  # rare: draw more until the lengths cover n
        lens = np.concatenate([lens, uniform_int32(m, 1, hi, seed + len(lens)).astype(np.int64)])
        ends = np.cumsum(lens)
    k = int(np.searchsorted(ends, n, side="left"))
    return np.concatenate([[0], ends[:k], [n]]).astype(np.uint64)


def workload_poisson_counts(n: int, lam: float = 8.0, seed: int = 4) -> np.ndarray:
    """Radix-digit-histogram style counts: Poisson(8) as uint32."""
    return poisson_u32(n, lam, seed)


def structured_i_mod_8(n: int) -> np.ndarray:
    """x_i = (i % 8) + 1 as fp32: every prefix is an exact integer < 2**24."""
    return ((np.arange(n, dtype=np.int64) % 8) + 1).astype(np.float32)


def structured_period4(n: int) -> np.ndarray:
    """x_i = 2.0 where i % 4 == 3, else 1.0 (fp32, exact prefixes)."""
    x = np.ones(n, dtype=np.float32)
    x[3::4] = 2.0
    return x
