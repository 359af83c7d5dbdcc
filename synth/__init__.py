"""Seeded synthetic inputs for the KV-cache eviction path.

This module is shared by the CUDA parity tests, the oracle tests and the
benchmark.  It holds no arithmetic of the eviction method itself: only random
numbers, shapes and the recipes that turn them into Q/K/V tensors, budgets'
means and a layer-sensitivity profile.

Random numbers come from one counter-based generator, written out twice from
the same definition: here in numpy (host) and in ``synth/csrc/synth_gen.cu``
(device, for the multi-GB configurations).  Both produce identical bits,
because every step is integer arithmetic or an exact float operation:

* ``mix64`` is the splitmix64 output function (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014, with Stafford's
  "Mix13" constants as used by splitmix64).
* Element ``e`` of tensor stream ``key`` takes the three words
  ``mix64(key + (3e + i + 1) * PHI)`` for ``i = 0, 1, 2`` (mod 2**64).
* Their twelve 16-bit fields ``u`` give an Irwin-Hall(12) normal deviate
  ``z = (sum(u) - 393210) / 65536`` (mean 0, variance 1 up to 2**-32, support
  [-6, 6]); the integer-to-float conversion and the division by 2**16 are exact.
* A value is ``z * scale`` with ``scale`` a power of two (exact), then rounded
  to bfloat16 with round-to-nearest-even on the float32 bits.

Layouts (all row-major, bfloat16 stored as uint16 bits):

* ``Q_win``: ``[num_requests][num_layers][num_q_heads][window][head_dim]``
* ``K``, ``V``: ``[num_layers][num_kv_heads][N_tot][head_dim]`` with the tokens of
  all requests packed along ``N_tot`` (``cu_seqlens``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

PHI = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1
IH12_CENTER = 393210  # 12 * 32767.5

# stream identifiers
S_Q, S_K, S_V, S_OUTLIER, S_HEAVY, S_LENGTH, S_PROFILE = 1, 2, 3, 4, 5, 6, 7


# --------------------------------------------------------------------------
# counter-based generator
# --------------------------------------------------------------------------
def mix64_int(z: int) -> int:
    """splitmix64 output function on a Python int (mod 2**64)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function, vectorised over a uint64 array (wrapping)."""
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> int:
    return mix64_int(((seed & _MASK64) * PHI + stream) & _MASK64)


def words(key: int, start: int, count: int) -> np.ndarray:
    """``count`` uint64 words ``mix64(key + (start + i + 1) * PHI)``."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    return mix64(idx * np.uint64(PHI) + np.uint64(key))


def uniform01(key: int, start: int, count: int) -> np.ndarray:
    """Float64 uniforms in [0, 1) from the top 53 bits of each word."""
    return (words(key, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normals_chunk(key: int, start: int, count: int) -> np.ndarray:
    return _normals_at(key, np.arange(start, start + count, dtype=np.uint64))


def _normals_at(key: int, e: np.ndarray) -> np.ndarray:
    """Irwin-Hall(12) deviates of the elements with indices ``e`` (any order), float32."""
    e = np.asarray(e, dtype=np.uint64)
    count = e.size
    base = e * np.uint64(3) + np.uint64(1)
    m = np.uint64(0x0000FFFF0000FFFF)
    acc = np.zeros(count, dtype=np.uint64)   # two 32-bit lanes of partial 16-bit sums
    for i in range(3):
        w = mix64((base + np.uint64(i)) * np.uint64(PHI) + np.uint64(key))
        acc += w & m
        w >>= np.uint64(16)
        w &= m
        acc += w
    total = (acc & np.uint64(0xFFFFFFFF)) + (acc >> np.uint64(32))
    return (total.astype(np.int64) - IH12_CENTER).astype(np.float32) * np.float32(1.0 / 65536.0)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import os
        _POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def normals_f32(key: int, start: int, count: int, chunk: int = 1 << 20) -> np.ndarray:
    """Irwin-Hall(12) deviates for elements ``start .. start+count-1``, float32.

    The sum of the twelve 16-bit fields is formed two fields at a time in the
    32-bit halves of a uint64 (each half stays below 2**19), then folded.
    """
    out = np.empty(count, dtype=np.float32)
    spans = [(c0, min(chunk, count - c0)) for c0 in range(0, count, chunk)]

    def work(span):
        c0, c = span
        out[c0:c0 + c] = _normals_chunk(key, start + c0, c)

    if len(spans) <= 1:
        for sp in spans:
            work(sp)
    else:
        list(_pool().map(work, spans))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.

    Finite inputs only (the generators never produce inf or NaN), so the
    uint32 sum below cannot wrap."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _distinct_ints(key: int, counter0: int, lo: int, hi: int, count: int) -> list[int]:
    """``count`` distinct integers in [lo, hi), in draw order, from a uniform stream."""
    span = hi - lo
    if count > span:
        raise ValueError("cannot draw %d distinct values from %d" % (count, span))
    got: list[int] = []
    seen: set[int] = set()
    c = counter0
    while len(got) < count:
        need = count - len(got)
        u = uniform01(key, c, 2 * need + 8)
        c += 2 * need + 8
        for x in np.floor(u * span).astype(np.int64):
            x = int(x) + lo
            if x not in seen:
                seen.add(x)
                got.append(x)
                if len(got) == count:
                    break
    return got


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the eviction path.

    ``budget_ratio`` (fraction of each request's length) or ``budget_tokens``
    (fixed) gives the mean per-head budget B of a request; ``budget_policy``
    says how the per-layer budgets spread around it.
    """
    name: str
    num_layers: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    window: int
    lengths: tuple = ()
    num_sinks: int = 4
    sigma_q: float = 1.0
    sigma_kv: float = 1.0
    num_outliers: int = 4
    outlier_scale: float = 8.0
    num_heavy: int = 64
    heavy_scale: float = 4.0
    budget_policy: str = "uniform"       # uniform | pyramid | ripple
    budget_ratio: Optional[float] = None
    budget_tokens: Optional[int] = None
    pyramid_max: float = 1.8
    pyramid_min: float = 0.2
    ripple_beta: float = 2.0
    ragged_range: Optional[tuple] = None  # (lo, hi, count): lengths drawn U[lo, hi]
    seed: int = 0

    # derived -------------------------------------------------------------
    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows(self) -> int:
        """R = G * w query rows that look at one KV head."""
        return self.group * self.window

    def seq_lengths(self) -> list[int]:
        if self.ragged_range is None:
            return list(self.lengths)
        lo, hi, cnt = self.ragged_range
        u = uniform01(stream_key(self.seed, S_LENGTH), 0, cnt)
        return [lo + int(x) for x in np.floor(u * (hi - lo + 1)).astype(np.int64)]

    @property
    def num_requests(self) -> int:
        return len(self.seq_lengths())

    def cu_seqlens(self) -> np.ndarray:
        n = self.seq_lengths()
        return np.concatenate([[0], np.cumsum(n)]).astype(np.int64)

    @property
    def num_units(self) -> int:
        return self.num_requests * self.num_layers * self.num_kv_heads

    def unit_index(self, r: int, l: int, h: int) -> int:
        return (r * self.num_layers + l) * self.num_kv_heads + h

    def unit_coords(self, u: int) -> tuple:
        h = u % self.num_kv_heads
        l = (u // self.num_kv_heads) % self.num_layers
        r = u // (self.num_kv_heads * self.num_layers)
        return r, l, h

    def mean_budgets(self) -> list[int]:
        """Mean per-head budget B_r of each request (tokens, sinks and window included)."""
        out = []
        for n in self.seq_lengths():
            if self.budget_tokens is not None:
                out.append(int(self.budget_tokens))
            else:
                out.append(int(math.floor(self.budget_ratio * n)))
        return out

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


def ripple_profile(wl: Workload) -> np.ndarray:
    """Seeded non-monotonic layer-sensitivity profile s_l (float64, length L).

    A Gaussian bump centred at l* ~ U(L/4, 3L/4) with width L/6, plus 0.3 x U(0,1)
    per layer.  Stands in for the offline KL-response profile of RippleKV
    (which needs a model and a calibration set).
    """
    L = wl.num_layers
    u = uniform01(stream_key(wl.seed, S_PROFILE), 0, L + 1)
    centre = L / 4.0 + u[0] * (L / 2.0)
    width = max(L / 6.0, 1.0)
    s = np.array([math.exp(-((l - centre) / width) ** 2) + 0.3 * u[l + 1] for l in range(L)])
    return s


def outlier_channels(wl: Workload) -> np.ndarray:
    """int32 [L][H][num_outliers]: channels of each (layer, KV head) scaled by outlier_scale."""
    L, H = wl.num_layers, wl.num_kv_heads
    out = np.zeros((L, H, max(wl.num_outliers, 1)), dtype=np.int32) - 1
    if wl.num_outliers == 0:
        return out[:, :, :0]
    key = stream_key(wl.seed, S_OUTLIER)
    for l in range(L):
        for h in range(H):
            ch = _distinct_ints(key, (l * H + h) * 4096, 0, wl.head_dim, wl.num_outliers)
            out[l, h, :] = sorted(ch)
    return out


def heavy_positions(wl: Workload) -> np.ndarray:
    """int32 [req][L][H][num_heavy]: token positions (within the request) of heavy keys.

    Uniform over the middle candidates [num_sinks, n - window), without replacement.
    """
    L, H = wl.num_layers, wl.num_kv_heads
    lens = wl.seq_lengths()
    out = np.zeros((len(lens), L, H, wl.num_heavy), dtype=np.int32)
    if wl.num_heavy == 0:
        return out
    key = stream_key(wl.seed, S_HEAVY)
    for r, n in enumerate(lens):
        for l in range(L):
            for h in range(H):
                seg = (r * L + l) * H + h
                p = _distinct_ints(key, seg * (1 << 20), wl.num_sinks, n - wl.window, wl.num_heavy)
                out[r, l, h, :] = sorted(p)
    return out


def q_window(wl: Workload) -> np.ndarray:
    """uint16 bf16 bits [req][L][H_q][w][d]: the observation-window queries."""
    shape = (wl.num_requests, wl.num_layers, wl.num_q_heads, wl.window, wl.head_dim)
    cnt = int(np.prod(shape))
    z = normals_f32(stream_key(wl.seed, S_Q), 0, cnt)
    return f32_to_bf16_bits(z * np.float32(wl.sigma_q)).reshape(shape)


def heavy_rows(wl: Workload, q_bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits [req][L][H][d]: the heavy key row of each (request, layer, KV head).

    heavy_scale x (RMS key norm sigma_kv * sqrt(d)) x unit(mean of the group's
    window queries), computed in float64, rounded to float32 then bfloat16.
    """
    R, L, Hq, w, d = q_bits.shape
    H, G = wl.num_kv_heads, wl.group
    q = bf16_bits_to_f32(q_bits).astype(np.float64).reshape(R, L, H, G * w, d)
    mean = q.mean(axis=3)
    norm = np.sqrt((mean * mean).sum(axis=-1, keepdims=True))
    norm = np.where(norm > 0, norm, 1.0)
    vec = (wl.heavy_scale * wl.sigma_kv * math.sqrt(d)) * mean / norm
    return f32_to_bf16_bits(vec.astype(np.float32))


def _channel_scale(wl: Workload, l: int, h: int, outl: np.ndarray) -> np.ndarray:
    sc = np.full(wl.head_dim, np.float32(wl.sigma_kv), dtype=np.float32)
    if wl.num_outliers:
        sc[outl[l, h]] *= np.float32(wl.outlier_scale)
    return sc


def kv_unit(wl: Workload, r: int, l: int, h: int, *, outl=None, heavy_pos=None,
            heavy_vec=None) -> tuple[np.ndarray, np.ndarray]:
    """Host regeneration of one unit's K and V rows: two uint16 arrays [n_r][d].

    Bit-identical to the rows the device generator writes into the packed
    ``[L][H][N_tot][d]`` tensors.
    """
    d = wl.head_dim
    cu = wl.cu_seqlens()
    N_tot = int(cu[-1])
    n = int(cu[r + 1] - cu[r])
    row0 = (l * wl.num_kv_heads + h) * N_tot + int(cu[r])
    if outl is None:
        outl = outlier_channels(wl)
    sc = _channel_scale(wl, l, h, outl)
    out = []
    for sid in (S_K, S_V):
        z = normals_f32(stream_key(wl.seed, sid), row0 * d, n * d).reshape(n, d)
        out.append(f32_to_bf16_bits(z * sc[None, :]))
    k, v = out
    if wl.num_heavy:
        if heavy_pos is None:
            heavy_pos = heavy_positions(wl)
        if heavy_vec is None:
            heavy_vec = heavy_rows(wl, q_window(wl))
        k[heavy_pos[r, l, h]] = heavy_vec[r, l, h]
    return k, v


def kv_rows(wl: Workload, r: int, l: int, h: int, rows, *, outl=None, heavy_pos=None,
            heavy_vec=None) -> tuple[np.ndarray, np.ndarray]:
    """Host regeneration of chosen K and V rows of one unit: ``rows`` are token indices
    within request r; returns two uint16 arrays [len(rows)][d], bit-identical to
    ``kv_unit(wl, r, l, h)[i][rows]`` without generating the whole unit."""
    d = wl.head_dim
    cu = wl.cu_seqlens()
    N_tot = int(cu[-1])
    row0 = (l * wl.num_kv_heads + h) * N_tot + int(cu[r])
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    if outl is None:
        outl = outlier_channels(wl)
    sc = _channel_scale(wl, l, h, outl)
    e = ((row0 + rows)[:, None] * d + np.arange(d, dtype=np.int64)[None, :]).reshape(-1)
    out = []
    for sid in (S_K, S_V):
        z = _normals_at(stream_key(wl.seed, sid), e.astype(np.uint64)).reshape(rows.size, d)
        out.append(f32_to_bf16_bits(z * sc[None, :]))
    k, v = out
    if wl.num_heavy:
        if heavy_pos is None:
            heavy_pos = heavy_positions(wl)
        if heavy_vec is None:
            heavy_vec = heavy_rows(wl, q_window(wl))
        k[np.isin(rows, heavy_pos[r, l, h])] = heavy_vec[r, l, h]
    return k, v


def kv_full_host(wl: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Whole packed K, V on the host (small workloads only): uint16 [L][H][N_tot][d]."""
    cu = wl.cu_seqlens()
    N_tot = int(cu[-1])
    L, H, d = wl.num_layers, wl.num_kv_heads, wl.head_dim
    K = np.empty((L, H, N_tot, d), dtype=np.uint16)
    V = np.empty_like(K)
    outl = outlier_channels(wl)
    hp = heavy_positions(wl)
    hv = heavy_rows(wl, q_window(wl)) if wl.num_heavy else None
    for r in range(wl.num_requests):
        for l in range(L):
            for h in range(H):
                k, v = kv_unit(wl, r, l, h, outl=outl, heavy_pos=hp, heavy_vec=hv)
                K[l, h, cu[r]:cu[r + 1]] = k
                V[l, h, cu[r]:cu[r + 1]] = v
    return K, V


# --------------------------------------------------------------------------
# the five configurations of the benchmark description, and small variants
# --------------------------------------------------------------------------
TINY = Workload("tiny_1L_gqa4_d64_n2048", num_layers=1, num_kv_heads=1, num_q_heads=4,
                head_dim=64, window=16, lengths=(2048,), sigma_q=0.125, sigma_kv=0.125,
                num_outliers=0, num_heavy=8, budget_tokens=256)
LLAMA8B_32K = Workload("llama8b_32L_8kv_32q_d128_n32768", num_layers=32, num_kv_heads=8,
                       num_q_heads=32, head_dim=128, window=32, lengths=(32768,),
                       budget_ratio=0.05)
LONG_128K = Workload("long_32L_8kv_32q_d128_n131072_pyramid10", num_layers=32, num_kv_heads=8,
                     num_q_heads=32, head_dim=128, window=64, lengths=(131072,),
                     budget_ratio=0.10, budget_policy="pyramid")
QWEN7B_128K = Workload("qwen7b_28L_4kv_28q_d128_n131072_ripple5", num_layers=28, num_kv_heads=4,
                       num_q_heads=28, head_dim=128, window=64, lengths=(131072,),
                       budget_ratio=0.05, budget_policy="ripple")
RAGGED_MISTRAL = Workload("ragged8_mistral7b_32L_8kv_32q_d128_n16k-128k", num_layers=32,
                          num_kv_heads=8, num_q_heads=32, head_dim=128, window=32,
                          ragged_range=(16384, 131072, 8), budget_ratio=0.30)

CONFIGS = [TINY, LLAMA8B_32K, LONG_128K, QWEN7B_128K, RAGGED_MISTRAL]
# Reduced copies for kernel profiles: the same per-unit shapes, few units
# (K+V still larger than L2, a few GB on the device at most).
PROFILE_CASES = [
    LONG_128K.scaled(name="long_2L_2kv_8q_d128_n131072_pyramid10", num_layers=2,
                     num_kv_heads=2, num_q_heads=8),
    QWEN7B_128K.scaled(name="qwen7b_2L_2kv_14q_d128_n131072_ripple5", num_layers=2,
                       num_kv_heads=2, num_q_heads=14),
    LLAMA8B_32K.scaled(name="llama8b_2L_8kv_32q_d128_n32768", num_layers=2),
    RAGGED_MISTRAL.scaled(name="ragged8_mistral7b_2L_2kv_8q_d128_n16k-128k", num_layers=2,
                          num_kv_heads=2, num_q_heads=8),
]
BY_NAME = {c.name: c for c in CONFIGS + PROFILE_CASES}


def small_variant(wl: Workload, n: int, layers: int = 2, kv_heads: int = 2,
                  requests: Optional[list] = None, seed: int = 7) -> Workload:
    """A reduced copy of ``wl`` that the oracle finishes in seconds (same d, G, w, policy)."""
    G = wl.group
    kw = dict(name=wl.name + "_small", num_layers=min(layers, wl.num_layers),
              num_kv_heads=min(kv_heads, wl.num_kv_heads),
              num_q_heads=min(kv_heads, wl.num_kv_heads) * G, seed=seed,
              num_heavy=min(wl.num_heavy, 8))
    if requests is not None:
        kw.update(lengths=tuple(requests), ragged_range=None)
    else:
        kw.update(lengths=(n,), ragged_range=None)
    return replace(wl, **kw)
