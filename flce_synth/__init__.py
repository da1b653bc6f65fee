"""Seeded synthetic inputs for the fused linear cross-entropy path.

This module only draws numbers: it holds none of the loss arithmetic, so the
CPU oracle (``oracle/``) and the CUDA library both consume exactly the same
tensors without sharing any code of the method itself.

Generator (portable between x86-64 and aarch64, independent of numpy/torch RNG
streams): element ``k`` of stream ``s`` is SplitMix64 evaluated at counter
``k`` of a stream key derived from ``(seed, s)``:

    z_k = mix64(key_s + (k + 1) * 0x9E3779B97F4A7C15)
    mix64(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
               z *= 0x94D049BB133111EB; z ^= z >> 31

(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014).  Uniforms are ``((z >> 11) + 0.5) * 2**-53`` in (0, 1).
Normals use the Box-Muller transform on the uniform pair (2j, 2j+1): element
2j takes the cosine branch and 2j+1 the sine branch.  Values are formed in
float64, rounded to float32 (round-to-nearest-even) and, for bf16 inputs,
rounded again float32 -> bf16 (round-to-nearest-even).

Targets: uniform draws ``floor(u * V)``; Zipf(s) draws rank r in [1, V] with
P(r) proportional to r**-s by inverse CDF over a float64 table, then maps it
through a seeded permutation of the vocabulary (argsort of SplitMix64 keys).
Exactly ``floor(p * N)`` positions, chosen by a seeded permutation of the
rows, are set to the ignore index.

The workload shapes follow the pages' low-level API example
(``nn.Linear(128, 256)``, ``randn(4, 128)``, ``randint(256, (4,))`` in the
Liger-Kernel project overview, "Método de API de Baixo Nível") and the model
heads the overview lists (Llama-3, Qwen2; "Arquiteturas de Modelo
Suportadas"), as synthetic stand-ins for the checkpoints and datasets named
there, which are not used.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per worker task (even, so Box-Muller pairs never split)

# stream ids inside one seed
STREAM_X, STREAM_W, STREAM_T, STREAM_PERM_V, STREAM_PERM_N = 1, 2, 3, 4, 5


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of stream ``stream`` under ``seed`` (one mix of seed*256+stream)."""
    v = np.array([(int(seed) * 256 + int(stream)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix64(v)[0]


def splitmix64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs for counters ``start .. start+count-1``."""
    k = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + (k + np.uint64(1)) * _GAMMA
    return _mix64(z)


def uniform(key: np.uint64, start: int, count: int) -> np.ndarray:
    z = splitmix64(key, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def _normal_block(key: np.uint64, start: int, count: int) -> np.ndarray:
    """float64 normals for elements start .. start+count-1 (start even)."""
    assert start % 2 == 0
    npair = (count + 1) // 2
    u = uniform(key, start, 2 * npair)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    out = np.empty(2 * npair, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:count]


def _fill(out: torch.Tensor, fn, key: np.uint64, start: int, threads: int | None) -> None:
    """Fill the flat tensor ``out`` with fn(key, start+i, n) in parallel chunks."""
    flat = out.view(-1)
    n = flat.numel()
    if n == 0:
        return
    bounds = [(i, min(n, i + _CHUNK)) for i in range(0, n, _CHUNK)]

    def work(b):
        lo, hi = b
        vals = fn(key, start + lo, hi - lo).astype(np.float32)
        flat[lo:hi].copy_(torch.from_numpy(vals).to(flat.dtype))

    nthreads = threads or min(len(bounds), os.cpu_count() or 1)
    if nthreads <= 1 or len(bounds) == 1:
        for b in bounds:
            work(b)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(work, bounds))


def normal_tensor(shape, std: float, seed: int, stream: int, dtype: torch.dtype,
                  row_offset: int = 0, threads: int | None = None) -> torch.Tensor:
    """N(0, std^2) values; row r of the result is row (row_offset + r) of the
    infinite stream, so a prefix of rows can be drawn without the rest."""
    key = stream_key(seed, stream)
    out = torch.empty(shape, dtype=dtype)
    cols = shape[-1] if len(shape) > 1 else 1
    start = row_offset * cols
    if start % 2:
        raise ValueError("row_offset * cols must be even")
    if std == 1.0:
        fn = _normal_block
    else:
        fn = lambda k, s, c: _normal_block(k, s, c) * std  # noqa: E731
    _fill(out, fn, key, start, threads)
    return out


def uniform_tensor(shape, lo: float, hi: float, seed: int, stream: int,
                   dtype: torch.dtype, threads: int | None = None) -> torch.Tensor:
    key = stream_key(seed, stream)
    out = torch.empty(shape, dtype=dtype)
    _fill(out, lambda k, s, c: lo + (hi - lo) * uniform(k, s, c), key, 0, threads)
    return out


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    """Seeded permutation of range(n): stable argsort of SplitMix64 keys."""
    keys = splitmix64(stream_key(seed, stream), 0, n)
    return np.argsort(keys, kind="stable").astype(np.int64)


def targets(n: int, vocab: int, dist: str, seed: int, ignore_num: int = 0,
            ignore_den: int = 100, ignore_index: int = -100,
            zipf_s: float = 1.1) -> np.ndarray:
    """Target ids [n] int64: 'uniform' or 'zipf', with exactly
    floor(n * ignore_num / ignore_den) positions set to ``ignore_index``."""
    u = uniform(stream_key(seed, STREAM_T), 0, n)
    if dist == "uniform":
        t = np.minimum(np.floor(u * vocab).astype(np.int64), vocab - 1)
    elif dist == "zipf":
        ranks = np.arange(1, vocab + 1, dtype=np.float64)
        cdf = np.cumsum(ranks ** (-zipf_s))
        cdf /= cdf[-1]
        idx = np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1)
        perm = permutation(vocab, seed, STREAM_PERM_V)
        t = perm[idx]
    else:
        raise ValueError(f"unknown target distribution {dist!r}")
    n_ign = (n * ignore_num) // ignore_den
    if n_ign:
        pos = permutation(n, seed, STREAM_PERM_N)[:n_ign]
        t = t.copy()
        t[pos] = ignore_index
    return t.astype(np.int64)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and the input recipe."""
    name: str
    N: int
    H: int
    V: int
    dtype: str                 # "bf16" or "fp32"
    seed: int
    w_dist: str                # "normal0.02" or "linear_init" (U(-1/sqrt(H), 1/sqrt(H)))
    t_dist: str                # "uniform" or "zipf"
    ignore_num: int = 0        # ignored fraction = ignore_num / 100
    ignore_index: int = -100
    note: str = field(default="", compare=False)

    @property
    def n_ignored(self) -> int:
        return (self.N * self.ignore_num) // 100

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_worked_4x128x256_fp32", 4, 128, 256, "fp32", 1000,
                 "linear_init", "uniform", 0,
                 note="the overview's nn.Linear(128,256) / randn(4,128) example"),
        Workload("small_head_2048x2048x32000", 2048, 2048, 32000, "bf16", 1001,
                 "normal0.02", "uniform", 5),
        Workload("llama3_8b_head_8192x4096x128256", 8192, 4096, 128256, "bf16", 1002,
                 "normal0.02", "zipf", 2),
        Workload("qwen2_7b_head_16384x3584x152064", 16384, 3584, 152064, "bf16", 1003,
                 "normal0.02", "uniform", 10),
        Workload("long_context_65536x4096x128256", 65536, 4096, 128256, "bf16", 1004,
                 "normal0.02", "zipf", 1),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def make_inputs(w: Workload, rows: int | None = None, threads: int | None = None):
    """(X [rows, H], W [V, H], target [rows] int64) as CPU torch tensors.

    ``rows`` < N draws the first ``rows`` tokens of the full workload (the same
    values the full draw has in those rows)."""
    n = w.N if rows is None else rows
    dt = w.torch_dtype
    X = normal_tensor((n, w.H), 1.0, w.seed, STREAM_X, dt, threads=threads)
    if w.w_dist == "normal0.02":
        W = normal_tensor((w.V, w.H), 0.02, w.seed, STREAM_W, dt, threads=threads)
    elif w.w_dist == "linear_init":
        b = 1.0 / math.sqrt(w.H)
        W = uniform_tensor((w.V, w.H), -b, b, w.seed, STREAM_W, dt, threads=threads)
    else:
        raise ValueError(w.w_dist)
    t_full = targets(w.N, w.V, w.t_dist, w.seed, w.ignore_num, 100, w.ignore_index)
    t = torch.from_numpy(t_full[:n].copy())
    return X, W, t


def make_case(N: int, H: int, V: int, dtype: str = "bf16", seed: int = 7,
              w_std: float = 0.02, t_dist: str = "uniform", ignore_num: int = 0,
              ignore_index: int = -100, x_std: float = 1.0):
    """Arbitrary-size case with the same recipe (used for ragged/edge tests)."""
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    X = normal_tensor((N, H), x_std, seed, STREAM_X, dt)
    W = normal_tensor((V, H), w_std, seed, STREAM_W, dt)
    t = torch.from_numpy(targets(N, V, t_dist, seed, ignore_num, 100, ignore_index))
    return X, W, t
