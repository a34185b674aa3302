"""Seeded synthetic inputs for the dense GEMM C = alpha*A*B + beta*C.

This module only draws random numbers and rounds them to the storage type of
an operand. It holds none of the GEMM arithmetic, so the CPU oracle and the
GPU path can both take their inputs from here without sharing any of the
method's code.

Generator
---------
A counter-based splitmix64.  The splitmix64 step (Steele, Lea, Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) is

    state += 0x9E3779B97F4A7C15
    z = state
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    return z ^ (z >> 31)

so the i-th output (i = 0, 1, ...) of a sequence whose state starts at s0 is
mix(s0 + (i + 1) * 0x9E3779B97F4A7C15).  Every element is therefore a pure
function of (seed, stream, index) and can be computed in any order.  The
start state of a stream is s0 = mix(seed ^ (stream * 0xD1B54A32D192ED03)).

Distributions (element i of a stream)
-------------------------------------
* ``uniform``  : x_i >> 40 is a 24-bit integer u; value = u * 2**-23 - 1, in
  [-1, 1 - 2**-23].  Exactly representable in fp32.
* ``normal``   : Box-Muller in double on draws 2i and 2i+1:
  u1 = ((x_2i >> 11) + 1) * 2**-53 in (0, 1], u2 = (x_2i+1 >> 11) * 2**-53,
  z = sqrt(-2 ln u1) * cos(2 pi u2); value = sigma * z, rounded once to fp32
  (round to nearest even) and then, for bf16 operands, once more to bf16
  (round to nearest even).  The stored bf16 bits are the operand.
* ``integer``  : value = (x_i mod 5) - 2, in {-2, -1, 0, 1, 2}.

Seeds: the workloads use seed = 0x5EED0000 + workload index, streams 0, 1, 2
for A, B and the input C, and seed + 0x100 for the integer-valued pass.
"""

from __future__ import annotations

import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "splitmix64_stream",
    "splitmix64_from_state",
    "uniform_f32",
    "normal_f32",
    "integer_f32",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "draw",
    "WORKLOAD_SEED_BASE",
    "INTEGER_PASS_OFFSET",
]

WORKLOAD_SEED_BASE = 0x5EED0000
INTEGER_PASS_OFFSET = 0x100

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = 0xD1B54A32D192ED03
_MASK64 = (1 << 64) - 1
_CHUNK = 1 << 22


def _mix_py(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _stream_state(seed: int, stream: int) -> int:
    return _mix_py((seed ^ ((stream * _STREAM_MUL) & _MASK64)) & _MASK64)


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def splitmix64_from_state(s0: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of a splitmix64 sequence whose state
    starts at s0 (uint64)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(s0) + idx * _GOLDEN
        return _mix_np(z)


def splitmix64_stream(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of stream ``stream`` under ``seed`` (uint64)."""
    return splitmix64_from_state(_stream_state(seed, stream), start, count)


_pool = None
_pool_lock = threading.Lock()


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def _map_chunks(n: int, work) -> None:
    """Runs work(lo, hi) over [0, n) in chunks of _CHUNK elements, on a
    thread pool when there is more than one chunk.  Every element is a pure
    function of its index, so the result does not depend on the split."""
    spans = [(lo, min(n, lo + _CHUNK)) for lo in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for lo, hi in spans:
            work(lo, hi)
        return
    global _pool
    with _pool_lock:
        if _pool is None:
            _pool = ThreadPoolExecutor(max_workers=_threads())
    for f in [_pool.submit(work, lo, hi) for lo, hi in spans]:
        f.result()


def _chunked(n: int, fn, offset: int = 0) -> np.ndarray:
    """fn(first_index, count) over [offset, offset + n) in chunks."""
    out = np.empty(n, dtype=np.float32)

    def work(lo, hi):
        out[lo:hi] = fn(offset + lo, hi - lo)

    _map_chunks(n, work)
    return out


def uniform_f32(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Elements offset .. offset+n-1: uniform on the 2**-23 grid of [-1, 1)
    (exact fp32)."""

    def gen(lo, cnt):
        x = splitmix64_stream(seed, stream, lo, cnt)
        u = (x >> np.uint64(40)).astype(np.float64)
        return (u * 2.0**-23 - 1.0).astype(np.float32)

    return _chunked(n, gen, offset)


def normal_f32(seed: int, stream: int, n: int, sigma: float = 1.0,
               offset: int = 0) -> np.ndarray:
    """Elements offset .. offset+n-1: sigma * N(0, 1) by Box-Muller in
    double, rounded to fp32."""

    def gen(lo, cnt):
        x = splitmix64_stream(seed, stream, 2 * lo, 2 * cnt)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0**-53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (sigma * z).astype(np.float32)

    return _chunked(n, gen, offset)


def integer_f32(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Elements offset .. offset+n-1: integers in {-2..2} stored as fp32."""

    def gen(lo, cnt):
        x = splitmix64_stream(seed, stream, lo, cnt)
        return ((x % np.uint64(5)).astype(np.int64) - 2).astype(np.float32)

    return _chunked(n, gen, offset)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    NaNs map to a quiet NaN; infinities and overflow to infinity follow from
    the rounding itself.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)

    def work(lo, hi):
        xs = flat[lo:hi]
        b = xs.view(np.uint32).astype(np.uint64)
        lsb = (b >> np.uint64(16)) & np.uint64(1)
        r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
        nan = np.isnan(xs)
        if nan.any():
            r[nan] = ((b[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
        out[lo:hi] = r

    _map_chunks(flat.size, work)
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to fp32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def draw(kind: str, seed: int, stream: int, shape, sigma: float = 1.0,
         dtype: str = "f32", offset: int = 0) -> np.ndarray:
    """One operand of ``shape`` (row-major), drawn from ``kind``; its
    elements are stream elements offset, offset+1, ...

    kind: "uniform" | "normal" | "integer"; dtype: "f32" returns float32,
    "bf16" returns the uint16 bf16 bits.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    if kind == "uniform":
        v = uniform_f32(seed, stream, n, offset)
    elif kind == "normal":
        v = normal_f32(seed, stream, n, sigma, offset)
    elif kind == "integer":
        v = integer_f32(seed, stream, n, offset)
    else:
        raise ValueError(f"unknown distribution {kind!r}")
    v = v.reshape(shape)
    if dtype == "f32":
        return v
    if dtype == "bf16":
        return f32_to_bf16_bits(v).reshape(shape)
    raise ValueError(f"unknown dtype {dtype!r}")
