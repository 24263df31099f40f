"""The oracle on token (or row) shards over the host's threads.

Test infrastructure, like the oracle itself.  Every per-token step of the
path (top-k, the per-token cast, the SwiGLU cast, combine) treats each token
or row on its own, so running the unchanged single-threaded C oracle on
disjoint shards and concatenating the results gives exactly the whole-array
result; each shard is one C call, which releases the GIL.  The route map is
not per token and always runs once over all tokens.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def shard_bounds(n: int, parts: int):
    """[(a, b)] covering range(n) in `parts` nearly equal, non-empty pieces."""
    parts = max(1, min(parts, n))
    edges = np.linspace(0, n, parts + 1).round().astype(np.int64)
    return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]


def _map(fn, bounds, threads):
    if threads <= 1 or len(bounds) <= 1:
        return [fn(ab) for ab in bounds]
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(fn, bounds))


def topk_gate(scores: np.ndarray, k: int, threads: int | None = None):
    """oracle.topk_gate over token shards -> (idx [T, k], w [T, k])."""
    threads = threads or host_threads()
    parts = _map(lambda ab: oracle.topk_gate(scores[ab[0]:ab[1]], k),
                 shard_bounds(scores.shape[0], 4 * threads), threads)
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))


def per_token_cast(x_bits: np.ndarray, threads: int | None = None):
    """oracle.per_token_cast over token shards -> (q [T, H], sf [T, H/128])."""
    threads = threads or host_threads()
    T, H = x_bits.shape
    q = np.empty((T, H), dtype=np.uint8)
    sf = np.empty((T, H // 128), dtype=np.float32)

    def one(ab):
        a, b = ab
        q[a:b], sf[a:b] = oracle.per_token_cast(x_bits[a:b])

    _map(one, shard_bounds(T, 4 * threads), threads)
    return q, sf


def swiglu_cast_fp8(x_bits: np.ndarray, threads: int | None = None):
    """oracle.swiglu_cast_fp8 over row shards -> (q [M, N], sf [M, N/128])."""
    threads = threads or host_threads()
    M, N2 = x_bits.shape
    q = np.empty((M, N2 // 2), dtype=np.uint8)
    sf = np.empty((M, N2 // 256), dtype=np.float32)

    def one(ab):
        a, b = ab
        q[a:b], sf[a:b] = oracle.swiglu_cast_fp8(x_bits[a:b])

    _map(one, shard_bounds(M, 4 * threads), threads)
    return q, sf


def combine_gathered(y_rows_bits: np.ndarray, w: np.ndarray, threads: int | None = None):
    """oracle.combine of tokens whose k rows were gathered in slot order:
    y_rows_bits [n*k, H] holds token i's row j at i*k + j.
    -> (out_f32 [n, H], out_bf16_bits [n, H], abs_sum [n, H])."""
    threads = threads or host_threads()
    n, k = w.shape
    H = y_rows_bits.shape[1]
    o32 = np.empty((n, H), dtype=np.float32)
    o16 = np.empty((n, H), dtype=np.uint16)
    mag = np.empty((n, H), dtype=np.float32)

    def one(ab):
        a, b = ab
        lpos = np.arange((b - a) * k, dtype=np.int32).reshape(b - a, k)
        o32[a:b], o16[a:b], mag[a:b] = oracle.combine(y_rows_bits[a * k:b * k], w[a:b], lpos)

    _map(one, shard_bounds(n, 4 * threads), threads)
    return o32, o16, mag


def per_token_cast_fp4(x_bits: np.ndarray, group: int, threads: int | None = None):
    """The FP4 E2M1 cast of every token (oracle.expand_cast_fp4 with one copy
    per token, on token shards) -> (q [T, H/2] packed, sf [T, H/group])."""
    threads = threads or host_threads()
    T, H = x_bits.shape
    q = np.empty((T, H // 2), dtype=np.uint8)
    sf = np.empty((T, H // group), dtype=np.float32)

    def one(ab):
        a, b = ab
        ident = np.arange(b - a, dtype=np.int32)[:, None]
        q[a:b], sf[a:b] = oracle.expand_cast_fp4(x_bits[a:b], ident, group=group)

    _map(one, shard_bounds(T, 4 * threads), threads)
    return q, sf


def swiglu_cast_fp4(x_bits: np.ndarray, group: int, threads: int | None = None):
    """oracle.swiglu_cast_fp4 over row shards -> (q [M, N/2], sf [M, N/group])."""
    threads = threads or host_threads()
    M, N2 = x_bits.shape
    q = np.empty((M, N2 // 4), dtype=np.uint8)
    sf = np.empty((M, N2 // 2 // group), dtype=np.float32)

    def one(ab):
        a, b = ab
        q[a:b], sf[a:b], _ = oracle.swiglu_cast_fp4(x_bits[a:b], group=group)

    _map(one, shard_bounds(M, 4 * threads), threads)
    return q, sf
