"""Shared pieces of the GPU parity tests.

The tolerance every floating-point comparison uses, elementwise:
|y - y_ref| <= 1e-2 + 1e-2 |y_ref|, y_ref the oracle's fp64 output (H rounded
to bf16 between the layers, as the kernels store it).

The oracle is single-threaded C called through ctypes, which releases the
interpreter lock for the duration of each call, so many rows of a full-size
workload are computed at once by splitting them over host threads (no
processes: nothing is forked after the GPU is in use).  Each thread runs the
oracle unchanged on its own rows; the results are concatenated in row order.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ATOL = 1e-2
RTOL = 1e-2


def assert_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    assert np.isfinite(got).all(), f"{what}: {int((~np.isfinite(got)).sum())} non-finite outputs"
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def threads():
    return max(1, min(32, os.cpu_count() or 1))


def oracle_rows(fn, rows, nthreads=None):
    """fn(list of rows) -> array [len(rows) x P], computed over host threads
    in contiguous chunks of the row list; returns the rows in the given order."""
    rows = [int(r) for r in rows]
    n = nthreads or threads()
    n = max(1, min(n, len(rows)))
    chunks = [rows[i * len(rows) // n:(i + 1) * len(rows) // n] for i in range(n)]
    chunks = [c for c in chunks if c]
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        parts = list(ex.map(fn, chunks))
    return np.concatenate(parts, axis=0)


def band_rows(M, band=256, offsets=(0, 127, 128, 255)):
    """Rows at the given offsets of every band of `band` rows (the engine's
    pair tile: rows 0-127 belong to the leader CTA, 128-255 to its peer),
    clipped to M, plus the last row."""
    out = set()
    for b0 in range(0, M, band):
        for o in offsets:
            if b0 + o < M:
                out.add(b0 + o)
    out.add(M - 1)
    return sorted(out)


def moe_tail_tokens(perm, offsets, k, band=256, per_expert=2):
    """Tokens whose grouped row lies in the last, partly filled band of its
    expert's segment (the band that is zero-padded), up to per_expert each."""
    perm = np.asarray(perm)
    offsets = np.asarray(offsets)
    toks = []
    for e in range(len(offsets) - 1):
        c = int(offsets[e + 1] - offsets[e])
        if c == 0 or c % band == 0:
            continue
        first_tail = (c // band) * band
        picks = [first_tail, c - 1][:per_expert]
        for j in picks:
            toks.append(int(perm[offsets[e] + j]) // k)
    return sorted(set(toks))


def with_random(chosen, total, n, seed):
    """The chosen indices plus distinct random ones from [0, total) until
    there are n (or all of them), sorted."""
    out = set(int(x) for x in chosen)
    rng = np.random.default_rng(seed)
    for x in rng.permutation(total):
        if len(out) >= min(n, total):
            break
        out.add(int(x))
    return sorted(out)
