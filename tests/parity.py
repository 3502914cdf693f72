"""Comparison rules between the CUDA path and the fp64 oracle.

Values: bf16 operands with fp32 accumulation against exact fp64 are held to
    max|err| <= 2e-2 * max|ref|   and   mean|err| / mean|ref| <= 5e-3
(relative L1 for the mean, so near-zero references do not dominate).
Gates: fp32 against fp64, |dw| <= (n + 8) * 2^-24 with n the number of
terms in the softmax denominator (k renormalised, E otherwise).
Integers (indices, counts, offsets, rows) must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_REL = 2e-2
MEAN_REL = 5e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def value_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    max_rel = err.max() / max(np.abs(ref).max(), 1e-300)
    mean_rel = err.mean() / max(np.abs(ref).mean(), 1e-300)
    return float(max_rel), float(mean_rel)


def assert_values_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if ref.size == 0:
        return
    if np.abs(ref).max() == 0:
        assert np.abs(got).max() == 0, what
        return
    max_rel, mean_rel = value_errors(got, ref)
    assert max_rel <= MAX_REL and mean_rel <= MEAN_REL, f"{what}: max_rel={max_rel:.3e} mean_rel={mean_rel:.3e}"


def gate_tolerance(n_terms: int) -> float:
    return (n_terms + 8) * 2.0 ** -24


def assert_gates_close(got, ref, n_terms, what="gates"):
    err = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64))
    tol = gate_tolerance(n_terms)
    assert err.max(initial=0.0) <= tol, f"{what}: max |dw| = {err.max():.3e} > {tol:.3e}"


class ExpertSlices:
    """Per-expert weight matrices fetched from the device when indexed, as
    float64 host arrays (exact bf16 values), indexable like [E, ...].
    Nothing is kept: the oracle reads each expert's matrices once, so host
    memory holds one expert at a time even when the sample touches all of
    them (at the 1T-layer shape, 264 MB per expert against 100 GB for all)."""

    def __init__(self, w: torch.Tensor):
        self.w = w
        self.shape = tuple(w.shape)

    def __getitem__(self, e):
        return self.w[int(e)].double().cpu().numpy()


TILE_TOKENS = 512  # tokens of one paired-GEMM tile at most (two MMAs of up to 256)
PART_TOKENS = 256  # tokens of the first MMA of a tile


def paired_token_tiles(rows: int):
    """(start, valid) of the token tiles the paired grouped GEMM cuts an
    expert's rows into: ceil(rows / 512) near-equal tiles of S rows, S a
    multiple of 16, the last one holding the rest."""
    if rows <= 0:
        return []
    n0 = -(-rows // TILE_TOKENS)
    S = (-(-rows // n0) + 15) // 16 * 16
    return [(i * S, min(S, rows - i * S)) for i in range(-(-rows // S))]


def tile_edge_rows(offsets: np.ndarray, experts) -> list:
    """Rows at the edges of each token tile of the given experts: the first
    and last row of every tile (the last one inside the tile's last, often
    partial, 16-row group), and the last row of the first MMA and the first
    of the second where a tile holds more than 256 tokens."""
    rows = []
    for e in experts:
        base = int(offsets[e])
        for start, valid in paired_token_tiles(int(offsets[e + 1]) - base):
            r0 = base + start
            rows += [r0, r0 + valid - 1]
            if valid > PART_TOKENS:
                rows += [r0 + PART_TOKENS - 1, r0 + PART_TOKENS]
    return sorted(set(rows))


def pick_sample_tokens(idx: np.ndarray, counts: np.ndarray, n_random: int, seed: int = 0, offsets=None,
                       src_token=None, n_edge_experts: int = 4):
    """Seeded token sample: random tokens plus tokens routed to the largest
    and to the smallest non-empty expert group; with offsets and src_token,
    also the tokens of the tile-edge rows (tile_edge_rows) of those two
    groups and of n_edge_experts more chosen at random."""
    rng = np.random.default_rng(seed)
    T = idx.shape[0]
    toks = set(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    nz = np.nonzero(counts)[0]
    big = nz[np.argmax(counts[nz])]
    small = nz[np.argmin(counts[nz])]
    for e in (big, small):
        hit = np.nonzero((idx == e).any(axis=1))[0]
        toks.update(hit[:4].tolist())
    if offsets is not None and src_token is not None:
        more = rng.choice(nz, size=min(n_edge_experts, len(nz)), replace=False).tolist()
        rows = tile_edge_rows(offsets, sorted({int(big), int(small), *more}))
        toks.update(np.asarray(src_token)[rows].tolist())
    return np.array(sorted(toks), dtype=np.int64)
