"""Seeded synthetic SIFT-shaped descriptors for the exhaustive-matching workloads.

This module only makes inputs. It holds none of the matcher's arithmetic (no dot
products, no top-2, no ratio test), so both the CUDA path's tests and the oracle's
tests draw their inputs from here without sharing any matching code.

Recipe (stated once, used by every workload below):

* base descriptor: z ~ N(0, 1)^128 in float64; x = z**2; x /= ||x||; x = min(x, 0.2);
  x /= ||x||; u8 = min(255, floor(512 * x)).  This is the usual SIFT normalise /
  clip-at-0.2 / renormalise shaping, quantised at 512 so that ||u8||^2 <= 512^2.
* planted copy of a source row: take the source's float vector (after clip and
  renormalise), add N(0, sigma) per dimension, clamp negatives to 0, L2-renormalise
  (no second clip), quantise as above.  The copy goes to a seeded, distinct slot of
  the receiving image.
* every random stream comes from ``numpy.random.default_rng([seed, workload, item,
  role])`` so that any image or pair can be regenerated on its own.

The pages measure on a 589-image UAV survey and the south-building subset; neither
is available, so these seeded inputs stand in for them with the same descriptor
length (128 x u8), feature counts of the stated sizes and a planted share of true
correspondences.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DIM = 128
QUANT_SCALE = 512.0

# role tags for the sub-streams
_ROLE_BASE = 0
_ROLE_PICK = 1
_ROLE_NOISE = 2
_ROLE_SLOT = 3
_ROLE_SIZE = 4


def _rng(seed: int, workload: int, item: int, role: int) -> np.random.Generator:
    return np.random.default_rng([seed, workload, item, role])


def quantize(x: np.ndarray) -> np.ndarray:
    """float vectors with unit L2 norm -> uint8 by floor(512 x), capped at 255."""
    q = np.floor(QUANT_SCALE * x)
    return np.minimum(q, 255.0).astype(np.uint8)


def _normalise(x: np.ndarray) -> np.ndarray:
    nrm = np.sqrt((x * x).sum(axis=1, keepdims=True))
    nrm[nrm == 0] = 1.0
    return x / nrm


def base_float(rng: np.random.Generator, n: int) -> np.ndarray:
    """SIFT-shaped float descriptors (n, 128), unit norm, entries <= 0.2 before renorm."""
    z = rng.standard_normal((n, DIM))
    x = _normalise(z * z)
    x = np.minimum(x, 0.2)
    return _normalise(x)


def noisy_copy(rng: np.random.Generator, src: np.ndarray, sigma: float) -> np.ndarray:
    """Planted copies: src + N(0, sigma), negatives clamped, renormalised, quantised."""
    y = src + rng.normal(0.0, sigma, size=src.shape)
    y = np.maximum(y, 0.0)
    return quantize(_normalise(y))


@dataclass
class Pair:
    """One image pair: descriptors of A and B plus the planted (i, j) ground truth."""
    a: np.ndarray
    b: np.ndarray
    truth: np.ndarray  # (k, 2) int64 rows (i in A, j in B)


@dataclass
class ImageSet:
    """Images of one exhaustive run and the pairs (i, j), i < j, to match."""
    images: list
    pairs: np.ndarray  # (P, 2) image indices
    truth: dict = field(default_factory=dict)  # (i, j) -> (k, 2) planted rows


def make_pair(seed: int, workload: int, item: int, n_a: int, n_b: int,
              frac: float, sigma: float, planted: int | None = None) -> Pair:
    """A pair where `planted` (default floor(frac * n_a)) rows of A are planted into B."""
    fa = base_float(_rng(seed, workload, item, _ROLE_BASE), n_a)
    fb = base_float(_rng(seed, workload, item, _ROLE_BASE + 10), n_b)
    a = quantize(fa)
    b = quantize(fb)
    k = int(np.floor(frac * n_a)) if planted is None else int(planted)
    k = min(k, n_a, n_b)
    src = _rng(seed, workload, item, _ROLE_PICK).choice(n_a, size=k, replace=False)
    dst = _rng(seed, workload, item, _ROLE_SLOT).choice(n_b, size=k, replace=False)
    if k:
        b[dst] = noisy_copy(_rng(seed, workload, item, _ROLE_NOISE), fa[src], sigma)
    truth = np.stack([src, dst], axis=1).astype(np.int64) if k else np.zeros((0, 2), np.int64)
    order = np.argsort(truth[:, 0], kind="stable")
    return Pair(a=a, b=b, truth=truth[order])


def make_ring(seed: int, workload: int, n_images: int, n_desc: int, frac: float,
              sigma: float, reach: int) -> ImageSet:
    """Images on a ring; image i plants frac * n of its rows into (i + d) mod n_images
    for d = 1..reach.  Each receiver's incoming slots are disjoint (one permutation of
    its rows cut into `reach` chunks) and every planted source row is one its image
    never overwrites, so each planted row is a true correspondence."""
    floats = [base_float(_rng(seed, workload, i, _ROLE_BASE), n_desc) for i in range(n_images)]
    images = [quantize(f) for f in floats]
    k = int(np.floor(frac * n_desc))
    # incoming slots of receiver r: chunk d-1 receives from (r - d) mod n
    slots = {}
    for r in range(n_images):
        perm = _rng(seed, workload, r, _ROLE_SLOT).permutation(n_desc)
        for d in range(1, reach + 1):
            slots[(r, d)] = perm[(d - 1) * k: d * k]
    truth = {}
    for i in range(n_images):
        overwritten = np.concatenate([slots[(i, d)] for d in range(1, reach + 1)])
        kept = np.setdiff1d(np.arange(n_desc), overwritten)
        for d in range(1, reach + 1):
            r = (i + d) % n_images
            src = _rng(seed, workload, i * 1000 + d, _ROLE_PICK).choice(kept, size=k, replace=False)
            dst = slots[(r, d)]
            images[r][dst] = noisy_copy(_rng(seed, workload, i * 1000 + d, _ROLE_NOISE),
                                        floats[i][src], sigma)
            t = np.stack([src, dst], axis=1).astype(np.int64)
            if i < r:
                truth[(i, r)] = t[np.argsort(t[:, 0], kind="stable")]
            else:
                t = t[:, ::-1]
                truth[(r, i)] = t[np.argsort(t[:, 0], kind="stable")]
    iu = np.array([(i, j) for i in range(n_images) for j in range(i + 1, n_images)], np.int64)
    return ImageSet(images=images, pairs=iu, truth=truth)


# ---------------------------------------------------------------- the five workloads

def single_pair_2000(seed: int = 0) -> Pair:
    """2,000 x 2,000, 30% of A planted into B at sigma = 0.05."""
    return make_pair(seed, 0, 0, 2000, 2000, 0.30, 0.05)


def single_pair_8192(seed: int = 0) -> Pair:
    """8,192 x 8,192, 25% planted at sigma = 0.08."""
    return make_pair(seed, 1, 0, 8192, 8192, 0.25, 0.08)


def ring_12x8192(seed: int = 0) -> ImageSet:
    """12 images x 8,192; each shares 20% (sigma 0.06) with each of its 3 ring
    neighbours (image i plants into i+1, i+2, i+3 mod 12); all 66 pairs."""
    return make_ring(seed, 2, 12, 8192, 0.20, 0.06, 3)


def ragged_sizes(seed: int = 0, n_pairs: int = 256) -> np.ndarray:
    """Per-image feature counts of the ragged batch: uniform on {1000, ..., 16384}."""
    return _rng(seed, 3, 0, _ROLE_SIZE).integers(1000, 16384, size=(n_pairs, 2), endpoint=True)


def ragged_pair(seed: int, p: int, sizes: np.ndarray) -> Pair:
    """Pair p of the ragged batch: 15% of min(nA, nB) planted at sigma = 0.05."""
    n_a, n_b = int(sizes[p, 0]), int(sizes[p, 1])
    k = int(np.floor(0.15 * min(n_a, n_b)))
    return make_pair(seed, 3, p + 1, n_a, n_b, 0.15, 0.05, planted=k)


def survey_100x8192(seed: int = 0) -> ImageSet:
    """100 images x 8,192, each sharing 10% (sigma 0.05) with its 6 nearest indices
    (plants go i -> i+1, i+2, i+3 mod 100, so each image meets i-3..i+3); 4,950 pairs."""
    return make_ring(seed, 4, 100, 8192, 0.10, 0.05, 3)


def survey_spot_pairs(seed: int = 0, n: int = 50, n_pairs: int = 4950) -> np.ndarray:
    """The seeded spot-check subset of the 4,950 survey pairs (lexicographic order)."""
    return np.sort(np.random.default_rng(seed).choice(n_pairs, n, replace=False))


def random_u8(seed: int, n: int, low: int = 0, high: int = 256) -> np.ndarray:
    """Plain uniform bytes (edge cases, ties, adversarial magnitudes)."""
    return np.random.default_rng([seed, 99, n, low, high]).integers(
        low, high, size=(n, DIM), dtype=np.int64).astype(np.uint8)
