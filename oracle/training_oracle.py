"""CPU oracle for P-EAGLE's long-context training layout -- TEST INFRASTRUCTURE.

Plain statements of the training-side index work: conditional drop-token
(COD) sampling of the prediction-depth positions, the attention mask over
(position, depth) rows, its amortized form (one mask for the longest
sequence, sliced per sample), and the sequence partitioning that splits one
long sequence into segments for gradient accumulation within a sequence.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; it shares no code with the CUDA library.

Sources (cited by page title and section):
  [paper]  "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training"
           (summary page): section 3 challenge analysis (n x K positions, COD
           keeps later depths at a geometric rate r), 3.1 "Amortized Mask
           Construction", 3.2 "Sequence Partitioning" (the four steps, and
           the 8192-token, K = 8, r = 0.8 example of about 34 thousand
           positions).
  [abstract page] ScienceStack page for the paper: Figure 3 caption
           (the mask of a shorter sequence is the top-left submatrix of a
           longer one's), Figure 4 caption (n = 16, K = 4; position 8 at
           depth 2 depends on position 7 at depth 1).

Readings taken where the pages are silent (listed with their reasons in the
design notes of the repository):
  T1 rows: row (p, d) is depth d at position p, d = 0..K-1; depth 0 is the
     ordinary next-token row of position p; depth d >= 1 is the d-th MASK
     row of the draft whose next-token row is (p - d, 0), so it exists only
     for p >= d.  Rows are laid out position-major: index p * K + d.
  T2 attention: (p, d) attends depth-0 rows q <= p - d (the context and the
     draft's own next-token row) and the draft's MASK rows (p - d + e, e)
     for 1 <= e <= d.  This is what a request's rows attend at inference
     (cache positions before the next-token row, the next-token row, the
     MASK rows up to itself).
  T3 COD: depth 0 is kept whole; (p, d >= 1) is kept when its dependency
     (p - 1, d - 1) is kept and its own draw u[p, d] < r, so depth d keeps
     a fraction r^d in expectation.
  T4 partition boundaries: S segments over depth-0 indices,
     bounds[0] = 0 < ... < bounds[S] = n; "all depth-0 positions up to its
     boundary" is read as the depth-0 rows before the segment's end; those
     owned by earlier segments are context (keys only) in this one.
"""

from __future__ import annotations

import dataclasses
from typing import List

import numpy as np


def row_index(p: int, d: int, K: int) -> int:
    """Position-major layout of the (position, depth) rows (T1)."""
    return p * K + d


def attends(p: int, d: int, q: int, e: int) -> bool:
    """May row (p, d) attend row (q, e)?  (T2; [abstract page] Figure 3.)"""
    if e == 0:
        return q <= p - d
    return 1 <= e <= d and q - e == p - d


def build_mask(n: int, K: int) -> np.ndarray:
    """Boolean [n K, n K] mask from the rule, row by row (small n only)."""
    N = n * K
    m = np.zeros((N, N), dtype=bool)
    for p in range(n):
        for d in range(K):
            if p < d:
                continue  # no such row (its draft would start before 0)
            i = row_index(p, d, K)
            for q in range(n):
                for e in range(K):
                    if q >= e and attends(p, d, q, e):
                        m[i, row_index(q, e, K)] = True
    return m


def slice_mask(mask_max: np.ndarray, n: int, K: int) -> np.ndarray:
    """[paper] 3.1: the mask of an n-token sample is the top-left n K x n K
    block of the precomputed mask (a view, no copy)."""
    return mask_max[: n * K, : n * K]


def cod_keep(n: int, K: int, r: float, u: np.ndarray) -> np.ndarray:
    """[paper] 3 (COD) with reading T3: kept rows [n, K] from the draws u
    [n, K] (float32, compared with float32 r)."""
    rr = np.float32(r)
    keep = np.zeros((n, K), dtype=bool)
    keep[:, 0] = True
    for d in range(1, K):
        for p in range(d, n):
            keep[p, d] = bool(keep[p - 1, d - 1]) and bool(np.float32(u[p, d]) < rr)
    return keep


def expected_kept(n: int, K: int, r: float) -> float:
    """E[number of kept rows] under T3: sum over d of (n - d) r^d."""
    return float(sum(max(0, n - d) * r ** d for d in range(K)))


@dataclasses.dataclass
class Segments:
    seg: np.ndarray           # int32 [n, K]: owning segment, -1 for dropped rows
    offsets: np.ndarray       # int32 [S + 1] into rows / owned
    rows: np.ndarray          # int32: layout indices of each segment's rows
    owned: np.ndarray         # uint8: 1 = row owned (loss counted) here


def segment_of_index(p: int, bounds) -> int:
    """The segment whose depth-0 index range [bounds[s], bounds[s+1]) holds p."""
    for s in range(len(bounds) - 1):
        if bounds[s] <= p < bounds[s + 1]:
            return s
    raise ValueError(f"position {p} outside the boundaries")


def partition(keep: np.ndarray, bounds) -> Segments:
    """[paper] 3.2, the four steps in order.

    1. boundaries over depth-0 indices (given);
    2. depth 0 and depth 1 rows go to the segment of their own index;
    3. depth d >= 2, in increasing d: a row goes where its dependency
       (p - 1, d - 1) went;
    4. every segment also holds the depth-0 rows before its end (context).
    Each segment's rows are listed in layout order.
    """
    n, K = keep.shape
    S = len(bounds) - 1
    seg = -np.ones((n, K), dtype=np.int64)
    for d in range(min(K, 2)):
        for p in range(n):
            if keep[p, d]:
                seg[p, d] = segment_of_index(p, bounds)
    for d in range(2, K):
        for p in range(n):
            if keep[p, d]:
                seg[p, d] = seg[p - 1, d - 1]
    offsets = [0]
    rows: List[int] = []
    owned: List[int] = []
    for s in range(S):
        mine = []
        for p in range(n):
            for d in range(K):
                if seg[p, d] == s:
                    mine.append((row_index(p, d, K), 1))
                elif d == 0 and p < bounds[s + 1]:
                    mine.append((row_index(p, 0, K), 0))
        mine.sort()
        rows += [i for i, _ in mine]
        owned += [o for _, o in mine]
        offsets.append(len(rows))
    return Segments(seg.astype(np.int32), np.asarray(offsets, np.int32),
                    np.asarray(rows, np.int32), np.asarray(owned, np.uint8))


def partition_by_index(keep: np.ndarray, bounds) -> np.ndarray:
    """The naive split the pages contrast with (Figure 4): every row goes to
    the segment of its own position index."""
    n, K = keep.shape
    seg = -np.ones((n, K), dtype=np.int64)
    for p in range(n):
        for d in range(K):
            if keep[p, d]:
                seg[p, d] = segment_of_index(p, bounds)
    return seg.astype(np.int32)


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     allowed: np.ndarray) -> np.ndarray:
    """softmax(q k^T) v over the allowed keys of each query (fp64)."""
    s = q @ k.T
    s = np.where(allowed, s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=1, keepdims=True)
    return w @ v
