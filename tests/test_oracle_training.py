"""Pins for the training-side oracle (CPU only): the attention rule over
(position, depth) rows, the amortized mask, COD sampling and the sequence
partitioning of "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training"
(paper summary page, sections 3, 3.1 and 3.2; ScienceStack page, Figures 3
and 4)."""

import numpy as np
import pytest

from oracle import training_oracle as TO


def _draws(n, K, seed):
    return np.random.default_rng(seed).random((n, K), dtype=np.float32)


# ----------------------------------------------------------------- mask rule

@pytest.mark.parametrize("K", [1, 2, 4])
def test_each_row_sees_exactly_the_positions_an_inference_row_sees(K):
    """At inference a drafting row at position p attends positions 0..p of its
    request: the cached context, the next-token row, and the draft's MASK
    rows up to itself.  Row (p, d) of the training layout must see each of
    those positions exactly once: as the depth-0 row for positions up to the
    draft's next-token row p - d, as the draft's own MASK row after it."""
    n = 11
    m = TO.build_mask(n, K)
    for p in range(n):
        for d in range(K):
            i = TO.row_index(p, d, K)
            cols = np.nonzero(m[i])[0]
            if p < d:
                assert cols.size == 0
                continue
            seen = sorted((c // K, c % K) for c in cols)
            assert [q for q, _ in seen] == list(range(p + 1))
            for q, e in seen:
                assert e == (0 if q <= p - d else q - (p - d))


def test_mask_is_position_invariant_and_slices_from_the_longest():
    """Figure 3: the mask of a shorter sequence is the top-left block of a
    longer one's, so one mask built for n_max serves every sample."""
    K, n_max = 3, 13
    big = TO.build_mask(n_max, K)
    for n in range(1, n_max + 1):
        view = TO.slice_mask(big, n, K)
        assert np.shares_memory(view, big)
        assert np.array_equal(view, TO.build_mask(n, K))
    # entries depend on p - q only (block Toeplitz over positions)
    rng = np.random.default_rng(3)
    for _ in range(200):
        p, q = rng.integers(K, n_max - 2, size=2)
        d, e = rng.integers(0, K, size=2)
        a = big[TO.row_index(p, d, K), TO.row_index(q, e, K)]
        b = big[TO.row_index(p + 2, d, K), TO.row_index(q + 2, e, K)]
        assert a == b


def test_depth_zero_block_is_the_ordinary_causal_mask():
    """With K = 1 there are no MASK rows: plain causal attention."""
    m = TO.build_mask(9, 1)
    assert np.array_equal(m, np.tril(np.ones((9, 9), dtype=bool)))


def test_mask_size_of_the_long_context_example():
    """[paper] section 3.2's example: 8192 tokens and K = 8 give 65,536 rows;
    a bf16 mask over them is 8.59 GB, the figure the amortized mask costs."""
    N = 8192 * 8
    assert N == 65536
    assert abs(N * N * 2 / 1e9 - 8.59) < 0.005


# ----------------------------------------------------------------------- COD

def test_cod_keeps_depth_zero_and_only_rows_whose_dependency_is_kept():
    n, K = 40, 6
    keep = TO.cod_keep(n, K, 0.7, _draws(n, K, 1))
    assert keep[:, 0].all()
    for p in range(n):
        for d in range(1, K):
            if keep[p, d]:
                assert p >= d and keep[p - 1, d - 1]
    assert TO.cod_keep(n, K, 1.0, _draws(n, K, 2)).sum() == sum(n - d for d in range(K))
    assert TO.cod_keep(n, K, 0.0, _draws(n, K, 2)).sum() == n


def test_cod_keeps_depth_d_at_rate_r_to_the_d():
    """[paper] section 3: COD retains later depths at a geometric rate r, so
    the expected row count is sum_d (n - d) r^d (closed form), checked by
    Monte Carlo within four standard errors."""
    n, K, r = 64, 5, 0.7
    counts = np.array([TO.cod_keep(n, K, r, _draws(n, K, s)).sum(axis=0) for s in range(300)])
    for d in range(K):
        want = (n - d) * r ** d
        se = counts[:, d].std(ddof=1) / np.sqrt(len(counts)) + 1e-9
        assert abs(counts[:, d].mean() - want) < 4 * se + 1e-9, (d, counts[:, d].mean(), want)


def test_cod_row_count_of_the_long_context_example():
    """[paper] section 3.2: 8192 tokens, K = 8, r = 0.8 keep about 34 thousand
    positions (n sum r^d = 34,088; the d < n edge takes ten off)."""
    n, K, r = 8192, 8, 0.8
    assert round(n * sum(r ** d for d in range(K))) == 34088
    assert abs(TO.expected_kept(n, K, r) - 34078.0) < 1.0


# ----------------------------------------------------------------- partition

def _fig4_keep():
    """n = 16, K = 4 with every draw below r: rows (7, 1) and (8, 2) exist."""
    n, K = 16, 4
    return TO.cod_keep(n, K, 0.5, np.zeros((n, K), np.float32))


def test_figure4_dependency_stays_in_one_segment():
    """Figure 4: split at depth-0 index 8, the naive split puts position 8 at
    depth 2 and its dependency, position 7 at depth 1, in different
    segments; the algorithm keeps them together."""
    keep = _fig4_keep()
    bounds = [0, 8, 16]
    naive = TO.partition_by_index(keep, bounds)
    assert naive[7, 1] == 0 and naive[8, 2] == 1
    seg = TO.partition(keep, bounds).seg
    assert seg[7, 1] == seg[8, 2] == 0
    assert seg[9, 3] == 0          # (9, 3) depends on (8, 2)
    assert seg[8, 1] == 1 and seg[8, 0] == 1


def _check_partition(keep, bounds, parts):
    n, K = keep.shape
    S = len(bounds) - 1
    seg = parts.seg
    # every kept row owned exactly once, dropped rows nowhere
    assert np.array_equal(seg >= 0, keep)
    owned_rows = []
    for s in range(S):
        lo, hi = parts.offsets[s], parts.offsets[s + 1]
        rows = parts.rows[lo:hi]
        own = parts.owned[lo:hi]
        assert np.all(np.diff(rows) > 0)
        owned_rows += list(rows[own == 1])
        present = set(int(i) for i in rows)
        for i in rows[own == 1]:
            p, d = divmod(int(i), K)
            assert seg[p, d] == s
            if d >= 2:
                assert seg[p - 1, d - 1] == s
            # every key the row may attend is in the segment
            for q in range(n):
                for e in range(K):
                    if keep[q, e] and TO.attends(p, d, q, e):
                        assert TO.row_index(q, e, K) in present, (s, p, d, q, e)
        for i in rows[own == 0]:
            assert int(i) % K == 0 and int(i) // K < bounds[s]
    assert sorted(owned_rows) == [TO.row_index(p, d, K) for p in range(n) for d in range(K)
                                  if keep[p, d]]


@pytest.mark.parametrize("seed", range(4))
def test_partition_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    n, K = int(rng.integers(20, 60)), int(rng.integers(1, 7))
    S = int(rng.integers(1, 6))
    cuts = sorted(rng.choice(np.arange(1, n), size=S - 1, replace=False).tolist())
    bounds = [0] + cuts + [n]
    keep = TO.cod_keep(n, K, 0.75, _draws(n, K, seed))
    _check_partition(keep, bounds, TO.partition(keep, bounds))


def test_the_naive_split_fails_the_same_checks():
    """A plausible wrong partition (by index) is caught by the invariants."""
    keep = _fig4_keep()
    bounds = [0, 8, 16]
    parts = TO.partition(keep, bounds)
    bad = TO.Segments(TO.partition_by_index(keep, bounds), parts.offsets, parts.rows, parts.owned)
    with pytest.raises(AssertionError):
        _check_partition(keep, bounds, bad)


def test_segmented_attention_equals_whole_sequence_attention():
    """[paper] 3.2: gradient accumulation within one sequence preserves every
    cross-depth dependency -- each owned row's attention over its segment's
    rows equals its attention over the whole sampled sequence."""
    rng = np.random.default_rng(7)
    n, K, dh = 37, 4, 8
    keep = TO.cod_keep(n, K, 0.8, _draws(n, K, 9))
    bounds = [0, 9, 20, 31, 37]
    parts = TO.partition(keep, bounds)
    full = TO.build_mask(n, K)
    kept = np.array([i for i in range(n * K) if keep[i // K, i % K]])
    q, k, v = (rng.normal(size=(n * K, dh)) for _ in range(3))
    whole = TO.masked_attention(q[kept], k[kept], v[kept], full[np.ix_(kept, kept)])
    at = {int(i): whole[j] for j, i in enumerate(kept)}
    for s in range(len(bounds) - 1):
        rows = parts.rows[parts.offsets[s]:parts.offsets[s + 1]]
        own = parts.owned[parts.offsets[s]:parts.offsets[s + 1]] == 1
        out = TO.masked_attention(q[rows[own]], k[rows], v[rows], full[np.ix_(rows[own], rows)])
        for j, i in enumerate(rows[own]):
            assert np.allclose(out[j], at[int(i)], rtol=0, atol=1e-12)


# ------------------------------------------------------- hand-worked fixtures

def _golden():
    import json
    import os
    p = os.path.join(os.path.dirname(__file__), "golden", "training_worked_examples.json")
    return json.load(open(p))


def test_mask_matches_the_hand_worked_example():
    g = _golden()["mask"]
    m = TO.build_mask(g["n"], g["K"])
    got = [np.nonzero(m[i])[0].tolist() for i in range(g["n"] * g["K"])]
    assert got == g["allowed_columns"]


def test_partition_matches_the_hand_worked_example():
    g = _golden()["partition"]
    keep = np.zeros((g["n"], g["K"]), dtype=bool)
    for p, d in g["kept"]:
        keep[p, d] = True
    parts = TO.partition(keep, g["bounds"])
    for key, s in g["expected_segment"].items():
        p, d = (int(x) for x in key.split(","))
        assert parts.seg[p, d] == s, key
    assert TO.partition_by_index(keep, g["bounds"])[4, 2] == g["naive_segment_of_4_2"]
    assert parts.offsets.tolist() == g["offsets"]
    assert parts.rows.tolist() == g["rows"]
    assert parts.owned.tolist() == g["owned"]
    # the same keep pattern drawn through COD: draws below r on kept rows
    u = np.where(keep, 0.0, 0.99).astype(np.float32)
    assert np.array_equal(TO.cod_keep(g["n"], g["K"], 0.5, u), keep)
