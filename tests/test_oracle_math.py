"""Closed-form pins for the oracle's building blocks (CPU only).

RMSNorm, SiLU and rotate-half RoPE are the LLaMA 3 layer pieces the P-EAGLE
drafter is built from (paper summary "P-EAGLE: Parallel-Drafting EAGLE with
Scalable Training", section 2).  RoPE's relative-position property is the
subject of Theorem 2.1 on the ScienceStack page; the top-left-submatrix
property of the causal mask is Figure 3's caption.
"""

import numpy as np
import pytest

import oracle as O
from tests import brute


def test_rms_norm_closed_forms():
    g = np.linspace(0.5, 1.5, 8)
    c = 3.0
    y = O.rms_norm(np.full((1, 8), c), g, 1e-5)
    assert np.allclose(y[0], g * c / np.sqrt(c * c + 1e-5), rtol=0, atol=1e-15)
    x = np.random.default_rng(0).normal(size=(3, 8))
    # with eps = 0 the norm is scale invariant and has unit RMS before the gain
    y1 = O.rms_norm(x, np.ones(8), 0.0)
    y2 = O.rms_norm(17.0 * x, np.ones(8), 0.0)
    assert np.allclose(y1, y2, atol=1e-14)
    assert np.allclose(np.sqrt((y1 ** 2).mean(1)), 1.0, atol=1e-14)


def test_silu_closed_forms():
    assert O.silu(np.array([0.0]))[0] == 0.0
    x = np.array([-3.0, -0.5, 0.25, 2.0, 40.0])
    assert np.allclose(O.silu(x), x / (1 + np.exp(-x)), atol=0)
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(O.silu(np.array([1.0]))[0] - 0.7310585786300049) < 1e-15


def test_rope_position_zero_is_identity_and_norm_preserving():
    x = np.random.default_rng(1).normal(size=(5, 3, 16))
    pos = np.array([0, 1, 7, 100, 20000])
    y = O.rope(x, pos, 150000.0)
    assert np.array_equal(y[0], x[0])
    # each (i, i + dh/2) pair is rotated, so pair norms are preserved
    pn = lambda t: t[..., :8] ** 2 + t[..., 8:] ** 2
    assert np.allclose(pn(y), pn(x), atol=1e-12)


def test_rope_two_dim_is_plane_rotation():
    # dh = 2: inv_freq = theta^0 = 1, so position p rotates by p radians
    x = np.array([[[1.0, 0.0]], [[0.3, -0.7]]])
    p = np.array([2, 5])
    y = O.rope(x, p, 10000.0)
    for i in range(2):
        c, s = np.cos(p[i]), np.sin(p[i])
        want = np.array([[c, -s], [s, c]]) @ x[i, 0]
        assert np.allclose(y[i, 0], want, atol=1e-15)


def test_rope_matches_complex_rotation():
    x = np.random.default_rng(2).normal(size=(4, 2, 64))
    pos = np.array([3, 64, 4095, 19999])
    assert np.allclose(O.rope(x, pos, 150000.0),
                       brute.rope_complex(x, pos, 150000.0), atol=1e-12)


@pytest.mark.parametrize("shift", [1, 37, 4096])
def test_rope_scores_depend_only_on_relative_position(shift):
    rng = np.random.default_rng(3)
    q = rng.normal(size=(1, 1, 64))
    k = rng.normal(size=(1, 1, 64))
    s0 = (O.rope(q, np.array([90]), 1e4) * O.rope(k, np.array([41]), 1e4)).sum()
    s1 = (O.rope(q, np.array([90 + shift]), 1e4)
          * O.rope(k, np.array([41 + shift]), 1e4)).sum()
    assert abs(s0 - s1) <= 1e-9 * max(1.0, abs(s0))


def test_attention_special_cases_and_brute_force():
    rng = np.random.default_rng(4)
    S, Hq, Hkv, dh = 9, 4, 2, 8
    k = rng.normal(size=(S, Hkv, dh))
    v = rng.normal(size=(S, Hkv, dh))
    # one visible key: output is its value
    out = O.attention_one_row(rng.normal(size=(Hq, dh)), k, v, 0)
    for h in range(Hq):
        assert np.allclose(out[h], v[0, h // 2])
    # zero query: uniform weights over positions 0..P
    out = O.attention_one_row(np.zeros((Hq, dh)), k, v, 5)
    for h in range(Hq):
        assert np.allclose(out[h], v[:6, h // 2].mean(0), atol=1e-15)
    # brute force with a dense mask matrix
    q = rng.normal(size=(Hq, dh))
    for P in range(S):
        want = np.zeros((Hq, dh))
        for h in range(Hq):
            sc = np.array([q[h] @ k[t, h * Hkv // Hq] for t in range(S)]) / np.sqrt(dh)
            sc = np.where(np.arange(S) <= P, sc, -np.inf)
            w = np.exp(sc - sc.max())
            w /= w.sum()
            want[h] = sum(w[t] * v[t, h * Hkv // Hq] for t in range(S))
        assert np.allclose(O.attention_one_row(q, k, v, P), want, atol=1e-13)


def _mask_by_probe(S):
    # read the mask the oracle applies: zero queries give uniform weights and
    # one-hot values expose which positions each row reads
    vals = np.eye(S)[:, None, :]          # [S, 1, S]
    keys = np.zeros((S, 1, S))
    m = np.zeros((S, S), bool)
    for P in range(S):
        m[P] = O.attention_one_row(np.zeros((1, S)), keys, vals, P)[0] > 0
    return m


def test_mask_of_shorter_sequence_is_top_left_submatrix():
    long_m, short_m = _mask_by_probe(11), _mask_by_probe(6)
    assert np.array_equal(short_m, long_m[:6, :6])
    assert np.array_equal(long_m, np.tril(np.ones((11, 11), bool)))


def test_linear_matches_explicit_loops_and_chunking():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(3, 5))
    w = rng.normal(size=(7, 5)).astype(np.float32)
    want = np.array([[sum(x[r, i] * float(w[o, i]) for i in range(5))
                      for o in range(7)] for r in range(3)])
    assert np.allclose(O.linear(x, w, "f32", rows_per_chunk=2), want, atol=1e-13)
    # bf16 weights: 0x3F80 + i encodes 1 + i/128 exactly (i < 128)
    bits = (0x3F80 + np.arange(35).reshape(7, 5)).astype(np.uint16)
    wf = 1.0 + np.arange(35).reshape(7, 5) / 128.0
    want = np.array([[sum(x[r, i] * wf[o, i] for i in range(5)) for o in range(7)]
                     for r in range(3)])
    assert np.allclose(O.linear(x, bits, "bf16", rows_per_chunk=3), want, atol=1e-13)


def test_bf16_decoding_known_values():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x3E80, 0x4049], np.uint16)
    assert O.to_f64(bits, "bf16").tolist() == [1.0, -2.0, 0.0, 0.25, 3.140625]


def test_lm_head_argmax_ties_take_the_lowest_index():
    """Reading R8: greedy argmax, lowest vocabulary index on exact ties.
    Duplicated LM-head rows give bit-identical logits; a hidden row equal to
    the duplicated row makes them the maximum (|w|^2 against cross terms of
    a few percent of it), so the oracle must return the lower copy."""
    from synthetic import workloads as W
    V, d = 96, 32
    sh = W.small_shape("tie", d=d, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=32,
                       ffn=32, vocab=V)
    lm = W.normal(5, "tie-lm", (V, d), 0.02, "bf16")
    pairs = [(9, 40), (0, V - 1), (70, 71), (3, 95 - 1)]
    for lo, hi in pairs:
        lm[lo] = lm[hi]
    y = O.to_f64(np.stack([lm[hi] for _, hi in pairs]), "bf16")
    logits, tokens = O.lm_head_argmax(sh, {"lm_head": lm}, y)
    for r, (lo, hi) in enumerate(pairs):
        assert logits[r, lo] == logits[r, hi]
        others = np.delete(logits[r], [lo, hi])
        assert logits[r, lo] > others.max()
        assert tokens[r] == lo
    # three-way tie: the first of the three
    lm2 = lm.copy()
    lm2[50] = lm2[20] = lm2[80]
    _, t2 = O.lm_head_argmax(sh, {"lm_head": lm2}, O.to_f64(lm2[80][None], "bf16"))
    assert t2[0] == 20
