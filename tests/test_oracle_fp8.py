"""Pins for the oracle's fp8 (e4m3) KV cache (CPU only): the code table
against the OCP FP8 E4M3 definition's fixed points, the encoder against a
brute-force nearest search (ties to the even code, saturation, NaN, signed
zero), and the fp8 drafter path against the exact one within the format's
rounding error."""

import numpy as np
import pytest

import oracle as O
from oracle import fp8_kv as F
from synthetic import workloads as W


def test_code_table_fixed_points():
    t = F.E4M3_TABLE
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    assert t[0x38] == 1.0 and t[0xB8] == -1.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0          # largest finite
    assert t[0x01] == 2.0 ** -9                              # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9 and t[0x08] == 2.0 ** -6  # subnormal -> normal
    assert t[0x30] == 0.5 and t[0x40] == 2.0 and t[0x3C] == 1.5
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                          # codes ordered by value
    assert np.array_equal(t[0x80:0xFF], -pos)                # sign-magnitude
    assert np.count_nonzero(np.isfinite(t)) == 254


def _brute(v):
    """Nearest finite code by distance to all 254 values; ties to the even
    code; beyond the range the largest magnitude."""
    if np.isnan(v):
        return 0x7F
    codes = [c for c in range(256) if np.isfinite(F.E4M3_TABLE[c])]
    sign_ok = [c for c in codes if (c & 0x80) == (0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0)]
    d = [abs(F.E4M3_TABLE[c] - v) for c in sign_ok]
    best = min(d)
    cands = [c for c, x in zip(sign_ok, d) if x == best]
    even = [c for c in cands if c % 2 == 0]
    return (even or cands)[0]


def test_encoder_matches_brute_force_nearest():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.normal(size=300) * 10.0 ** rng.uniform(-4, 2.8, size=300),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, size=100),          # subnormal range
        [0.0, -0.0, 447.9, 448.0, 460.0, 464.0, 1e6, -1e6, np.nan],
    ])
    got = F.e4m3_encode(xs)
    for x, c in zip(xs, got):
        assert int(c) == _brute(x), (x, hex(int(c)), hex(_brute(x)))


def test_encoder_round_trips_and_rounds_ties_to_even():
    finite = [c for c in range(256) if np.isfinite(F.E4M3_TABLE[c])]
    assert np.array_equal(F.e4m3_encode(F.E4M3_TABLE[finite]), np.array(finite, np.uint8))
    # midpoints: 1.0625 between 0x38 (1.0) and 0x39 (1.125) -> 0x38 (even)
    assert F.e4m3_encode([1.0625])[0] == 0x38
    assert F.e4m3_encode([1.1875])[0] == 0x3A
    # the midpoint between the largest subnormal and the smallest normal
    assert F.e4m3_encode([7.5 * 2.0 ** -9])[0] == 0x08
    # half the smallest subnormal ties to zero (even); just above it rounds up
    assert F.e4m3_encode([2.0 ** -10])[0] == 0x00
    assert F.e4m3_encode([2.0 ** -10 * 1.01])[0] == 0x01
    # saturation to +-448
    assert F.e4m3_encode([1e9])[0] == 0x7E and F.e4m3_encode([-500.0])[0] == 0xFE


def test_quantisation_error_is_within_half_a_step():
    rng = np.random.default_rng(1)
    x = rng.normal(size=2000) * 3.0
    s = 0.05
    y = F.dequantize(F.quantize(x, s), s)
    # relative half-step of a 3-bit mantissa: 2^-4 (normals)
    normal = np.abs(x / s) >= 2.0 ** -6
    assert np.all(np.abs(y - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 + 1e-15)


def _fp8_caches(kc, vc, dtype, ks, vs):
    kq = [F.quantize(O.to_f64(k, dtype), ks) for k in kc]
    vq = [F.quantize(O.to_f64(v, dtype), vs) for v in vc]
    return kq, vq


def test_fp8_cache_step_tracks_the_exact_step():
    """The step with an fp8 cache (context pages and this step's writes in
    e4m3) stays within the format's error of the exact step, moves away from
    it (the quantisation is applied), and its KV writes are the codes of
    k / k_scale."""
    wl = W.tiny_fp32()
    inp = W.make_step_inputs(wl)
    w = W.make_weights(wl.shape, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    ref = O.draft_step(wl.shape, w, wl.K, inp, kc, vc)
    scales = [(0.05, 0.04)] * wl.shape.n_layers
    kq, vq = _fp8_caches(kc, vc, wl.shape.dtype, 0.05, 0.04)
    got = O.draft_step(wl.shape, w, wl.K, inp, kq, vq, kv_scales=scales)
    for l in range(wl.shape.n_layers):
        a, b = got.drafter.layer_attn[l], ref.drafter.layer_attn[l]
        err = np.abs(a - b).max() / np.abs(b).max()
        assert 1e-5 < err < 0.1, (l, err)
        kw = got.drafter.kv_writes[l]
        assert np.array_equal(kw["k_codes"], F.quantize(kw["k"], 0.05))
        assert np.array_equal(kw["v_codes"], F.quantize(kw["v"], 0.04))
    rel = np.abs(got.out_hidden - ref.out_hidden).max() / np.abs(ref.out_hidden).max()
    assert rel < 0.1


def test_fp8_scale_sits_on_the_values_the_attention_reads():
    """The attention reads code * scale: a cache quantised with one v_scale
    and read with another moves the attention output by far more than the
    rounding error (a scale dropped or applied twice would fail this)."""
    wl = W.tiny_fp32()
    inp = W.make_step_inputs(wl)
    w = W.make_weights(wl.shape, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    kq, vq = _fp8_caches(kc, vc, wl.shape.dtype, 0.05, 0.04)
    L = wl.shape.n_layers
    good = O.draft_step(wl.shape, w, wl.K, inp, kq, vq, kv_scales=[(0.05, 0.04)] * L)
    bad = O.draft_step(wl.shape, w, wl.K, inp, kq, vq, kv_scales=[(0.05, 0.08)] * L)
    a, b = good.drafter.layer_attn[0], bad.drafter.layer_attn[0]
    assert np.abs(a - b).max() > 0.2 * np.abs(a).max()
