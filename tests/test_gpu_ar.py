"""Autoregressive drafting on the same kernels: K sequential passes of the
K = 1 step (the EAGLE baseline the pages compare against: K serial drafter
passes, each needing the previous token).  Pass 0 takes the verify window
and drafts the first token; pass i takes one row per request at the next
position, carrying the previous pass's draft token, and drafts the next.

Checked pass by pass against the oracle on identical inputs: the oracle is
given the GPU's draft token and the GPU's KV pools as they stand before
the pass (so one flipped near-tie cannot make the two sides diverge), and
the pass's metadata, hidden rows, logits, tokens (margin rule) and KV writes
are compared as in the one-step parity tests.
"""

import dataclasses

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2

SMALL = W.small_shape("small-bf16", d=512, n_layers=2, n_heads=8, n_kv_heads=2,
                      head_dim=64, ffn=1024, vocab=4096)


def _pass_parity(wl_pass, w, inp, kc, vc, dr):
    """One K=1 pass on the GPU and the oracle; returns the GPU tokens and the
    device KV pools after the pass (host copies)."""
    B = G.library()
    sh = wl_pass.shape
    st = G.DeviceStep(wl_pass, inp, kc, vc)
    G.remember_host_caches(st, kc, vc)
    res = G.run_step(dr, st, want_logits=True)
    assert res["err"] == 0, res["err"]
    ref = O.draft_step(sh, w, 1, inp, kc, vc)
    G.check_expand(res["ex"], ref.expanded, int(inp.cu_in[-1]))
    got_h = G.f64(B.to_host(res["out_hidden"]), sh.dtype)
    hs = np.abs(ref.out_hidden).max()
    assert np.abs(got_h - ref.out_hidden).max() <= TOL_BF16 * hs
    got_l = B.to_host(res["logits"]).astype(np.float64)
    ls = np.abs(ref.logits).max()
    assert np.abs(got_l - ref.logits).max() <= TOL_BF16 * ls
    got_t = B.to_host(res["tokens"])
    G.token_rule_stats(wl_pass.name, ref.logits, ref.tokens, got_t,
                       max(1e-2, 2 * TOL_BF16 * ls))
    G.margin_ok_tokens(ref.logits, ref.tokens, got_t, margin=1e-2)
    G.check_kv(st, ref, sh, TOL_BF16 * 2)
    return got_t, [B.to_host(k) for k in st.kc], [B.to_host(v) for v in st.vc]


def test_autoregressive_passes_match_the_oracle_pass_by_pass():
    K = 4
    contexts, windows, accepted = [100, 37, 250], [K + 1] * 3, [4, 1, 2]
    wl = W.custom("ar-small", 83, SMALL, K, contexts, windows, accepted, gains="random")
    inp0 = W.make_step_inputs(wl)
    w = W.make_weights(SMALL, wl.config_id, gains="random")
    kc, vc = W.make_kv_cache(wl, inp0)
    Bn = wl.B
    dr = G.make_drafter(SMALL, w, max(wl.T, Bn), Bn)
    # pass 0: the verify window with K = 1
    wl0 = W.custom("ar-pass0", 83, SMALL, 1, contexts, windows, accepted, gains="random")
    toks, kc, vc = _pass_parity(wl0, w, inp0, kc, vc, dr)
    # passes 1..K-1: one row per request at the next position
    last = [int(inp0.cu_in[r]) + accepted[r] for r in range(Bn)]
    p0 = np.array([int(inp0.target_pos[i]) + 1 for i in last], np.int32)
    wl1 = W.custom("ar-pass", 83, SMALL, 1, contexts, [1] * Bn, [0] * Bn, gains="random")
    for i in range(1, K):
        inp = dataclasses.replace(
            inp0, target_ids=np.zeros(Bn, np.int32), target_pos=(p0 + i - 1).astype(np.int32),
            cu_in=np.arange(Bn + 1, dtype=np.int32), num_accepted=np.zeros(Bn, np.int32),
            sampled_ids=np.asarray(toks, np.int32),
            target_hidden=np.ascontiguousarray(inp0.target_hidden[last]))
        toks, kc, vc = _pass_parity(wl1, w, inp, kc, vc, dr)
        assert np.all((toks >= 0) & (toks < SMALL.vocab))
