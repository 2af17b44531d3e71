"""Step-level pins for the oracle (CPU only, tiny shapes).

What the pages fix and these tests check:
  * brute force: an independent dense-mask restatement of the drafter agrees;
  * with K=1 the parallel step is one autoregressive EAGLE step (vLLM blog
    summary, "P-EAGLE drafter": NTP position works like AR EAGLE);
  * draft token 1 does not depend on K (causality: MASK rows follow it);
  * requests are independent (batch invariance) and paging is transparent;
  * rejected rows never write the KV cache (blog, KV-cache bullet: -1 slots).
"""

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W
from tests import brute

SHAPE_F32 = W.small_shape("pin-f32", d=64, n_layers=2, n_heads=4, n_kv_heads=2,
                          head_dim=16, ffn=96, vocab=128, dtype="f32")
SHAPE_BF16 = W.small_shape("pin-bf16", d=64, n_layers=2, n_heads=4,
                           n_kv_heads=1, head_dim=16, ffn=96, vocab=128,
                           dtype="bf16")


def _setup(shape, cid, K, contexts, window, accepted, order="random"):
    wl = W.custom("pin", cid, shape, K, contexts, window, accepted, order,
                  gains="random")
    inp = W.make_step_inputs(wl)
    w = W.make_weights(shape, cid, gains="random", std=0.2)
    k, v = W.make_kv_cache(wl, inp)
    return wl, inp, w, k, v


@pytest.mark.parametrize("shape", [SHAPE_F32, SHAPE_BF16], ids=["f32", "bf16"])
def test_oracle_matches_brute_force(shape):
    wl, inp, w, k, v = _setup(shape, 11, 3, [5, 17, 33], [4, 2, 3], [1, 0, 2])
    res = O.draft_step(shape, w, wl.K, inp, k, v)
    ex = res.expanded
    rows = res.row_index
    seq = {r: int(ex.seq_lens[r]) for r in range(wl.B)}
    want = brute.drafter(shape, w, ex.ids[rows], res.hidden[rows],
                         ex.pos[rows], ex.request_of_row[rows],
                         inp.block_table, seq, k, v)
    got = res.drafter.residual
    assert np.allclose(got, want, rtol=1e-10, atol=1e-12)
    assert np.all(np.isfinite(res.logits))   # no NaN sentinel was read


def test_k1_equals_one_autoregressive_eagle_step():
    wl, inp, w, k, v = _setup(SHAPE_F32, 12, 1, [9, 30, 16, 1], [3, 1, 2, 4],
                              [2, 0, 1, 3])
    res = O.draft_step(SHAPE_F32, w, 1, inp, k, v)
    logits, tokens = O.ar_eagle_step(SHAPE_F32, w, inp, k, v)
    assert np.array_equal(res.tokens, tokens)
    assert np.allclose(res.logits, logits, rtol=0, atol=1e-12)


def test_first_draft_token_does_not_depend_on_k():
    outs = []
    # one set of inputs (its page tables sized for the largest K)
    wl, inp, w, k, v = _setup(SHAPE_F32, 13, 7, [20, 40], [3, 3], [1, 2])
    for K in (2, 4, 7):
        res = O.draft_step(SHAPE_F32, w, K, inp, k, v)
        outs.append((res.tokens[::K], res.logits[::K]))
    for tok, lg in outs[1:]:
        assert np.array_equal(tok, outs[0][0])
        assert np.allclose(lg, outs[0][1], rtol=0, atol=1e-11)


def test_requests_are_independent():
    wl, inp, w, k, v = _setup(SHAPE_F32, 14, 3, [7, 25, 13], [4, 4, 4], [3, 0, 1])
    full = O.draft_step(SHAPE_F32, w, 3, inp, k, v)
    for r in range(3):
        one = O.draft_step(SHAPE_F32, w, 3, inp, k, v, requests=[r])
        assert np.array_equal(one.tokens, full.tokens[3 * r:3 * r + 3])
        assert np.allclose(one.logits, full.logits[3 * r:3 * r + 3], rtol=0, atol=1e-11)


def test_paging_is_transparent():
    _, inp, w, k, v = _setup(SHAPE_F32, 15, 4, [18, 35], [5, 5], [4, 2],
                             order="identity")
    base = O.draft_step(SHAPE_F32, w, 4, inp, k, v)
    perm = np.random.default_rng(0).permutation(inp.num_blocks)
    # physical block b moves to perm[b]; the table follows it
    inv_k = [np.empty_like(c) for c in k]
    inv_v = [np.empty_like(c) for c in v]
    for l in range(len(k)):
        inv_k[l][perm] = k[l]
        inv_v[l][perm] = v[l]
    bt = np.where(inp.block_table >= 0, perm[np.maximum(inp.block_table, 0)], -1)
    inp2 = W.StepInputs(inp.target_ids, inp.target_pos, inp.cu_in,
                        inp.num_accepted, inp.sampled_ids, bt.astype(np.int32),
                        inp.num_blocks, inp.target_hidden)
    moved = O.draft_step(SHAPE_F32, w, 4, inp2, inv_k, inv_v)
    assert np.array_equal(base.tokens, moved.tokens)
    assert np.array_equal(base.logits, moved.logits)


def test_rejected_rows_never_write_kv():
    wl, inp, w, k, v = _setup(SHAPE_F32, 16, 5, [10, 3, 50], [6, 6, 6], [0, 5, 2])
    res = O.draft_step(SHAPE_F32, w, 5, inp, k, v)
    ex = res.expanded
    valid_slots = sorted(int(s) for s in ex.slot if s >= 0)
    for wr in res.drafter.kv_writes:
        assert sorted(int(s) for s in wr["slot"]) == valid_slots
    rejected = np.nonzero(ex.is_rejected)[0]
    assert len(rejected) == (6 - 1 - 0) + 0 + (6 - 1 - 2)
    assert not set(rejected.tolist()) & set(res.row_index.tolist())
