"""Pins for the oracle's batch expansion and hidden broadcast (CPU only).

Sources: vLLM blog summary "P-EAGLE: Faster LLM Inference with Parallel
Speculative Decoding in vLLM" -- input formula (Input_i cases), prompt
position handling (row at position i carries the hidden state of i-1), and
the engineering section (fused expansion kernel outputs, hidden-state map
then masked select of h_shared, slot mapping -1 for rejected tokens).
"""

import json
import os

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden", "expand_worked_example.json")


def test_worked_example_matches_hand_derivation():
    g = json.load(open(GOLD))
    bt = np.array(g["block_table"])
    ex = O.expand_batch(g["K"], np.array(g["target_ids"]), np.array(g["target_pos"]),
                        np.array(g["cu_in"]), np.array(g["num_accepted"]),
                        np.array(g["sampled_ids"]), bt, g["page_size"],
                        g["mask_token_id"])
    for key, want in g["expected"].items():
        got = getattr(ex, key)
        assert got.tolist() == want, key


def _random_batch(seed, B, K, page=16, V=500, window=None):
    rng = np.random.default_rng(seed)
    n = rng.integers(1, K + 2, size=B) if window is None else np.full(B, window)
    a = np.array([rng.integers(0, ni) for ni in n])
    C = rng.integers(1, 60, size=B)
    wl = W.custom("t", 900 + seed, W.small_shape(vocab=V, dtype="f32"), K,
                  C, n, a)
    return wl, W.make_step_inputs(wl)


def _slot_of(bt_row, p, page):
    # independent formulation: enumerate the request's slots in order
    table = np.concatenate([np.arange(b * page, (b + 1) * page)
                            for b in bt_row if b >= 0])
    return int(table[p])


@pytest.mark.parametrize("seed,B,K", [(0, 1, 1), (1, 3, 2), (2, 5, 4),
                                      (3, 8, 7), (4, 4, 8), (5, 2, 3)])
def test_expand_invariants(seed, B, K):
    wl, inp = _random_batch(seed, B, K)
    sh = wl.shape
    ex = O.expand_batch(K, inp.target_ids, inp.target_pos, inp.cu_in,
                        inp.num_accepted, inp.sampled_ids, inp.block_table,
                        sh.page_size, sh.mask_token_id)
    T = int(inp.cu_in[-1])
    assert ex.ids.shape[0] == T + B * (K - 1)
    hid = O.expand_hidden(inp.target_hidden, ex.hidden_map, ex.is_masked,
                          np.full(sh.hidden3, 7.0, np.float32))
    written = []
    for r in range(B):
        lo, hi = int(inp.cu_in[r]), int(inp.cu_in[r + 1])
        n, a, s = hi - lo, int(inp.num_accepted[r]), int(inp.sampled_ids[r])
        out = int(ex.cu_out[r])
        assert out == lo + r * (K - 1)
        # shift by one: the row fed by target row t sits at position q_t + 1
        for j in range(n):
            row = int(ex.hidden_map[lo + j])
            assert row == out + j
            assert ex.pos[row] == inp.target_pos[lo + j] + 1
            assert np.array_equal(hid[row], inp.target_hidden[lo + j])
            assert ex.is_masked[row] == 0
            assert ex.is_rejected[row] == (1 if j > a else 0)
            if j < a:   # accepted rows carry the next accepted target token
                assert ex.ids[row] == inp.target_ids[lo + j + 1]
        # input formula: row 1 = emb(new) (+) h_context ...
        ntp = int(ex.new_idx[r * K])
        assert ntp == out + a and ex.ids[ntp] == s
        assert np.array_equal(hid[ntp], inp.target_hidden[lo + a])
        # ... rows 2..K = emb(mask) (+) h_shared
        for k in range(1, K):
            row = int(ex.new_idx[r * K + k])
            assert ex.ids[row] == sh.mask_token_id
            assert ex.is_masked[row] == 1 and ex.is_rejected[row] == 0
            assert np.all(hid[row] == 7.0)
            assert ex.pos[row] == ex.pos[ntp] + k
        # valid positions form one contiguous run ending at seq_len - 1
        valid = [i for i in range(out, out + n + K - 1) if not ex.is_rejected[i]]
        vpos = sorted(int(ex.pos[i]) for i in valid)
        assert vpos == list(range(vpos[0], vpos[0] + len(vpos)))
        assert vpos[0] == inp.target_pos[lo] + 1
        assert ex.seq_lens[r] == vpos[-1] + 1
        # slot mapping: table lookup for valid rows, -1 for rejected rows
        for i in range(out, out + n + K - 1):
            if ex.is_rejected[i]:
                assert ex.slot[i] == -1
            else:
                assert ex.slot[i] == _slot_of(inp.block_table[r], int(ex.pos[i]), sh.page_size)
                written.append(int(ex.slot[i]))
    # every cache write in a step is unique, and rejected rows write nothing
    assert len(written) == len(set(written))
    assert int((ex.slot >= 0).sum()) == int((ex.is_rejected == 0).sum())


def test_expand_rejects_bad_accepted_count():
    with pytest.raises(ValueError):
        O.expand_batch(2, np.array([1, 2]), np.array([0, 1]), np.array([0, 2]),
                       np.array([2]), np.array([3]), np.array([[0]]), 16, 9)


def test_bf16_hidden_copy_is_bitwise():
    wl, inp = _random_batch(7, 4, 5)
    bits = W.normal(1, "h", (inp.target_hidden.shape[0], 12), 1.0, "bf16")
    h_shared = W.normal(1, "hs", (12,), 1.0, "bf16")
    ex = O.expand_batch(5, inp.target_ids, inp.target_pos, inp.cu_in,
                        inp.num_accepted, inp.sampled_ids, inp.block_table,
                        16, 499)
    out = O.expand_hidden(bits, ex.hidden_map, ex.is_masked, h_shared)
    assert out.dtype == np.uint16
    for t in range(bits.shape[0]):
        assert np.array_equal(out[ex.hidden_map[t]], bits[t])
    assert np.all(out[ex.is_masked.astype(bool)] == h_shared)
