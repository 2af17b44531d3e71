"""Helpers for the GPU parity tests: run one drafting step through the C ABI
on seeded synthetic inputs and compare it with the CPU oracle."""

import json
import os

import numpy as np

import oracle as O
from synthetic import workloads as W


def torch_mod():
    import torch
    return torch


def library():
    from speculative_drafting_expand_gb300 import binding as B
    B.lib()  # fails loudly if the library is missing
    return B


class DeviceStep:
    """Device copies of one step's inputs and caches."""

    def __init__(self, wl, inp, kc, vc):
        B = library()
        torch = torch_mod()
        dt = wl.shape.dtype
        self.wl, self.inp = wl, inp
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
        self.target_ids = i32(inp.target_ids)
        self.target_pos = i32(inp.target_pos)
        self.cu_in = i32(inp.cu_in)
        self.num_accepted = i32(inp.num_accepted)
        self.sampled_ids = i32(inp.sampled_ids)
        self.block_table = i32(inp.block_table)
        self.target_hidden = B.to_device(inp.target_hidden, dt)
        self.kc = [B.to_device(k, dt) for k in kc]
        self.vc = [B.to_device(v, dt) for v in vc]


def run_step(dr, st: "DeviceStep", want_logits=True):
    B = library()
    torch = torch_mod()
    wl, sh = st.wl, st.wl.shape
    K = wl.K
    Bn = wl.B
    T = int(st.inp.cu_in[-1])
    T_out = T + Bn * (K - 1)
    ex = B.Expanded(T_out, T, Bn, K, sh.hidden3, sh.dtype)
    B.pe_expand_batch(dr, K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                      st.sampled_ids, st.block_table, st.inp.num_blocks, st.target_hidden, ex)
    tdt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
    out_hidden = torch.empty(Bn * K, sh.d, dtype=tdt, device="cuda")
    B.pe_draft_forward(dr, ex, st.block_table, st.kc, st.vc, st.inp.num_blocks, out_hidden)
    tokens = torch.empty(Bn * K, dtype=torch.int32, device="cuda")
    logits = torch.empty(Bn * K, sh.vocab, dtype=torch.float32, device="cuda") if want_logits else None
    B.pe_lmhead_argmax(dr, out_hidden, tokens, logits)
    torch.cuda.synchronize()
    err = B.pe_get_device_error(dr)
    return dict(ex=ex, out_hidden=out_hidden, tokens=tokens, logits=logits, err=err)


def f64(a, dtype):
    return O.to_f64(a, dtype)


def margin_ok_tokens(ref_logits, ref_tokens, got_tokens, margin=1e-2):
    """Tokens must agree wherever the oracle's top-2 margin exceeds `margin`;
    elsewhere the GPU's token must be within `margin` of the top logit."""
    srt = np.sort(ref_logits, axis=1)
    gap = srt[:, -1] - srt[:, -2]
    for i in range(len(ref_tokens)):
        if gap[i] > margin:
            assert got_tokens[i] == ref_tokens[i], (i, gap[i])
        else:
            assert ref_logits[i, got_tokens[i]] >= srt[i, -1] - margin, i
    return int((gap <= margin).sum())


def token_rule_stats(name, ref_logits, ref_tokens, got_tokens, loose_margin):
    """How many draft tokens the spec rule (identical wherever the
    oracle's top-2 margin exceeds 1e-2) pins, how many the rule this suite
    applies end to end (margin above `loose_margin`) pins, and how many
    tokens with 1e-2 < margin <= loose_margin disagree.  Printed, and
    appended as a JSON line to $PE_TOKEN_STATS when that is set."""
    srt = np.sort(ref_logits, axis=1)
    gap = srt[:, -1] - srt[:, -2]
    agree = np.asarray(got_tokens) == np.asarray(ref_tokens)
    between = (gap > 1e-2) & (gap <= loose_margin)
    st = {"workload": name, "tokens": int(len(gap)),
          "pinned_at_1e-2": int((gap > 1e-2).sum()),
          "pinned_at_loose": int((gap > loose_margin).sum()),
          "loose_margin": float(loose_margin),
          "disagree_between": int((between & ~agree).sum()),
          "disagree_at_or_below_1e-2": int(((gap <= 1e-2) & ~agree).sum()),
          "min_margin_of_a_disagreement": (float(gap[~agree].min()) if (~agree).any() else None)}
    print("TOKEN-RULE", json.dumps(st))
    path = os.environ.get("PE_TOKEN_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(st) + "\n")
    return st


def check_expand(res_ex, ref_ex, T):
    B = library()
    for f in ("ids", "pos", "slot", "new_idx", "cu_out", "seq_lens"):
        got = B.to_host(getattr(res_ex, f))
        assert np.array_equal(got, getattr(ref_ex, f)), f
    assert np.array_equal(B.to_host(res_ex.hidden_map), ref_ex.hidden_map)
    assert np.array_equal(B.to_host(res_ex.is_rejected), ref_ex.is_rejected)
    assert np.array_equal(B.to_host(res_ex.is_masked), ref_ex.is_masked)


def check_kv(st, ref, shape, tol_rel):
    """Written slots hold the oracle's k/v; every other slot is unchanged."""
    B = library()
    P = shape.page_size
    for l in range(shape.n_layers):
        for name, dev, host in (("k", st.kc[l], None), ("v", st.vc[l], None)):
            got = B.to_host(dev)
            orig = (st_host_cache(st, name, l))
            wr = ref.drafter.kv_writes[l]
            written = np.zeros(got.shape[0] * P, bool)
            for i, s in enumerate(wr["slot"]):
                blk, off = divmod(int(s), P)
                g = f64(got[blk, :, off, :], shape.dtype)
                want = wr[name][i]
                scale = max(1e-30, np.abs(want).max())
                assert np.abs(g - want).max() <= tol_rel * scale, (l, name, i)
                written[s] = True
            # untouched slots: bitwise identical to the input pool
            g2 = got.transpose(0, 2, 1, 3).reshape(-1, got.shape[1], got.shape[3])
            o2 = orig.transpose(0, 2, 1, 3).reshape(-1, got.shape[1], got.shape[3])
            assert np.array_equal(g2[~written].view(np.uint8), o2[~written].view(np.uint8)), (l, name)


_HOST_CACHES = {}


def remember_host_caches(st, kc, vc):
    _HOST_CACHES[id(st)] = (kc, vc)


def st_host_cache(st, name, l):
    kc, vc = _HOST_CACHES[id(st)]
    return (kc if name == "k" else vc)[l]


def make_drafter(shape, weights, max_tokens, max_reqs):
    B = library()
    return B.Drafter(shape, weights, max_tokens, max_reqs)


def full_parity(wl, tol, gains=None, requests=None, check_cache=True, strict_tokens=True,
                configure=None):
    """Run one step on the GPU and the oracle; assert parity.  Returns both.

    strict_tokens (default): end-to-end tokens identical to the fp64
    oracle's wherever its top-2 margin exceeds 1e-2, the spec rule
    itself.  Measured on every configuration of the suite, no token with a
    margin between 1e-2 and twice the logit tolerance disagreed, so the
    looser bound (strict_tokens=False) is only reported, not applied."""
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=gains or wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    max_tokens = max(wl.T_out, wl.B * wl.K)
    dr = make_drafter(sh, w, max_tokens, wl.B)
    if configure is not None:
        configure(dr)      # e.g. select the small-batch streaming path
    st = DeviceStep(wl, inp, kc, vc)
    remember_host_caches(st, kc, vc)
    torch = torch_mod()
    B = library()
    tdt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
    qd = sh.n_heads * sh.head_dim
    attn_trace = torch.zeros(sh.n_layers, max_tokens, qd, dtype=tdt, device="cuda")
    B.pe_set_trace(dr, None, attn_trace)
    res = run_step(dr, st, want_logits=True)
    assert res["err"] == 0, res["err"]
    ref = O.draft_step(sh, w, wl.K, inp, kc, vc, requests=requests)
    check_expand(res["ex"], ref.expanded, wl.T)
    # attention output of every row the oracle computed, layer by layer
    at = B.to_host(attn_trace)
    for l in range(sh.n_layers):
        got_a = f64(at[l][ref.row_index], sh.dtype)
        want_a = ref.drafter.layer_attn[l].reshape(len(ref.row_index), qd)
        scale = np.abs(want_a).max()
        err = np.abs(got_a - want_a).max()
        assert err <= 1.5 * tol * scale, ("attention", l, err / scale)
    ex = ref.expanded
    dead = [i for i in range(len(ex.ids)) if ex.is_rejected[i]
            and int(ex.request_of_row[i]) in set(ref.requests)]
    for l in range(sh.n_layers):
        assert not np.any(f64(at[l][dead], sh.dtype)), ("rejected rows attend", l)
    rows = np.concatenate([np.arange(r * wl.K, (r + 1) * wl.K) for r in ref.requests])
    got_h = f64(B.to_host(res["out_hidden"]), sh.dtype)[rows]
    hs = np.abs(ref.out_hidden).max()
    assert np.abs(got_h - ref.out_hidden).max() <= tol * hs, np.abs(got_h - ref.out_hidden).max() / hs
    got_l = B.to_host(res["logits"]).astype(np.float64)[rows]
    ls = np.abs(ref.logits).max()
    assert np.abs(got_l - ref.logits).max() <= tol * ls, np.abs(got_l - ref.logits).max() / ls
    got_t = B.to_host(res["tokens"])[rows]
    # End to end the logits may differ from the fp64 statement by up to
    # tol x max|logit|, so a token is pinned wherever the oracle's top-2
    # margin is more than twice that (for fp32 the stated 1e-2 margin).
    loose = max(1e-2, 2 * tol * ls)
    token_rule_stats(wl.name, ref.logits, ref.tokens, got_t, loose)
    margin_ok_tokens(ref.logits, ref.tokens, got_t, margin=1e-2 if strict_tokens else loose)
    # The argmax decision itself, taken in the same precision on both sides:
    # the oracle's LM head on the GPU's own final hidden rows.  Logits agree
    # to the GEMM's fp32 accumulation and tokens wherever the margin > 1e-3.
    lm_logits, lm_tokens = O.lm_head_argmax(sh, w, f64(B.to_host(res["out_hidden"]), sh.dtype)[rows])
    lm_err = np.abs(got_l - lm_logits).max()
    assert lm_err <= 1e-4 * np.abs(lm_logits).max(), lm_err
    margin_ok_tokens(lm_logits, lm_tokens, got_t, margin=1e-3)
    if check_cache and requests is None:
        check_kv(st, ref, sh, tol * 2)
    return res, ref, dr, st


def tokens_only_parity(wl, tol, requests=None):
    """The benchmarked path: pe_lmhead_argmax with no logits buffer (the
    argmax epilogue alone).  Its tokens must equal the oracle's LM head on
    the GPU's own final hidden rows wherever that margin exceeds 1e-3, and
    the fp64 oracle's end to end under the same rule as full_parity."""
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    dr = make_drafter(sh, w, max(wl.T_out, wl.B * wl.K), wl.B)
    st = DeviceStep(wl, inp, kc, vc)
    res = run_step(dr, st, want_logits=False)
    assert res["err"] == 0, res["err"]
    B = library()
    ref = O.draft_step(sh, w, wl.K, inp, kc, vc, requests=requests)
    rows = np.concatenate([np.arange(r * wl.K, (r + 1) * wl.K) for r in ref.requests])
    got_t = B.to_host(res["tokens"])[rows]
    hid = f64(B.to_host(res["out_hidden"]), sh.dtype)[rows]
    lm_logits, lm_tokens = O.lm_head_argmax(sh, w, hid)
    margin_ok_tokens(lm_logits, lm_tokens, got_t, margin=1e-3)
    ls = np.abs(ref.logits).max()
    token_rule_stats(wl.name + "-tokens-only", ref.logits, ref.tokens, got_t,
                     max(1e-2, 2 * tol * ls))
    margin_ok_tokens(ref.logits, ref.tokens, got_t, margin=1e-2)
    dr.close()
    return got_t, ref
