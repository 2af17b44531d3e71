"""GPU parity of the whole drafting step (pe_expand_batch -> pe_draft_forward
-> pe_lmhead_argmax) against the CPU oracle.

Bar: metadata bit-exact; final hidden states and logits within
max-abs <= tol x max|value| (1e-4 for the fp32 path, 2e-2 for bf16); draft
tokens identical wherever the fp64 oracle's top-2 logit margin exceeds 1e-2
(elsewhere within 1e-2 of the top logit); the LM-head argmax decision on
the GPU's own final hidden rows identical to the oracle's wherever the
margin exceeds 1e-3; KV writes at exactly the non-rejected slots, every
other slot untouched.
"""

import numpy as np
import pytest

from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def test_tiny_fp32_config():
    """Tiny fp32 drafter: d=256, 2 layers, 4x64 heads, ctx 64, K=4."""
    G.full_parity(W.tiny_fp32(), TOL_F32)


def test_tiny_fp32_with_rejections_and_random_gains():
    wl = W.custom("tiny-rej", 61, W.TINY, 5, [40, 17, 90], [6, 6, 3], [2, 5, 0],
                  gains="random")
    G.full_parity(wl, TOL_F32)


SMALL = W.small_shape("small-bf16", d=512, n_layers=2, n_heads=8, n_kv_heads=2,
                      head_dim=64, ffn=1024, vocab=4096)


@pytest.mark.parametrize("B,K", [(1, 7), (4, 5), (16, 8)])
def test_small_bf16_batches(B, K):
    rng = np.random.default_rng(B * 10 + K)
    ctx = rng.integers(1, 600, size=B)
    win = np.full(B, K + 1)
    acc = rng.integers(0, K + 1, size=B)
    wl = W.custom(f"small-b{B}", 70 + B, SMALL, K, ctx, win, acc, gains="random")
    G.full_parity(wl, TOL_BF16)


@pytest.mark.parametrize("B", [22, 40])
def test_rejected_rows_are_skipped_by_whole_token_tiles(B):
    """Every request accepts nothing (a = 0 of an 8-row window), so the
    layers run on B*K live rows of the 2*B*K expanded ones.  B = 22: 308
    rows in two 224-row token tiles, the second one dead (cluster split:
    its clusters exit); B = 40: 560 rows in three tiles, one dead.  The
    attention trace of every rejected row must still read zero and the KV
    cache must change at the live slots only."""
    K = 7
    rng = np.random.default_rng(900 + B)
    ctx = rng.integers(1, 400, size=B)
    wl = W.custom(f"dead-b{B}", 90 + B, SMALL, K, ctx, np.full(B, K + 1), np.zeros(B, int),
                  gains="random")
    G.full_parity(wl, TOL_BF16)


def test_small_bf16_head_dim_128():
    sh = W.small_shape("small-dh128", d=512, n_layers=2, n_heads=4, n_kv_heads=2,
                       head_dim=128, ffn=768, vocab=2048)
    wl = W.custom("dh128", 80, sh, 4, [33, 250], [5, 5], [4, 1], gains="random")
    G.full_parity(wl, TOL_BF16)


def test_k1_is_one_autoregressive_step_on_gpu():
    import oracle as O
    wl = W.custom("k1", 81, SMALL, 1, [100, 7, 300], [2, 3, 1], [1, 2, 0], gains="random")
    res, ref, dr, st = G.full_parity(wl, TOL_BF16)
    kc, vc = W.make_kv_cache(wl, st.inp)   # the pools as they were before the step
    logits, tokens = O.ar_eagle_step(SMALL, W.make_weights(SMALL, 81, gains="random"),
                                     st.inp, kc, vc)
    B = G.library()
    G.token_rule_stats("k1-ar-eagle", logits, tokens, B.to_host(res["tokens"]),
                       2 * TOL_BF16 * np.abs(logits).max())
    G.margin_ok_tokens(logits, tokens, B.to_host(res["tokens"]), margin=1e-2)


def test_gpt_oss_b1_full_size():
    """GPT-OSS-20B-shaped drafter, bf16, one request, K=7, context 4096."""
    G.full_parity(W.gpt_oss_b1(), TOL_BF16)


def _sample_requests(wl, n=3):
    """The longest context, a request with everything rejected (if any), and
    one more: requests are independent, so the oracle checks a sample."""
    order = np.argsort(-wl.contexts)
    pick = [int(order[0])]
    zero = [i for i in range(wl.B) if wl.accepted[i] == 0 and i not in pick]
    if zero:
        pick.append(zero[0])
    for i in range(wl.B):
        if len(pick) >= n:
            break
        if i not in pick:
            pick.append(i)
    return sorted(pick)


def test_gpt_oss_b64_full_size_sampled_requests():
    """GPT-OSS-20B-shaped drafter at batch 64, K=7, lognormal contexts."""
    wl = W.gpt_oss_b64()
    G.full_parity(wl, TOL_BF16, requests=_sample_requests(wl))


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 8])
def test_qwen_b16_full_size_sampled_requests(K):
    """Qwen3-Coder-30B-shaped drafter (head_dim 128), batch 16, the K sweep
    1..8 of the configuration (K = 1 is one autoregressive EAGLE step)."""
    wl = W.qwen_b16(K)
    G.full_parity(wl, TOL_BF16, requests=_sample_requests(wl, 2))


@pytest.mark.parametrize("make_wl,sample", [(W.gpt_oss_b1, False), (W.gpt_oss_b64, True)],
                         ids=["gpt-oss-b1", "gpt-oss-b64"])
def test_benchmarked_path_without_logits(make_wl, sample):
    """pe_lmhead_argmax with out_logits = NULL, the call the benchmark
    times: tokens against the oracle's LM head on the GPU's own hidden rows
    (margin 1e-3) and against the fp64 oracle end to end."""
    wl = make_wl()
    G.tokens_only_parity(wl, TOL_BF16, requests=_sample_requests(wl) if sample else None)


@pytest.mark.parametrize("make_wl,repeats", [(W.gpt_oss_b1, 40), (W.gpt_oss_b64, 40)],
                         ids=["gpt-oss-b1", "gpt-oss-b64"])
def test_repeated_steps_are_bitwise_identical(make_wl, repeats):
    """Every kernel of the step is deterministic (split-ordered merges, a
    fixed stream-K fix-up order), and rewriting the KV slots with the same
    values is idempotent, so the same step run again must give bit-identical
    attention outputs, hidden states and tokens, with no device error.  A
    race between the warps of a kernel (barrier phases completed early, a
    buffer read before it is written) shows up here as a mismatch or as a
    recorded timeout, even when one run happens to pass the parity tests."""
    wl = make_wl()
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    max_tokens = max(wl.T_out, wl.B * wl.K)
    dr = G.make_drafter(sh, w, max_tokens, wl.B)
    st = G.DeviceStep(wl, inp, kc, vc)
    torch = G.torch_mod()
    B = G.library()
    qd = sh.n_heads * sh.head_dim
    trace = torch.zeros(sh.n_layers, max_tokens, qd, dtype=torch.bfloat16, device="cuda")
    B.pe_set_trace(dr, None, trace)
    first = G.run_step(dr, st, want_logits=False)
    assert first["err"] == 0, first["err"]
    trace0 = trace.clone()
    for i in range(repeats - 1):
        trace.zero_()
        res = G.run_step(dr, st, want_logits=False)
        assert res["err"] == 0, (i, res["err"])
        assert torch.equal(trace, trace0), ("attention", i)
        assert torch.equal(res["out_hidden"], first["out_hidden"]), ("hidden", i)
        assert torch.equal(res["tokens"], first["tokens"]), ("tokens", i)


@pytest.mark.parametrize("B,K,shape", [(1, 7, "small"), (2, 7, "small"), (3, 5, "dh128"),
                                       (1, 7, "gpt-oss")],
                         ids=["small-b1-k7", "small-b2-k7-tile32", "dh128-b3-k5",
                              "gpt-oss-b1-k7"])
def test_small_batch_stream_matches_the_per_projection_path(B, K, shape):
    """Up to 32 expanded rows the step can run its projections as persistent
    segments (RMSNorm folded into the consuming projection as a row scale,
    RoPE and the KV write in the QKV epilogue).  That path must match the
    oracle on its own, and agree with the per-projection kernels to the
    bf16 tolerance."""
    torch = G.torch_mod()
    Bm = G.library()
    if shape == "gpt-oss":
        wl = W.gpt_oss_b1()
    else:
        sh = SMALL if shape == "small" else W.small_shape(
            "small-dh128", d=512, n_layers=2, n_heads=4, n_kv_heads=1, head_dim=128, ffn=768,
            vocab=2048)
        rng = np.random.default_rng(700 + B * 10 + K)
        wl = W.custom(f"stream-{shape}-b{B}", 700 + B, sh, K, rng.integers(20, 500, size=B),
                      np.full(B, K + 1), rng.integers(0, K + 1, size=B), gains="random")
    # Its bf16 roundings differ from the default path's (it rounds x g and
    # scales by r after the product), and on the GPT-OSS b1 step that flips
    # one token whose fp64 margin is 0.017: end-to-end tokens are held to
    # twice the logit tolerance here, the argmax itself still to 1e-3.
    G.full_parity(wl, TOL_BF16, configure=lambda dr: Bm.pe_set_small_batch_stream(dr, True),
                  strict_tokens=False)
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    outs = []
    for stream in (True, False):
        dr = G.make_drafter(sh, w, max(wl.T_out, wl.B * wl.K), wl.B)
        Bm.pe_set_small_batch_stream(dr, stream)
        st = G.DeviceStep(wl, inp, kc, vc)
        res = G.run_step(dr, st, want_logits=True)
        assert res["err"] == 0
        outs.append((G.f64(Bm.to_host(res["out_hidden"]), sh.dtype),
                     Bm.to_host(res["logits"]).astype(np.float64),
                     [G.f64(Bm.to_host(k), sh.dtype) for k in st.kc]))
        dr.close()
    (h1, l1, k1), (h2, l2, k2) = outs
    assert np.abs(h1 - h2).max() <= TOL_BF16 * np.abs(h2).max()
    assert np.abs(l1 - l2).max() <= TOL_BF16 * np.abs(l2).max()
    for a, b in zip(k1, k2):
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin)          # the same slots written
        assert np.abs(a[fin] - b[fin]).max() <= TOL_BF16 * np.abs(b[fin]).max()


@pytest.mark.parametrize("mask", ["none", "rope_kv", "all"])
@pytest.mark.parametrize("B,K,shape", [(4, 5, "small"), (1, 7, "dh128"), (1, 7, "gpt-oss")])
def test_projection_fusions_match_the_oracle(mask, B, K, shape):
    """Each fusion option of the per-projection path (none; RoPE + KV write
    in the QKV epilogue; that plus RMSNorm folded into the projections as a
    row scale) matches the oracle on its own.  The RoPE epilogue reads the
    QKV weight as an interleaved copy the drafter makes when the option is
    switched on."""
    Bm = G.library()
    m = {"none": 0, "rope_kv": Bm.PE_FUSE_ROPE_KV, "all": Bm.PE_FUSE_ALL}[mask]
    if shape == "gpt-oss":
        wl = W.gpt_oss_b1()
    else:
        sh = SMALL if shape == "small" else W.small_shape(
            "small-dh128", d=512, n_layers=2, n_heads=4, n_kv_heads=1, head_dim=128, ffn=768,
            vocab=2048)
        rng = np.random.default_rng(900 + B * 10 + K)
        wl = W.custom(f"fuse-{shape}-b{B}", 900 + B, sh, K, rng.integers(20, 500, size=B),
                      np.full(B, K + 1), rng.integers(0, K + 1, size=B), gains="random")
    G.full_parity(wl, TOL_BF16, configure=lambda dr: Bm.pe_set_fusions(dr, m))


@pytest.mark.parametrize("B,K,shape", [(1, 7, "gpt-oss"), (4, 7, "small"), (2, 5, "dh128")])
def test_pushed_and_pulled_split_reductions_are_bit_identical(B, K, shape):
    """The cluster split-K projections add their partials in rank order
    whether the partials are pushed to the owning CTA or pulled by it, so
    the whole step's outputs agree bit for bit; the pushed default also
    matches the oracle on its own."""
    Bm = G.library()
    if shape == "gpt-oss":
        wl = W.gpt_oss_b1()
    else:
        sh = SMALL if shape == "small" else W.small_shape(
            "small-dh128", d=512, n_layers=2, n_heads=4, n_kv_heads=1, head_dim=128, ffn=768,
            vocab=2048)
        rng = np.random.default_rng(950 + B * 10 + K)
        wl = W.custom(f"reduce-{shape}-b{B}", 950 + B, sh, K, rng.integers(20, 500, size=B),
                      np.full(B, K + 1), rng.integers(0, K + 1, size=B), gains="random")
    G.full_parity(wl, TOL_BF16, configure=lambda dr: Bm.pe_set_split_reduce(dr, Bm.PE_REDUCE_PUSH))
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    outs = []
    for mode in (Bm.PE_REDUCE_PUSH, Bm.PE_REDUCE_PULL):
        dr = G.make_drafter(sh, w, max(wl.T_out, wl.B * wl.K), wl.B)
        Bm.pe_set_split_reduce(dr, mode)
        st = G.DeviceStep(wl, inp, kc, vc)
        res = G.run_step(dr, st, want_logits=True)
        assert res["err"] == 0
        outs.append((Bm.to_host(res["out_hidden"]), Bm.to_host(res["logits"]),
                     Bm.to_host(res["tokens"]), [Bm.to_host(k) for k in st.kc]))
        dr.close()
    (h1, l1, t1, k1), (h2, l2, t2, k2) = outs
    assert h1.tobytes() == h2.tobytes()
    assert l1.tobytes() == l2.tobytes()
    assert np.array_equal(t1, t2)
    for a, b in zip(k1, k2):
        assert a.tobytes() == b.tobytes()
