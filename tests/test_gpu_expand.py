"""GPU parity of pe_expand_batch (metadata + hidden broadcast): bit-exact.

Rules: vLLM blog summary "P-EAGLE: Faster LLM Inference with Parallel
Speculative Decoding in vLLM", engineering section (fused expansion kernel,
hidden-state management, KV-cache slot mapping with -1 for rejected tokens).
"""

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _expand_drafter(shape, max_tokens, max_reqs):
    """A handle whose only real weight is h_shared (expansion needs no
    other); fc is read at pe_create (fc of h_shared), so it is full size."""
    dt = shape.dtype
    z = np.zeros(64, np.uint16 if dt == "bf16" else np.float32)
    w = {k: z for k in ("emb", "norm_final", "lm_head")}
    w["fc"] = np.zeros(shape.d * shape.hidden3, z.dtype)
    w["h_shared"] = W.normal(77, "h_shared", (shape.hidden3,), 0.02, dt)
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z, norm_post=z)
                   for _ in range(shape.n_layers)]
    return G.make_drafter(shape, w, max_tokens, max_reqs), w["h_shared"]


def _run(wl, shape=None):
    B = G.library()
    torch = G.torch_mod()
    shape = shape or wl.shape
    inp = W.make_step_inputs(wl)
    dr, h_shared = _expand_drafter(shape, wl.T_out, wl.B)
    st = G.DeviceStep(wl, inp, [], [])
    ex = B.Expanded(wl.T_out, wl.T, wl.B, wl.K, shape.hidden3, shape.dtype)
    B.pe_expand_batch(dr, wl.K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                      st.sampled_ids, st.block_table, inp.num_blocks, st.target_hidden, ex)
    torch.cuda.synchronize()
    assert B.pe_get_device_error(dr) == 0
    ref = O.expand_batch(wl.K, inp.target_ids, inp.target_pos, inp.cu_in, inp.num_accepted,
                         inp.sampled_ids, inp.block_table, shape.page_size, shape.mask_token_id)
    G.check_expand(ex, ref, wl.T)
    want_h = O.expand_hidden(inp.target_hidden, ref.hidden_map, ref.is_masked, h_shared)
    got_h = B.to_host(ex.hidden)
    assert got_h.dtype == want_h.dtype
    assert np.array_equal(got_h.view(np.uint8), want_h.view(np.uint8))
    return dr


def test_expand_microbench_config_bit_exact():
    """256 requests, K=7, accepted counts uniform 0..7, hidden width 8640."""
    _run(W.expand_b256())


EDGE = [
    # (contexts, windows, accepted, K)
    ([1], [1], [0], 1),                       # smallest: n=1, K=1
    ([15], [2], [1], 1),                      # K=1 (AR step), page boundary
    ([16], [8], [0], 7),                      # all drafts rejected
    ([17], [8], [7], 7),                      # all drafts accepted
    ([15, 16, 17], [3, 5, 9], [2, 0, 8], 8),  # ragged windows, K=8
    ([31, 1, 64, 100], [4, 1, 2, 6], [3, 0, 1, 2], 16),
]


@pytest.mark.parametrize("ctx,win,acc,K", EDGE)
def test_expand_edge_cases(ctx, win, acc, K):
    shape = W.small_shape("edge", d=64, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                          ffn=64, vocab=500)
    wl = W.custom("edge", 31, shape, K, ctx, win, acc)
    _run(wl)


@pytest.mark.parametrize("B", [1, 3, 64])
def test_expand_random_batches(B):
    rng = np.random.default_rng(B)
    K = int(rng.integers(1, 9))
    win = rng.integers(1, K + 2, size=B)
    acc = np.array([rng.integers(0, n) for n in win])
    ctx = rng.integers(1, 3000, size=B)
    shape = W.small_shape("rand", d=128, n_layers=1, n_heads=2, n_kv_heads=1, head_dim=64,
                          ffn=64, vocab=1000)
    _run(W.custom("rand", 40 + B, shape, K, ctx, win, acc))


def test_expand_f32_hidden_rows():
    shape = W.small_shape("f32", d=64, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                          ffn=64, vocab=300, dtype="f32")
    _run(W.custom("f32", 50, shape, 4, [20, 33], [5, 3], [4, 1]))


def test_bad_accepted_count_is_reported_not_trapped():
    shape = W.small_shape("bad", d=64, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                          ffn=64, vocab=300)
    B = G.library()
    torch = G.torch_mod()
    wl = W.custom("bad", 51, shape, 3, [20], [4], [2])
    inp = W.make_step_inputs(wl)
    inp.num_accepted[:] = 9          # outside [0, n-1]: a data-dependent violation
    dr, _ = _expand_drafter(shape, wl.T_out, wl.B)
    st = G.DeviceStep(wl, inp, [], [])
    ex = B.Expanded(wl.T_out, wl.T, wl.B, wl.K, shape.hidden3, shape.dtype)
    B.pe_expand_batch(dr, wl.K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                      st.sampled_ids, st.block_table, inp.num_blocks, st.target_hidden, ex)
    torch.cuda.synchronize()
    assert B.pe_get_device_error(dr) == 1          # PE_DEV_BAD_ACCEPTED
    assert B.pe_get_device_error(dr) == 0          # cleared by the read
