"""GPU pin of the draft-token rule (reading R8: greedy argmax, lowest
vocabulary index on exact ties) in the LM-head kernel's fused argmax.

LM-head rows are duplicated so that two vocabulary entries give the same
logit bit for bit (k = 64: one k-block, so every output tile is one
accumulation with the same order); a hidden row equal to the duplicated row
makes the pair the maximum.  The lower index must win whether the two rows
sit in one warp, in different tiles and CTAs, or at the two ends of the
vocabulary; with logits written and without (the benchmarked path), on
narrow token tiles and on the 224-token tiles of the batch-64 LM head.
"""

import numpy as np
import pytest

from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _lm_drafter(V, d, lm, max_tokens):
    sh = W.small_shape("tie", d=d, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                       ffn=64, vocab=V)
    z = np.zeros(64, np.uint16)
    w = {k: z for k in ("emb", "norm_final")}
    # fc is read at pe_create (fc of h_shared): full size
    w["fc"] = np.zeros(sh.d * sh.hidden3, np.uint16)
    w["lm_head"] = lm
    w["h_shared"] = np.zeros(sh.hidden3, np.uint16)
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z,
                        norm_post=z)]
    return G.make_drafter(sh, w, max_tokens, 1)


@pytest.mark.parametrize("V,M", [(4096, 7), (4096, 30), (80000, 300), (80000, 448)],
                         ids=["rows-7", "rows-30", "rows-300", "rows-448"])
@pytest.mark.parametrize("with_logits", [True, False], ids=["logits", "tokens-only"])
def test_exact_ties_return_the_lowest_index(V, M, with_logits):
    B = G.library()
    torch = G.torch_mod()
    d = 64
    lm = W.normal(17, "tie-lm", (V, d), 0.02, "bf16", V)
    pairs = [(130, 131), (3, V // 2 + 5), (0, V - 1), (700, 701 + 128), (V - 200, V - 3)]
    for lo, hi in pairs:
        lm[lo] = lm[hi]
    rows = [pairs[r % len(pairs)] for r in range(M)]
    hid = np.stack([lm[hi] for _, hi in rows])
    dr = _lm_drafter(V, d, lm, max(M, 16))
    hidden = B.to_device(hid, "bf16")
    tok = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    logits = torch.empty(M, V, dtype=torch.float32, device="cuda") if with_logits else None
    for _ in range(2):     # twice: the argmax keys must be left zero for the next call
        B.pe_lmhead_argmax(dr, hidden, tok, logits)
        torch.cuda.synchronize()
        assert B.pe_get_device_error(dr) == 0
        got = tok.cpu().numpy()
        want = np.array([lo for lo, _ in rows])
        assert np.array_equal(got, want), np.nonzero(got != want)
    if with_logits:
        lg = logits.cpu().numpy()
        for r, (lo, hi) in enumerate(rows):
            assert lg[r, lo] == lg[r, hi]
            assert lg[r, lo] > np.delete(lg[r], [lo, hi]).max()
    dr.close()
