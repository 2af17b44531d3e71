"""GPU check of the tensor-core projection kernel through pe_linear.

y = x w^T with bf16 operands and fp32 accumulation (tcgen05, TMEM) against
an fp64 product of the same bf16 values.  The shapes cover one tile, many
tiles, ragged token/feature/k tails, every token-tile width (16..224, 256) and
stream-K splits of a tile across CTAs (the deterministic fix-up path),
including projections with many feature tiles per SM at a few hundred rows
(the LM head at batch 64).
"""

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

CASES = [
    (1, 128, 64),       # one unit
    (14, 5120, 2880),   # GPT-OSS QKV at batch 1 (split across CTAs)
    (16, 300, 200),     # ragged features and k (k % 64 != 0)
    (7, 2880, 8640),    # fc-shaped, long k
    (40, 1000, 512),    # token tile 64
    (100, 640, 1024),   # token tile 128
    (300, 384, 256),    # token tile 256, two token tiles, ragged
    (896, 2880, 2880),  # batch-64 shape
    # at least four feature tiles per SM; ragged tokens, features, k
    (300, 80000, 200),   # two 224-token tiles, ragged
    (448, 80000, 2880),  # the batch-64 LM-head row count, long k
    (500, 80000, 200),   # two 256-token tiles, ragged
    (100, 80000, 256),
]


def _handle(max_tokens, widest=8192):
    # the handle's tile capacity follows its vocabulary and token count
    shape = W.small_shape("lin", d=64, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                          ffn=64, vocab=max(8192, widest))
    z = np.zeros(64, np.uint16)
    w = {k: z for k in ("emb", "norm_final", "lm_head")}
    w["h_shared"] = np.zeros(shape.hidden3, np.uint16)
    w["fc"] = np.zeros(shape.d * shape.hidden3, np.uint16)   # read at pe_create
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z, norm_post=z)]
    return G.make_drafter(shape, w, max_tokens, 1)


@pytest.mark.parametrize("M,N,K", CASES)
def test_linear_matches_fp64(M, N, K):
    B = G.library()
    torch = G.torch_mod()
    dr = _handle(max(M, 16), N)
    x = W.normal(7, "x", (M, K), 1.0, "bf16", M, N)
    w = W.normal(7, "w", (N, K), 0.05, "bf16", M, N)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.pe_linear(dr, B.to_device(x, "bf16"), B.to_device(w, "bf16"), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    want = O.to_f64(x, "bf16") @ O.to_f64(w, "bf16").T
    err = np.abs(got - want).max()
    assert np.isfinite(got).all()
    assert err <= 2e-5 * np.sqrt(K) * max(1.0, np.abs(want).max()), err


def test_linear_is_deterministic():
    B = G.library()
    torch = G.torch_mod()
    dr = _handle(16)
    x = B.to_device(W.normal(8, "x", (14, 2880), 1.0, "bf16"), "bf16")
    w = B.to_device(W.normal(8, "w", (5120, 2880), 0.05, "bf16"), "bf16")
    y1 = torch.empty(14, 5120, device="cuda")
    y2 = torch.empty(14, 5120, device="cuda")
    B.pe_linear(dr, x, w, y1)
    B.pe_linear(dr, x, w, y2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("M,N,K", [(448, 80000, 2880), (700, 70000, 1024), (300, 80000, 1024)])
def test_linear_tile_orders_match_fp64(M, N, K, order):
    # several token tiles under stream-K, weights larger than L2:
    # weight-tile-major, and token-tile-major with the grid cut to a
    # multiple of the token tiles (three of 256 at 700 rows: 150 CTAs);
    # the same sums split at other k-blocks
    B = G.library()
    torch = G.torch_mod()
    dr = _handle(max(M, 16), N)
    B.pe_set_tuning(dr, B.PE_TUNE_GEMM_TILE_ORDER, order)
    x = W.normal(9, "x", (M, K), 1.0, "bf16", M, N)
    w = W.normal(9, "w", (N, K), 0.05, "bf16", M, N)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.pe_linear(dr, B.to_device(x, "bf16"), B.to_device(w, "bf16"), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    want = O.to_f64(x, "bf16") @ O.to_f64(w, "bf16").T
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() <= 2e-5 * np.sqrt(K) * max(1.0, np.abs(want).max())


def test_tile_order_rejects_other_values():
    B = G.library()
    dr = _handle(16)
    for bad in (-1, 2):
        with pytest.raises(B.PeError):
            B.pe_set_tuning(dr, B.PE_TUNE_GEMM_TILE_ORDER, bad)
