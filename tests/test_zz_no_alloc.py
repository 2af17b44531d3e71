"""pe_linear_static: the projection entry point for callers that cannot
allocate device memory (allocator callbacks, frameworks that own all device
memory, paths that must stay out of the driver's allocator).  Its scratch is
a static array inside the library, so it needs no handle.

Checked through the C ABI against pe_linear (the handle-based entry point) on
two calls in a row -- the second call reuses the array the first one left
behind -- against an fp64 product of the same bf16 values, for its error
word (read and cleared by pe_linear_static_error), and for its refusal of
sizes beyond the array.  This file is
collected last so that a run stopping at the first failure has run every
other test already.
"""

import numpy as np
import pytest

import oracle as O
from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _reference_handle(max_tokens):
    shape = W.small_shape("static-ref", d=64, n_layers=1, n_heads=1, n_kv_heads=1,
                          head_dim=64, ffn=64, vocab=32768)
    z = np.zeros(64, np.uint16)
    w = {k: z for k in ("emb", "norm_final", "lm_head")}
    w["h_shared"] = np.zeros(shape.hidden3, np.uint16)
    w["fc"] = np.zeros(shape.d * shape.hidden3, np.uint16)   # read at pe_create
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z,
                        norm_post=z)]
    return G.make_drafter(shape, w, max_tokens, 1)


@pytest.mark.parametrize("M,N,K", [(14, 5120, 2880), (7, 2880, 8640), (32, 300, 200),
                                   (7, 20480, 2880)])
def test_static_entry_point_matches_pe_linear_twice(M, N, K):
    B = G.library()
    torch = G.torch_mod()
    dr = _reference_handle(max(M, 16))
    x = B.to_device(W.normal(9, "sx", (M, K), 1.0, "bf16", M, N), "bf16")
    w = B.to_device(W.normal(9, "sw", (N, K), 0.05, "bf16", M, N), "bf16")
    want = torch.empty(M, N, dtype=torch.float32, device="cuda")
    B.pe_linear(dr, x, w, want)
    torch.cuda.synchronize()
    ref = want.cpu().numpy().astype(np.float64)
    tol = 2e-5 * np.sqrt(K) * max(1.0, np.abs(ref).max())
    for _ in range(2):
        got = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        B.pe_linear_static(x, w, got)
        torch.cuda.synchronize()
        g = got.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        assert np.abs(g - ref).max() <= tol
    assert B.pe_linear_static_error() == 0


def test_static_entry_point_matches_fp64_product():
    """The static entry point against x . w^T in fp64 on the same bf16
    values (not only against the handle-based call, which runs the same
    kernel): the bf16 drafter tolerance of 2e-2 x max|y|."""
    B = G.library()
    torch = G.torch_mod()
    M, N, K = 14, 5120, 2880
    x = W.normal(11, "sx", (M, K), 1.0, "bf16", M, N)
    w = W.normal(11, "sw", (N, K), 0.05, "bf16", M, N)
    want = O.to_f64(x, "bf16") @ O.to_f64(w, "bf16").T
    for _ in range(2):
        got = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        B.pe_linear_static(B.to_device(x, "bf16"), B.to_device(w, "bf16"), got)
        torch.cuda.synchronize()
        g = got.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        assert np.abs(g - want).max() <= 2e-2 * np.abs(want).max()
    assert B.pe_linear_static_error() == 0


def test_static_entry_point_refuses_sizes_beyond_its_array():
    B = G.library()
    torch = G.torch_mod()
    x = torch.zeros(33, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(33, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(B.PeError) as info:
        B.pe_linear_static(x, w, y)
    assert info.value.status == B.PE_ERR_UNSUPPORTED
