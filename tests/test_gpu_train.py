"""GPU parity of the training-side index kernels (include/peagle_train.h)
against the training oracle: the amortized mask bit for bit (boolean and
additive bf16), its per-sample views, and COD sampling + sequence
partitioning (keep flags, owning segments, segment row lists) bit for bit,
on the Figure 4 shape (n = 16, K = 4), ragged random shapes, and the
8192-token, K = 8, r = 0.8 example of the paper summary's section 3.2."""

import numpy as np
import pytest

from oracle import training_oracle as TO

pytestmark = pytest.mark.gpu


def _lib():
    from speculative_drafting_expand_gb300 import binding as B
    return B


def _mask_gpu(n_max, K, mask_type, pad=0):
    import torch
    B = _lib()
    N = n_max * K
    eb = 1 if mask_type == B.PE_MASK_BOOL_U8 else 2
    ld = N + pad
    assert (ld * eb) % 16 == 0
    # prefilled with a value the kernel never writes, so a skipped chunk shows
    if eb == 1:
        out = torch.full((N, ld), 7, dtype=torch.uint8, device="cuda")
    else:
        out = torch.full((N, ld), 3.0, dtype=torch.bfloat16, device="cuda")
    B.pe_train_build_mask(out, n_max, K, mask_type)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("n_max,K,pad", [(12, 4, 0), (24, 2, 16), (16, 1, 0), (20, 8, 32)])
def test_boolean_mask_bit_exact_and_views(n_max, K, pad):
    import torch
    B = _lib()
    m = _mask_gpu(n_max, K, B.PE_MASK_BOOL_U8, pad)
    want = TO.build_mask(n_max, K)
    got = m.cpu().numpy()
    assert np.array_equal(got[:, : n_max * K], want.astype(np.uint8))
    assert not got[:, n_max * K:].any()
    for n in (1, n_max // 2, n_max):
        v = B.pe_train_mask_view(m, n_max, K, n)
        assert v.data_ptr() == m.data_ptr()
        assert torch.equal(v.cpu(), torch.from_numpy(TO.build_mask(n, K).astype(np.uint8)))


def test_additive_bf16_mask_bit_exact():
    import torch
    B = _lib()
    n_max, K = 16, 4
    m = _mask_gpu(n_max, K, B.PE_MASK_ADDITIVE_BF16, pad=8)
    bits = m.view(torch.int16).cpu().numpy().view(np.uint16)
    want = np.where(TO.build_mask(n_max, K), 0x0000, 0xFF80).astype(np.uint16)
    assert np.array_equal(bits[:, : n_max * K], want)
    assert np.all(bits[:, n_max * K:] == 0xFF80)


def test_full_size_mask_rows_attend_positions_zero_to_p():
    """The 8192-token, K = 8 mask (65,536 rows, 4.3 GB as bytes): each row
    (p, d) allows exactly p + 1 columns (none for p < d), and sampled rows
    equal the oracle's rule entry by entry."""
    import torch
    B = _lib()
    n_max, K = 8192, 8
    N = n_max * K
    m = torch.empty((N, N), dtype=torch.uint8, device="cuda")
    B.pe_train_build_mask(m, n_max, K, B.PE_MASK_BOOL_U8)
    assert int(m.max()) == 1
    sums = torch.zeros(N, dtype=torch.int64, device="cuda")
    for lo in range(0, N, 4096):
        sums[lo:lo + 4096] = torch.count_nonzero(m[lo:lo + 4096], dim=1)
    p = torch.arange(N, device="cuda") // K
    d = torch.arange(N, device="cuda") % K
    want = torch.where(p >= d, p + 1, torch.zeros_like(p))
    assert torch.equal(sums, want)
    rng = np.random.default_rng(5)
    for i in rng.integers(0, N, size=6).tolist() + [N - 1, 7 * K + 7]:
        row = m[i].cpu().numpy()
        pp, dd = divmod(i, K)
        cols = np.nonzero(row)[0]
        want_cols = [TO.row_index(q, e, K) for q in range(pp + 1) for e in range(K)
                     if pp >= dd and q >= e and TO.attends(pp, dd, q, e)]
        assert cols.tolist() == want_cols
    del m
    torch.cuda.empty_cache()


def _partition_parity(n, K, r, bounds, seed):
    import torch
    B = _lib()
    u = np.random.default_rng(seed).random((n, K), dtype=np.float32)
    out = B.pe_train_partition(n, K, r, torch.from_numpy(u).cuda(), bounds)
    torch.cuda.synchronize()
    keep = TO.cod_keep(n, K, r, u)
    ref = TO.partition(keep, bounds)
    assert np.array_equal(out["keep"].cpu().numpy(), keep.astype(np.uint8))
    assert np.array_equal(out["seg"].cpu().numpy(), ref.seg)
    offs = out["offsets"].cpu().numpy()
    assert np.array_equal(offs, ref.offsets)
    total = int(offs[-1])
    assert np.array_equal(out["rows"][:total].cpu().numpy(), ref.rows)
    assert np.array_equal(out["owned"][:total].cpu().numpy(), ref.owned)


def test_partition_figure4_shape():
    _partition_parity(16, 4, 0.8, [0, 8, 16], 4)
    _partition_parity(16, 4, 1.0, [0, 8, 16], 4)   # every row kept: (8, 2) joins (7, 1)


@pytest.mark.parametrize("seed", range(5))
def test_partition_random_ragged_shapes(seed):
    rng = np.random.default_rng(500 + seed)
    n = int(rng.integers(2, 3000))
    K = int(rng.integers(1, 9))
    S = int(rng.integers(1, min(n, 12) + 1))
    cuts = sorted(rng.choice(np.arange(1, n), size=S - 1, replace=False).tolist()) if S > 1 else []
    _partition_parity(n, K, float(rng.uniform(0.2, 1.0)), [0] + cuts + [n], seed)


def test_partition_long_context_example():
    """[paper] 3.2: 8192 tokens, K = 8, r = 0.8, four equal segments."""
    _partition_parity(8192, 8, 0.8, [0, 2048, 4096, 6144, 8192], 11)


def test_partition_one_segment_and_one_depth():
    _partition_parity(1, 1, 0.5, [0, 1], 1)
    _partition_parity(1000, 1, 0.5, [0, 1, 999, 1000], 2)
    _partition_parity(64, 3, 0.0, [0, 64], 3)
