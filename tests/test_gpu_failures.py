"""Failure detection without a GPU fault: data-dependent violations made on
the host are reported through the device error word (the offending write
skipped, no trap), and the bounded waits every kernel relies on give up
and report PE_DEV_TIMEOUT instead of hanging.

The pages' KV-cache rule (the blog's engineering section: rejected slots
map to -1 and never get a KV write) is the model: a row whose page cannot
be resolved gets slot -1 the same way, and the step goes on.
"""

import numpy as np
import pytest

from synthetic import workloads as W
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

SMALL = W.small_shape("fail-bf16", d=512, n_layers=2, n_heads=8, n_kv_heads=2,
                      head_dim=64, ffn=1024, vocab=4096)
BAD_BLOCK, BAD_POSITION, BAD_TOKEN, TIMEOUT, BAD_ROW = 2, 3, 4, 5, 6


def _step(wl, edit):
    """Inputs and KV pools as usual, then `edit(inp)` breaks one input;
    runs the whole step and returns (code, GPU slots, pools before/after)."""
    inp = W.make_step_inputs(wl)
    w = W.make_weights(wl.shape, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    edit(inp)
    dr = G.make_drafter(wl.shape, w, max(wl.T_out, wl.B * wl.K), wl.B)
    st = G.DeviceStep(wl, inp, kc, vc)
    res = G.run_step(dr, st, want_logits=False)
    B = G.library()
    code = res["err"]
    assert B.pe_get_device_error(dr) == 0            # the read cleared it
    slots = B.to_host(res["ex"].slot)
    after_k = [B.to_host(k) for k in st.kc]
    dr.close()
    return code, slots, kc, after_k


def _only_live_slots_written(slots, before, after, page):
    """Pool bytes differ from the input pools only at slots >= 0 of this step."""
    ok = np.zeros(before[0].shape[0] * page, bool)
    ok[slots[slots >= 0]] = True
    for b, a in zip(before, after):
        b2 = b.transpose(0, 2, 1, 3).reshape(ok.size, -1)
        a2 = a.transpose(0, 2, 1, 3).reshape(ok.size, -1)
        changed = np.any(b2.view(np.uint16) != a2.view(np.uint16), axis=1)
        assert not np.any(changed & ~ok)


def test_block_id_out_of_range_is_reported_and_not_written():
    K = 7
    wl = W.custom("bad-block", 301, SMALL, K, [100], [K + 1], [K])
    first_pos = 100                       # the first drafter row's position
    page = first_pos // 16

    def edit(inp):
        inp.block_table[0, page] = inp.num_blocks + 5

    code, slots, before, after = _step(wl, edit)
    assert code == BAD_BLOCK
    # every row whose position falls in the broken page gets slot -1
    rows_in_page = [i for i in range(wl.T_out) if (first_pos + i) // 16 == page]
    assert rows_in_page and all(slots[i] == -1 for i in rows_in_page)
    assert np.count_nonzero(slots >= 0) == wl.T_out - len(rows_in_page)
    _only_live_slots_written(slots, before, after, 16)


def test_position_beyond_the_block_table_is_reported_and_not_written():
    K = 4
    wl = W.custom("bad-pos", 302, SMALL, K, [40, 60], [K + 1, K + 1], [K, 2])

    def edit(inp):
        stride = inp.block_table.shape[1]
        # request 0's last window row (its accepted row) far past its table
        inp.target_pos[K] = stride * 16 + 3

    code, slots, before, after = _step(wl, edit)
    assert code == BAD_POSITION
    # request 0: its accepted row and its MASK rows lie past the table
    bad_rows = [K] + [K + k for k in range(1, K)]
    assert all(slots[i] == -1 for i in bad_rows)
    _only_live_slots_written(slots, before, after, 16)


def test_token_id_out_of_range_is_reported():
    K = 5
    wl = W.custom("bad-token", 303, SMALL, K, [70], [K + 1], [3])

    def edit(inp):
        inp.sampled_ids[0] = SMALL.vocab + 11

    code, slots, before, after = _step(wl, edit)
    assert code == BAD_TOKEN
    _only_live_slots_written(slots, before, after, 16)


def test_window_longer_than_k_plus_one_is_reported():
    """The attention plans its query tiles for at most K + 1 window rows per
    request (reading R11); with 4 query heads per KV head a tile holds 32
    rows, so at K = 16 request 0's 19 window rows + 15 MASK rows overflow the
    one tile planned for 32 and are reported (not read past)."""
    K = 16
    wl = W.custom("bad-row", 304, SMALL, K, [50, 30], [K + 3, 1], [K + 2, 0])
    code, slots, before, after = _step(wl, lambda inp: None)
    assert code == BAD_ROW
    _only_live_slots_written(slots, before, after, 16)


def test_bounded_waits_give_up_and_the_context_stays_usable():
    """An mbarrier nobody arrives on and a flag nobody sets: both waits
    give up after the 2 s limit, PE_DEV_TIMEOUT is recorded, and a normal
    step on the same context afterwards is correct."""
    B = G.library()
    torch = G.torch_mod()
    wl = W.custom("after-timeout", 305, SMALL, 4, [90, 20], [5, 5], [4, 1])
    inp = W.make_step_inputs(wl)
    w = W.make_weights(SMALL, wl.config_id, gains=wl.gains)
    dr = G.make_drafter(SMALL, w, wl.T_out, wl.B)
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    B.pe_check_bounded_wait(dr, out)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [1, 1]
    assert B.pe_get_device_error(dr) == TIMEOUT
    assert B.pe_get_device_error(dr) == 0
    dr.close()
    G.full_parity(wl, 2e-2)
