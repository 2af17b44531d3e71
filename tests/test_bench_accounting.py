"""The roofline accounting of bench.py against closed forms (CPU only): the
GPT-OSS-20B-shaped drafter's parameter counts (layers 386.3 M, fc 24.9 M, LM
head 579.1 M: 1.981 GB of bf16 weights streamed once a step), the batch-1
KV bytes, the batch-64 flop split (projections ~1.07 TFLOP on the valid
rows, attention ~0.23 TFLOP), and the fp8 pools' halved KV bytes."""

import numpy as np
import pytest

import bench
from synthetic import workloads as W


def _work(name, kv_es=None):
    wl = bench.workload(name)
    inp = W.make_step_inputs(wl)
    return wl, inp, bench.step_work(wl, inp, kv_es)


def test_weight_bytes_of_the_gpt_oss_drafter():
    wl, _, w = _work("b1")
    d, L, dh = 2880, 4, 64
    qkv = (64 + 2 * 8) * dh
    layers = qkv * 2 * d + (L - 1) * qkv * d + L * (d * 64 * dh + 3 * 7680 * d)
    fc, lm = d * 3 * d, 201088 * d
    assert round(layers / 1e5) / 10 == 386.3
    assert round(fc / 1e5) / 10 == 24.9 and round(lm / 1e5) / 10 == 579.1
    assert w["weight_bytes"] == 2 * (layers + fc + lm)
    assert abs(w["weight_bytes"] / 1e9 - 1.981) < 0.001


def test_batch1_kv_bytes_and_flops():
    wl, inp, w = _work("b1")
    seq = int(inp.target_pos[int(wl.accepted[0])]) + wl.K + 1     # positions read
    assert w["kv_bytes"] == 4 * 2 * seq * 8 * 64 * 2
    assert 33.5e6 < w["kv_bytes"] < 33.8e6
    # every one of the 14 rows is valid (all accepted): 2 flops a weight and row
    assert w["valid_rows"] == 14 == wl.T_out
    assert w["gemm_flops"] == pytest.approx(2 * 14 * (w["weight_bytes"] / 2 - 201088 * 2880)
                                            + 2 * 7 * 201088 * 2880)


def test_batch64_flop_split_and_fp8_kv():
    wl, inp, w = _work("b64")
    assert w["valid_rows"] == int(sum(int(a) + wl.K for a in wl.accepted)) == 666
    assert abs(w["gemm_flops"] / 1e12 - 1.07) < 0.01
    assert abs(w["attn_flops"] / 1e12 - 0.23) < 0.01
    assert w["lm_head_flops"] == 2.0 * 448 * 201088 * 2880
    _, _, w8 = _work("b64-fp8", 1)
    assert w8["kv_bytes"] * 2 == w["kv_bytes"]
    assert w8["weight_bytes"] == w["weight_bytes"]


def test_fp8_workloads_share_their_base_workload():
    a, b = bench.workload("b16"), bench.workload("b16-fp8")
    assert a.name == b.name and a.B == b.B and np.array_equal(a.accepted, b.accepted)
