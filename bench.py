"""Benchmark of the P-EAGLE parallel drafting step on GB300.

One step = pe_expand_batch + pe_draft_forward + pe_lmhead_argmax over one
batch of seeded synthetic input (all K draft tokens of every request from one
drafter pass).  Default workload: the GPT-OSS-20B-shaped drafter (bf16,
d=2880, 4 layers, 64x64 q heads, 8 kv heads, FFN 7680, vocab 201088), one
request, K=7, context 4096 in a paged KV cache.

`value` is device-timed throughput (draft steps/s, whole job) of the step
replayed as a CUDA graph with inputs resident in HBM; `e2e` is the same
metric through the public calls with pinned host inputs copied in and draft
tokens copied out inside the timed region.  Each rank of a multi-GPU run
drafts its own batch (requests are independent: weak scaling, no
collective on the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload b1|b16|b64|qwen-k<K>|expand|tiny|ar-<workload>|lmhead-<rows>|train-mask[-<tokens>]|train-partition]
                  [--no-configs]
                  (b1, b16, b64 take a "-fp8" suffix: e4m3 KV pools)

The default run (b1) also times the other configurations in the same
process and reports them under "configs": the batch-64 step, the Qwen-shaped
K sweep 1..8 and the expansion microbenchmark, each with its step roofline
and (for the steps) the split into attention and the rest from phase events.
With --gpus N > 1 and no launcher, bench.py starts the N ranks itself (one
process per GPU, 127.0.0.1 rendezvous).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import workloads as W  # noqa: E402

L2_BYTES = 129 * 2 ** 20
METRIC = "P-EAGLE draft steps/s & drafted tok/s at K=7, 1 GB300; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# fp8 (e4m3) KV pools of the "-fp8" workloads: one scale for every layer's K
# and V (the N(0,1) context values stay well inside the e4m3 range)
FP8_KV_SCALE = 0.05


def workload(name: str):
    if name.endswith("-fp8"):
        return workload(name[: -len("-fp8")])
    if name == "tiny":
        return W.tiny_fp32()
    if name == "b1":
        return W.gpt_oss_b1()
    if name == "b64":
        return W.gpt_oss_b64()
    if name == "b16":
        return W.gpt_oss_b64(16)
    if name.startswith("qwen-k"):
        return W.qwen_b16(int(name[len("qwen-k"):]))
    if name == "expand":
        return W.expand_b256()
    raise SystemExit(f"unknown workload {name}")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# algorithmic work of one step (bytes that must move, flops that must run)
# ---------------------------------------------------------------------------

def step_work(wl, inp, kv_es=None):
    sh = wl.shape
    es = 2 if sh.dtype == "bf16" else 4
    kv_es = es if kv_es is None else kv_es
    d, F, V = sh.d, sh.ffn, sh.vocab
    qd = sh.n_heads * sh.head_dim
    rows = wl.T_out
    valid = int(sum(int(a) + wl.K for a in wl.accepted))
    seq = [int(inp.target_pos[int(inp.cu_in[r]) + int(wl.accepted[r])]) + wl.K + 1
           for r in range(wl.B)]
    # projections: (weight elements, rows that carry a result); flops count
    # the valid rows only (accepted window rows and the K draft rows)
    proj = [(d * sh.hidden3, valid)]
    for l in range(sh.n_layers):
        proj += [(sh.qkv_rows * (2 * d if l == 0 else d), valid), (d * qd, valid),
                 (2 * F * d, valid), (F * d, valid)]
    lm = (V * d, wl.B * wl.K)
    parts = [(n * es, 2.0 * m * n) for n, m in proj + [lm]]
    kv_bytes = sh.n_layers * 2 * sum(seq) * sh.n_kv_heads * sh.head_dim * kv_es
    attn_flops = 0.0
    for r in range(wl.B):
        a = int(wl.accepted[r])
        C = seq[r] - (a + wl.K)
        for j in range(a + wl.K):
            attn_flops += 4.0 * sh.n_heads * sh.head_dim * (C + j + 1) * sh.n_layers
    parts.append((kv_bytes, attn_flops))
    weight_bytes = sum(n for n, _ in proj + [lm]) * es
    act_bytes = rows * sh.hidden3 * es + wl.B * wl.K * 4
    gemm_flops = sum(f for _, f in parts[:-1])
    lm_bytes = V * d * es + wl.B * wl.K * d * es + wl.B * wl.K * 4
    return dict(weight_bytes=weight_bytes, kv_bytes=kv_bytes, act_bytes=act_bytes,
                bytes=weight_bytes + kv_bytes + act_bytes, gemm_flops=gemm_flops,
                attn_flops=attn_flops, flops=gemm_flops + attn_flops, parts=parts,
                lm_head_bytes=lm_bytes, lm_head_flops=2.0 * wl.B * wl.K * V * d,
                valid_rows=valid, rows=rows)


def kernel_source_hash() -> str:
    """Hash of the GEMM kernel's sources: a recorded DRAM-traffic figure is
    only reported while the kernel it was measured on is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "gemm_tc.cuh", "pe_common.cuh"):
        with open(os.path.join(ROOT, "speculative_drafting_expand_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload_name: str):
    """dram bytes read + written per launch from profiles/traffic.txt
    (lines: kernel workload source-hash bytes), or None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and parts[0] == kernel and parts[1] == workload_name and parts[2] == src:
            return float(parts[3])
    return None


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier + max over ranks)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def spawn_ranks(n: int) -> int:
    """Run this command as n ranks (one process per GPU, LOCAL_RANK = GPU
    index) with a 127.0.0.1 rendezvous, as a launcher would; rank 0's output
    is this process's output.  Returns the worst exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + sys.argv[1:],
                                      env=env))
    codes = [p.wait() for p in procs]
    return max(codes, key=abs)


def aggregate_rate(world: int, steps_per_rank: int, elapsed_s: float) -> float:
    """Whole-job rate: every rank ran the same number of steps on its own batch
    (weak scaling), timed by the slowest rank."""
    return world * steps_per_rank / elapsed_s


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("num_threads")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def time_oracle(wl, inp, w, kc, vc, budget_s: float, max_steps: int):
    import oracle as O
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        O.draft_step(wl.shape, w, wl.K, inp, kc, vc)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    wl = workload(args.workload)
    inp = W.make_step_inputs(wl)
    w = W.make_weights(wl.shape, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    budget = float(os.environ.get("PE_REF_BUDGET_S", "120"))
    import oracle as O
    for _ in range(min(args.warmup, 1)):
        O.draft_step(wl.shape, w, wl.K, inp, kc, vc)
    sps, n, dt = time_oracle(wl, inp, w, kc, vc, budget, args.steps)
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": sps, "unit": "steps/s",
        "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * dt / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "drafted_tok_per_s": sps * wl.B * wl.K,
        "config": config_of(wl, args),
        "cpu_baseline": {"value": sps, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} full oracle steps of the workload "
                                   f"(of {args.steps} requested; time budget {budget:.0f} s)"},
        "e2e": {"value": sps, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(wl, args):
    sh = wl.shape
    return {"workload": wl.name, "drafter": sh.name, "B": wl.B, "K": wl.K,
            "window": int(wl.window[0]), "contexts_mean": float(np.mean(wl.contexts)),
            "d": sh.d, "layers": sh.n_layers, "heads": f"{sh.n_heads}x{sh.head_dim}",
            "kv_heads": sh.n_kv_heads, "ffn": sh.ffn, "vocab": sh.vocab,
            "page_size": sh.page_size, "parallelism": f"replicas x{args.gpus}",
            "kv_cache": (f"fp8 e4m3, scale {FP8_KV_SCALE}" if args.workload.endswith("-fp8")
                         else sh.dtype),
            "l2": "weights stream from HBM every step (working set > 129 MB L2)",
            "graph": "step replayed as one CUDA graph"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def check_device(B, dr):
    code = B.pe_get_device_error(dr)
    if code != 0:
        raise SystemExit(f"device-side error code {code} recorded by the drafting kernels")


class DeviceInputs:
    """One step's inputs and the paged KV pools, resident in HBM."""

    def __init__(self, wl, inp, kc, vc, B, torch):
        dt = wl.shape.dtype
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


def run_lmhead(args, local):
    """The LM-head GEMM + argmax alone on the GPT-OSS LM-head shape (d 2880,
    vocab 201088) for M rows (--workload lmhead-<M>): the launch the bench
    reports as its dominant kernel, for profiling it in isolation."""
    import torch

    from speculative_drafting_expand_gb300 import binding as B

    torch.cuda.set_device(local)
    M = int(args.workload[len("lmhead-"):])
    full = W.gpt_oss_b1().shape
    sh = W.small_shape("lm-head", d=full.d, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64,
                       ffn=64, vocab=full.vocab)
    z = np.zeros(64, np.uint16)
    g = torch.Generator().manual_seed(7)
    lm = (torch.randn(sh.vocab, sh.d, generator=g) * 0.02).to(torch.bfloat16)
    w = {k: z for k in ("emb", "norm_final")}
    w["fc"] = np.zeros(sh.d * sh.hidden3, np.uint16)   # read at pe_create (fc of h_shared)
    w["lm_head"] = lm.view(torch.int16).numpy().view(np.uint16)
    w["h_shared"] = np.zeros(sh.hidden3, np.uint16)
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z,
                        norm_post=z)]
    dr = B.Drafter(sh, w, max(M, 16), 1)
    hid = torch.randn(M, sh.d, generator=g).to(torch.bfloat16).cuda()
    tok = torch.empty(M, dtype=torch.int32, device="cuda")
    for _ in range(args.warmup):
        B.pe_lmhead_argmax(dr, hid, tok)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        B.pe_lmhead_argmax(dr, hid, tok)
    e1.record()
    torch.cuda.synchronize()
    check_device(B, dr)
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    print(json.dumps({"mode": "lm_head", "rows": M, "d": sh.d, "vocab": sh.vocab,
                      "us_per_launch": us, "weight_gbs": sh.vocab * sh.d * 2 / us / 1e3,
                      "tflops": 2.0 * M * sh.vocab * sh.d / us / 1e6}), flush=True)
    dr.close()
    return 0


def run_train(args, local):
    """Training-side index work (paper summary section 3) on the section 3.2
    example: 8192 tokens, K = 8.  train-mask: the amortized additive bf16
    mask over the 65,536 rows (8.59 GB written; HBM-write bound).
    train-partition: COD sampling (r = 0.8) and the partition into four
    equal segments of one sample."""
    import torch

    from speculative_drafting_expand_gb300 import binding as B

    torch.cuda.set_device(local)
    n, K = 8192, 8
    if args.workload.startswith("train-mask-"):          # a smaller mask (profiling)
        n = int(args.workload[len("train-mask-"):])
    pk, src = peaks()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.workload.startswith("train-mask"):
        N = n * K
        out = torch.empty((N, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup):
            B.pe_train_build_mask(out, n, K, B.PE_MASK_ADDITIVE_BF16)
        torch.cuda.synchronize()
        clk = ClockSampler(local)
        clk.start()
        e0.record()
        for _ in range(args.steps):
            B.pe_train_build_mask(out, n, K, B.PE_MASK_ADDITIVE_BF16)
        e1.record()
        torch.cuda.synchronize()
        clk.stop()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        nbytes = N * N * 2
        gbs = nbytes / us / 1e3
        peak = pk["hbm_gbs"]
        print(json.dumps({
            "mode": "train_mask", "metric": "amortized mask build (GB/s written)",
            "value": gbs, "unit": "GB/s", "us_per_build": us, "bytes": nbytes,
            "config": {"workload": f"mask {n} tokens x K={K} ({N} rows), additive bf16"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_source": src},
            "steps": args.steps, "warmup": args.warmup, "clocks": clk.summary()}), flush=True)
        return 0
    if args.workload != "train-partition":
        raise SystemExit(f"unknown workload {args.workload}")
    r, bounds = 0.8, [0, 2048, 4096, 6144, 8192]
    u = torch.rand((n, K), generator=torch.Generator().manual_seed(3)).cuda()
    for _ in range(args.warmup):
        o = B.pe_train_partition(n, K, r, u, bounds)
    torch.cuda.synchronize()
    kept = int(o["keep"].sum())
    # outputs preallocated once: time the calls alone
    lib = B.lib()
    S = len(bounds) - 1
    import ctypes
    hb = (ctypes.c_int32 * (S + 1))(*bounds)
    cap = int(sum(bounds[:-1])) + n * K
    st = B.stream_ptr()
    args_c = [B.ptr(o[k]) for k in ("keep", "seg", "counts", "offsets", "rows", "owned")]
    e0.record()
    for _ in range(args.steps):
        rc = lib.pe_train_partition(n, K, ctypes.c_float(r), B.ptr(u), S, hb, *args_c, cap, st)
        if rc != 0:
            raise SystemExit(f"pe_train_partition failed: {rc}")
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    print(json.dumps({
        "mode": "train_partition", "metric": "COD sampling + sequence partition latency",
        "value": us, "unit": "us/sample", "higher_is_better": False, "rows": n * K,
        "kept_rows": kept, "segments": S, "rows_listed": int(o["offsets"][-1]),
        "config": {"workload": "8192 tokens, K=8, r=0.8, 4 equal segments"},
        "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def run_ar(args, world, rank, local):
    """Autoregressive drafting of the same K tokens on the same kernels: K
    sequential passes of the K = 1 step (the pages' baseline, whose cost
    grows with K).  Pass 0 takes the verify window and drafts the first token;
    pass i takes one row per request at the next position, whose token is
    the previous pass's draft (copied on the device), and drafts the next.
    A reported step is all K passes (K draft tokens per request)."""
    import torch

    from speculative_drafting_expand_gb300 import binding as B

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    wl = workload(args.workload[len("ar-"):])
    sh, K = wl.shape, wl.K
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    dr = B.Drafter(sh, w, max(wl.T, wl.B), wl.B)
    st = DeviceInputs(wl, inp, kc, vc, B, torch)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    tdt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
    Bn = wl.B
    # pass 0: the window, K = 1
    passes = [dict(ids=st.target_ids, pos=st.target_pos, cu=st.cu_in, acc=st.num_accepted,
                   samp=st.sampled_ids, hid=st.target_hidden, T=wl.T)]
    # position of the sampled token's row in pass 0, per request
    p0 = np.array([int(inp.target_pos[int(inp.cu_in[r]) + int(wl.accepted[r])]) + 1
                   for r in range(Bn)], np.int64)
    last_rows = [int(inp.cu_in[r]) + int(wl.accepted[r]) for r in range(Bn)]
    hid1 = np.ascontiguousarray(inp.target_hidden[last_rows])
    for i in range(1, K):
        passes.append(dict(ids=i32(np.zeros(Bn)), pos=i32(p0 + i - 1), cu=i32(np.arange(Bn + 1)),
                           acc=i32(np.zeros(Bn)), samp=torch.zeros(Bn, dtype=torch.int32, device="cuda"),
                           hid=B.to_device(hid1, sh.dtype), T=Bn))
    exs = [B.Expanded(q["T"], q["T"], Bn, 1, sh.hidden3, sh.dtype) for q in passes]
    outs = [torch.empty(Bn, sh.d, dtype=tdt, device="cuda") for _ in passes]
    toks = [torch.empty(Bn, dtype=torch.int32, device="cuda") for _ in passes]

    def step():
        for i, q in enumerate(passes):
            if i > 0:
                q["samp"].copy_(toks[i - 1])
            B.pe_expand_batch(dr, 1, q["ids"], q["pos"], q["cu"], q["acc"], q["samp"],
                              st.block_table, inp.num_blocks, q["hid"], exs[i])
            B.pe_draft_forward(dr, exs[i], st.block_table, st.kc, st.vc, inp.num_blocks, outs[i])
            B.pe_lmhead_argmax(dr, outs[i], toks[i])

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    check_device(B, dr)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    n0 = B.pe_get_launch_count(dr)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step()
    launches_per_step = B.pe_get_launch_count(dr) - n0
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(world, e0.elapsed_time(e1))
    clocks.stop()
    check_device(B, dr)
    if rank == 0:
        ms = elapsed_ms / args.steps
        value = aggregate_rate(world, args.steps, elapsed_ms / 1e3)
        cfg = config_of(wl, args)
        cfg["workload"] = wl.name + "-autoregressive"
        cfg["drafting"] = f"autoregressive: {K} sequential passes of the K=1 step per draft step"
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": sh.dtype, "data": "synthetic (seeded random-init weights and inputs)",
            "config": cfg, "drafted_tok_per_s": value * Bn * K, "mode": "autoregressive",
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks.summary()}), flush=True)
    dr.close()
    return 0


def step_floor(work, hbm, tflops_sus):
    """Sum over the projections and the attention of the slower of bytes /
    measured HBM and flops / sustained bf16 peak (seconds)."""
    return sum(max(b / (hbm * 1e9), f / (tflops_sus * 1e12)) for b, f in work["parts"])


def step_roofline_of(work, step_s, hbm, tflops_sus):
    floor = step_floor(work, hbm, tflops_sus)
    return {"bytes": work["bytes"], "flops": work["flops"], "floor_us": floor * 1e6,
            "frac": floor / step_s, "peak_source": "measured HBM copy and sustained bf16",
            "hbm_frac": work["bytes"] / step_s / (hbm * 1e9),
            "tensor_frac": work["flops"] / step_s / (tflops_sus * 1e12),
            "tensor_peak": tflops_sus, "hbm_peak": hbm,
            "frac_vs_nominal_7900_gbs": work["bytes"] / step_s / 7.9e12,
            "gemm_flops": work["gemm_flops"], "attn_flops": work["attn_flops"]}


class StepRig:
    """One workload's step on the device: drafter, resident inputs, the
    step captured as a CUDA graph."""

    def __init__(self, wl, weights, torch, B, kc=None, vc=None, kv_seed=0, inp=None):
        self.wl, self.torch, self.B = wl, torch, B
        sh = wl.shape
        self.inp = inp if inp is not None else W.make_step_inputs(wl)
        self.dr = B.Drafter(sh, weights, max(wl.T_out, wl.B * wl.K), wl.B)
        if kc is None:
            kc, vc = W.device_kv_pools(sh, self.inp.num_blocks, kv_seed)
        self.st = DeviceInputs(wl, self.inp, kc, vc, B, torch)
        self.ex = B.Expanded(wl.T_out, wl.T, wl.B, wl.K, sh.hidden3, sh.dtype)
        tdt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
        self.out_hidden = torch.empty(wl.B * wl.K, sh.d, dtype=tdt, device="cuda")
        self.tokens = torch.empty(wl.B * wl.K, dtype=torch.int32, device="cuda")
        self.graph = None

    def step(self):
        B, wl, st, inp = self.B, self.wl, self.st, self.inp
        B.pe_expand_batch(self.dr, wl.K, st.target_ids, st.target_pos, st.cu_in,
                          st.num_accepted, st.sampled_ids, st.block_table, inp.num_blocks,
                          st.target_hidden, self.ex)
        B.pe_draft_forward(self.dr, self.ex, st.block_table, st.kc, st.vc, inp.num_blocks,
                           self.out_hidden)
        B.pe_lmhead_argmax(self.dr, self.out_hidden, self.tokens)

    def capture(self):
        """Eager warm-up, then the step as one CUDA graph; launches per step."""
        torch, B = self.torch, self.B
        for _ in range(2):
            self.step()
        torch.cuda.synchronize()
        check_device(B, self.dr)
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        n0 = B.pe_get_launch_count(self.dr)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                self.step()
        torch.cuda.synchronize()
        self.graph = g
        return B.pe_get_launch_count(self.dr) - n0

    def time_ms(self, n, warmup=3):
        torch = self.torch
        for _ in range(warmup):
            self.graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            self.graph.replay()
        e1.record()
        torch.cuda.synchronize()
        check_device(self.B, self.dr)
        return e0.elapsed_time(e1) / n

    def phase_split(self, n):
        """Attention vs the rest of pe_draft_forward, from events recorded
        between its kernels in a separately captured graph (the events break
        the overlap of neighbouring kernels, so both parts read a little
        slow).  Mean over n replays, microseconds."""
        torch, B, L = self.torch, self.B, self.wl.shape.n_layers
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * L)]
        B.pe_set_phase_events(self.dr, ev)
        try:
            self.step()
            torch.cuda.synchronize()
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    self.step()
            torch.cuda.synchronize()
            attn = total = 0.0
            for _ in range(n):
                g.replay()
                torch.cuda.synchronize()
                attn += sum(ev[1 + 2 * l].elapsed_time(ev[2 + 2 * l]) for l in range(L))
                total += ev[0].elapsed_time(ev[1 + 2 * L])
        finally:
            B.pe_set_phase_events(self.dr, None)
        check_device(B, self.dr)
        return {"attention_us": 1e3 * attn / n, "forward_us": 1e3 * total / n,
                "rest_of_forward_us": 1e3 * (total - attn) / n}

    def close(self):
        self.dr.close()


def measure_config(rig, n, hbm, tflops_sus, label):
    """A configuration's line under "configs": throughput, its step roofline
    and the attention / projection split."""
    wl = rig.wl
    launches = rig.capture()
    ms = rig.time_ms(n)
    work = step_work(wl, rig.inp)
    ph = rig.phase_split(max(5, n // 10))
    attn_s, rest_s = ph["attention_us"] * 1e-6, ph["rest_of_forward_us"] * 1e-6
    lm_flops = work["lm_head_flops"]
    proj_flops = work["gemm_flops"] - lm_flops
    proj_bytes = work["weight_bytes"] - work["lm_head_bytes"]
    ph.update({
        "attention_hbm_frac": work["kv_bytes"] / attn_s / (hbm * 1e9) if attn_s > 0 else None,
        "projections_tensor_frac": proj_flops / rest_s / (tflops_sus * 1e12) if rest_s > 0 else None,
        "projections_hbm_frac": proj_bytes / rest_s / (hbm * 1e9) if rest_s > 0 else None,
        "note": "rest_of_forward = fc, row kernels and the layer projections (the LM head "
                "is outside pe_draft_forward); events between kernels cost their overlap"})
    return {"workload": wl.name, "label": label, "B": wl.B, "K": wl.K,
            "steps_per_s": 1e3 / ms, "ms_per_step": ms, "steps": n,
            "drafted_tok_per_s": 1e3 / ms * wl.B * wl.K, "launches_per_step": launches,
            "step_roofline": step_roofline_of(work, ms * 1e-3, hbm, tflops_sus),
            "phase_split": ph,
            "inputs": "seeded synthetic; KV pools and (Qwen) weights drawn on the device"}


def expand_only(wl, torch, B, hbm, n):
    """The expansion kernel alone (steps a1 + a2), L2 flushed before each
    launch, on a drafter whose only live weight is h_shared."""
    sh = wl.shape
    z = np.zeros(64, np.uint16)
    w = {k: z for k in ("emb", "norm_final", "lm_head")}
    w["fc"] = np.zeros(sh.d * sh.hidden3, np.uint16)   # read at pe_create (fc of h_shared)
    w["h_shared"] = W.normal(wl.config_id, "h_shared", (sh.hidden3,), 0.02, sh.dtype)
    w["layers"] = [dict(qkv=z, o=z, gate=z, up=z, down=z, norm_e=z, norm_h=z, norm_in=z,
                        norm_post=z) for _ in range(sh.n_layers)]
    dr = B.Drafter(sh, w, wl.T_out, wl.B)
    inp = W.make_step_inputs(wl)
    st = DeviceInputs(wl, inp, [], [], B, torch)
    ex = B.Expanded(wl.T_out, wl.T, wl.B, wl.K, sh.hidden3, sh.dtype)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    evs = []
    for i in range(n + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        B.pe_expand_batch(dr, wl.K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                          st.sampled_ids, st.block_table, inp.num_blocks, st.target_hidden, ex)
        b.record(stream)
        if i >= 3:
            evs.append((a, b))
    torch.cuda.synchronize()
    check_device(B, dr)
    dr.close()
    del flush
    s_ = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    es = 2 if sh.dtype == "bf16" else 4
    Bn, Tn, To = wl.B, wl.T, wl.T_out
    # hidden rows read once (h_shared once) and written once; metadata in and out
    nbytes = (Tn + 1) * sh.hidden3 * es + To * sh.hidden3 * es + \
        Tn * 8 + Bn * 12 + To * 4 + To * 14 + Bn * wl.K * 4 + Tn * 4 + (2 * Bn + 1) * 4
    return {"bound": "hbm", "workload": wl.name, "launch_us": s_ * 1e6,
            "bytes_per_launch": nbytes, "achieved": nbytes / s_ / 1e9, "peak": hbm,
            "unit": "GB/s", "frac": nbytes / s_ / 1e9 / hbm, "launches": n,
            "note": "expansion kernel alone, L2 flushed before each launch"}


def other_configs(args, torch, B, b1_weights, hbm, tflops_sus):
    """The batch-64 step, the Qwen-shaped K sweep and the expansion
    microbenchmark, timed in the same run as the headline."""
    out = {}
    wl = W.gpt_oss_b64()
    rig = StepRig(wl, b1_weights, torch, B, kv_seed=64)
    out["gpt-oss-b64-k7"] = measure_config(rig, 200, hbm, tflops_sus,
                                           "GPT-OSS-20B-shaped, batch 64, K 7, lognormal contexts")
    rig.close()
    del rig
    torch.cuda.empty_cache()
    qw = W.device_weights(W.QWEN3_CODER_30B, seed=4)
    sweep = {}
    for K in range(1, 9):
        rig = StepRig(W.qwen_b16(K), qw, torch, B, kv_seed=100 + K)
        sweep[f"k{K}"] = measure_config(rig, 200, hbm, tflops_sus,
                                        f"Qwen3-Coder-30B-shaped, batch 16, K {K}")
        rig.close()
        del rig
    out["qwen-b16-k-sweep"] = sweep
    del qw
    torch.cuda.empty_cache()
    out["expand-b256-k7"] = expand_only(W.expand_b256(), torch, B, hbm, 100)
    return out


def run_ours(args, world, rank, local):
    import torch

    from speculative_drafting_expand_gb300 import binding as B

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    wl = workload(args.workload)
    sh = wl.shape
    inp = W.make_step_inputs(wl)
    w = W.make_weights(sh, wl.config_id, gains=wl.gains)
    kc, vc = W.make_kv_cache(wl, inp)
    dr = B.Drafter(sh, w, max(wl.T_out, wl.B * wl.K), wl.B)
    st = DeviceInputs(wl, inp, kc, vc, B, torch)
    kv_fp8 = args.workload.endswith("-fp8")
    if kv_fp8:
        # e4m3 codes of the same draws (torch's float8 conversion: input
        # preparation only; the step's own KV writes are the library's)
        to8 = lambda t: (t.float() / FP8_KV_SCALE).to(torch.float8_e4m3fn).view(torch.uint8)
        st.kc = [to8(k) for k in st.kc]
        st.vc = [to8(v) for v in st.vc]
        B.pe_set_kv_cache_fp8(dr, [FP8_KV_SCALE] * sh.n_layers, [FP8_KV_SCALE] * sh.n_layers)
    ex = B.Expanded(wl.T_out, wl.T, wl.B, wl.K, sh.hidden3, sh.dtype)
    tdt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
    out_hidden = torch.empty(wl.B * wl.K, sh.d, dtype=tdt, device="cuda")
    tokens = torch.empty(wl.B * wl.K, dtype=torch.int32, device="cuda")

    def step():
        B.pe_expand_batch(dr, wl.K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                          st.sampled_ids, st.block_table, inp.num_blocks, st.target_hidden, ex)
        B.pe_draft_forward(dr, ex, st.block_table, st.kc, st.vc, inp.num_blocks, out_hidden)
        B.pe_lmhead_argmax(dr, out_hidden, tokens)

    # eager warm-up, then capture the step as one CUDA graph
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    check_device(B, dr)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    n0 = B.pe_get_launch_count(dr)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step()
    launches_per_step = B.pe_get_launch_count(dr) - n0
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()

    # ---- device-timed region: K graph replays ------------------------------
    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    t_pre = time.time()
    while time.time() - t_pre < 0.4:          # load the GPU while the sampler starts
        g.replay()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(world, e0.elapsed_time(e1))
    clocks.stop()
    ms_per_step = elapsed_ms / args.steps
    value = aggregate_rate(world, args.steps, elapsed_ms / 1e3)
    check_device(B, dr)

    # ---- dominant kernel: the LM-head GEMM + argmax, timed on its stream ----
    work = step_work(wl, inp, 1 if kv_fp8 else None)
    stream = torch.cuda.current_stream()
    n_lm = max(20, min(args.steps, 200))
    lm_ms = []
    for _ in range(n_lm):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        B.pe_lmhead_argmax(dr, out_hidden, tokens)
        b.record(stream)
        lm_ms.append((a, b))
    torch.cuda.synchronize()
    lm_avg_s = statistics.mean(a.elapsed_time(b) for a, b in lm_ms) / 1e3
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    tflops = float(pk["bf16_tflops"])                      # burst: timed alone
    tflops_sus = float(pk.get("bf16_tflops_sustained", tflops))  # inside the step
    traffic = measured_traffic("lm_head", wl.name)
    # the LM head's bound: its flops per byte against the ridge point
    lm_intensity = work["lm_head_flops"] / work["lm_head_bytes"]
    if lm_intensity > tflops * 1e12 / (hbm * 1e9):
        lm_roof = {"bound": "tensor", "achieved": work["lm_head_flops"] / lm_avg_s / 1e12,
                   "peak": tflops, "unit": "TFLOP/s", "peak_source": f"{pk_kind} bf16_tflops"}
    else:
        lm_roof = {"bound": "hbm", "achieved": work["lm_head_bytes"] / lm_avg_s / 1e9,
                   "peak": hbm, "unit": "GB/s", "peak_source": f"{pk_kind} hbm_gbs"}
    lm_roof["frac"] = lm_roof["achieved"] / lm_roof["peak"]

    # ---- the expansion kernel alone (steps a1 + a2), L2 flushed before each --
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ex_ev = []
    for _ in range(n_lm):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        B.pe_expand_batch(dr, wl.K, st.target_ids, st.target_pos, st.cu_in, st.num_accepted,
                          st.sampled_ids, st.block_table, inp.num_blocks, st.target_hidden, ex)
        b.record(stream)
        ex_ev.append((a, b))
    torch.cuda.synchronize()
    del flush
    ex_s = statistics.mean(a.elapsed_time(b) for a, b in ex_ev) / 1e3
    es = 2 if sh.dtype == "bf16" else 4
    Bn, Tn, To = wl.B, wl.T, wl.T_out
    # hidden rows read once (h_shared once) and written once; metadata in and out
    ex_bytes = (Tn + 1) * sh.hidden3 * es + To * sh.hidden3 * es + \
        Tn * 8 + Bn * 12 + To * 4 + To * 14 + Bn * wl.K * 4 + Tn * 4 + (2 * Bn + 1) * 4
    expand_roof = {"bound": "hbm", "launch_us": ex_s * 1e6, "bytes_per_launch": ex_bytes,
                   "achieved": ex_bytes / ex_s / 1e9, "peak": hbm, "unit": "GB/s",
                   "frac": ex_bytes / ex_s / 1e9 / hbm,
                   "note": "expansion kernel alone, L2 flushed before each launch"}

    # ---- end to end through the public calls with host buffers -------------
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_ids, h_pos, h_cu = pin(inp.target_ids), pin(inp.target_pos), pin(inp.cu_in)
    h_acc, h_samp, h_bt = pin(inp.num_accepted), pin(inp.sampled_ids), pin(inp.block_table)
    h_hid = B.to_device(inp.target_hidden, sh.dtype, device="cpu").pin_memory()
    h_tok = torch.empty(wl.B * wl.K, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_ids, h_pos, h_cu, h_acc, h_samp, h_bt, h_hid))
    d2h = h_tok.numel() * h_tok.element_size()

    def e2e_step():
        st.target_ids.copy_(h_ids, non_blocking=True)
        st.target_pos.copy_(h_pos, non_blocking=True)
        st.cu_in.copy_(h_cu, non_blocking=True)
        st.num_accepted.copy_(h_acc, non_blocking=True)
        st.sampled_ids.copy_(h_samp, non_blocking=True)
        st.block_table.copy_(h_bt, non_blocking=True)
        st.target_hidden.copy_(h_hid, non_blocking=True)
        step()
        h_tok.copy_(tokens, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(10, min(args.steps, 500))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(world, time.perf_counter() - t0)
    e2e_value = aggregate_rate(world, n_e2e, e2e_s)
    check_device(B, dr)

    # ---- CPU oracle baseline (rank 0, one GPU only) -------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        budget = float(os.environ.get("PE_CPU_BUDGET_S", "15"))
        sps, n, dt = time_oracle(wl, inp, w, kc, vc, budget, 1000)
        cpu = {"value": sps, "unit": "steps/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{n} full oracle steps of the same workload in {dt:.1f} s"}

    configs = None
    if rank == 0 and world == 1 and not args.no_configs and args.workload == "b1":
        dr.close()
        del st
        torch.cuda.empty_cache()
        configs = other_configs(args, torch, B, w, hbm, tflops_sus)

    if rank == 0:
        # each projection and the attention at the slower of its bytes and
        # its flops (sustained tensor peak: they run inside a long step)
        step_s = ms_per_step / 1e3
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": sh.dtype, "data": "synthetic (seeded random-init weights and inputs)",
            "config": config_of(wl, args),
            "drafted_tok_per_s": value * wl.B * wl.K,
            "step_roofline": step_roofline_of(work, step_s, hbm, tflops_sus),
            "roofline": dict(lm_roof, kernel="LM-head GEMM + fused argmax",
                             scope="the dominant kernel alone; the whole step's fraction of "
                                   "its HBM floor is step_roofline.frac",
                             traffic=traffic, bytes_per_launch=work["lm_head_bytes"],
                             flops_per_launch=work["lm_head_flops"],
                             launch_us=lm_avg_s * 1e6),
            "expand_roofline": expand_roof,
            "e2e": {"value": e2e_value, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "launches_per_step": launches_per_step,
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
        }
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    dr.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="b1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline workload only (not the batch-64 step, "
                         "the Qwen K sweep and the expansion microbenchmark)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_ranks(args.gpus)
    world, rank, local = dist_setup()
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.workload.startswith("ar-"):
        return run_ar(args, world, rank, local)
    if args.workload.startswith("lmhead-"):
        return run_lmhead(args, local)
    if args.workload.startswith("train-"):
        return run_train(args, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
