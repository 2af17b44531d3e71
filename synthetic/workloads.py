"""Seeded synthetic inputs for the P-EAGLE parallel drafting step.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path
(``speculative_drafting_expand_gb300``).  It holds shapes and random numbers
only -- none of the method's arithmetic.  Every tensor is drawn from
``numpy.random.default_rng(SeedSequence([config_id, tensor_id, ...]))`` so
that both sides see the same bits.

Floating-point draws are float32 and are rounded to bfloat16 with
round-to-nearest-even when a workload is bf16; bf16 tensors are kept on the
host as ``uint16`` bit patterns.

Workload shapes follow the P-EAGLE pages:
  * drafter = N LLaMA-style layers over [token, MASK, ..., MASK] slots
    (P-EAGLE paper, section 2 "Architecture"; vLLM blog, "P-EAGLE drafter").
  * target hidden = concat of 3 target layers, width 3d (paper, Figure 2).
  * context lengths of the batch-64 workload are lognormal with median 3,891
    and P90 10,800, capped at 20,000 (paper, Figure 1; blog, "long sequence
    requirement").
  * K=7 is the depth where P-EAGLE peaks (blog, results item 2).
"""

from __future__ import annotations

import dataclasses
import math
import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np

PAGE_SIZE = 16
BF16_NAN_BITS = np.uint16(0x7FC0)

_CHUNK = 1 << 22  # elements per independently seeded chunk
_THREADS = max(1, min(16, os.cpu_count() or 1))


# --------------------------------------------------------------------------
# shapes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DrafterShape:
    """Shape of the LLaMA-style drafter (P-EAGLE paper section 2, Fig. 2)."""

    name: str
    d: int              # drafter hidden width
    n_layers: int       # N decoder layers
    n_heads: int        # query heads
    n_kv_heads: int     # key/value heads (GQA)
    head_dim: int
    ffn: int            # SwiGLU inner width
    vocab: int
    rope_theta: float
    dtype: str          # "bf16" or "f32"
    rms_eps: float = 1e-5
    page_size: int = PAGE_SIZE

    @property
    def hidden3(self) -> int:
        """Width of the concatenated target hidden states (3 target layers)."""
        return 3 * self.d

    @property
    def mask_token_id(self) -> int:
        return self.vocab - 1

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


TINY = DrafterShape("tiny", d=256, n_layers=2, n_heads=4, n_kv_heads=4,
                    head_dim=64, ffn=688, vocab=1024, rope_theta=1e4,
                    dtype="f32")
GPT_OSS_20B = DrafterShape("gpt-oss-20b-drafter", d=2880, n_layers=4,
                           n_heads=64, n_kv_heads=8, head_dim=64, ffn=7680,
                           vocab=201088, rope_theta=150000.0, dtype="bf16")
QWEN3_CODER_30B = DrafterShape("qwen3-coder-30b-drafter", d=2048, n_layers=4,
                               n_heads=32, n_kv_heads=4, head_dim=128,
                               ffn=6144, vocab=151936, rope_theta=1e6,
                               dtype="bf16")


def small_shape(name: str = "small-bf16", **kw) -> DrafterShape:
    """A reduced bf16 shape for parity tests that still spans several tiles."""
    base = dict(d=512, n_layers=2, n_heads=8, n_kv_heads=2, head_dim=64,
                ffn=1024, vocab=4096, rope_theta=1e4, dtype="bf16")
    base.update(kw)
    return DrafterShape(name, **base)


@dataclasses.dataclass
class StepWorkload:
    """One drafting step's batch: B requests, depth K, target windows."""

    name: str
    config_id: int
    shape: DrafterShape
    K: int
    contexts: np.ndarray     # [B] cached drafter positions C_r
    window: np.ndarray       # [B] target verify-window rows n_r
    accepted: np.ndarray     # [B] accepted drafts a_r in [0, n_r - 1]
    block_order: str = "random"   # "random" or "identity"
    gains: str = "one"            # "one" or "random" norm gains

    @property
    def B(self) -> int:
        return int(self.contexts.shape[0])

    @property
    def T(self) -> int:
        return int(self.window.sum())

    @property
    def T_out(self) -> int:
        return self.T + self.B * (self.K - 1)


# --------------------------------------------------------------------------
# seeded draws
# --------------------------------------------------------------------------

def _tensor_id(name: str) -> int:
    return zlib.crc32(name.encode()) & 0x7FFFFFFF


def _seed(config_id: int, name: str, *extra: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([config_id, _tensor_id(name), *extra])


def rng_for(config_id: int, name: str, *extra: int) -> np.random.Generator:
    return np.random.default_rng(_seed(config_id, name, *extra))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest-even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal(config_id: int, name: str, shape, std: float, dtype: str,
           *extra: int) -> np.ndarray:
    """N(0, std^2) draws, float32 or bf16 bits, generated in seeded chunks."""
    n = int(np.prod(shape))
    out_dtype = np.uint16 if dtype == "bf16" else np.float32
    out = np.empty(n, dtype=out_dtype)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.default_rng(_seed(config_id, name, *extra, c))
        buf = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            buf *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(buf) if dtype == "bf16" else buf

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def uniform(config_id: int, name: str, shape, lo: float, hi: float,
            dtype: str, *extra: int) -> np.ndarray:
    g = rng_for(config_id, name, *extra)
    x = g.uniform(lo, hi, size=shape).astype(np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------

def make_weights(shape: DrafterShape, config_id: int,
                 gains: str = "one", std: float = 0.02) -> Dict[str, object]:
    """Random-init drafter weights.  Matrices are row-major [out, in].

    Keys: emb [V,d], fc [d,3d], h_shared [3d], norm_final [d], lm_head [V,d],
    layers: list of dicts with qkv [(Hq+2Hkv)dh, d_in], o [d, Hq dh],
    gate [F,d], up [F,d], down [d,F], norm_post [d], and either
    norm_e/norm_h (layer 0) or norm_in (layers >= 1).  Layer 0's qkv takes the
    2d-wide concatenation of the normed embedding and normed fc output.
    """
    dt = shape.dtype
    d, F, V = shape.d, shape.ffn, shape.vocab
    qd = shape.n_heads * shape.head_dim

    def gain(name, layer):
        if gains == "one":
            ones = np.ones(d, np.float32)
            return f32_to_bf16_bits(ones) if dt == "bf16" else ones
        return uniform(config_id, name, (d,), 0.5, 1.5, dt, layer)

    w: Dict[str, object] = {
        "emb": normal(config_id, "emb", (V, d), std, dt),
        "fc": normal(config_id, "fc", (d, shape.hidden3), std, dt),
        "h_shared": normal(config_id, "h_shared", (shape.hidden3,), std, dt),
        "norm_final": gain("norm_final", 0),
        "lm_head": normal(config_id, "lm_head", (V, d), std, dt),
    }
    layers: List[Dict[str, np.ndarray]] = []
    for l in range(shape.n_layers):
        d_in = 2 * d if l == 0 else d
        lw = {
            "qkv": normal(config_id, "qkv", (shape.qkv_rows, d_in), std, dt, l),
            "o": normal(config_id, "o", (d, qd), std, dt, l),
            "gate": normal(config_id, "gate", (F, d), std, dt, l),
            "up": normal(config_id, "up", (F, d), std, dt, l),
            "down": normal(config_id, "down", (d, F), std, dt, l),
            "norm_post": gain("norm_post", l),
        }
        if l == 0:
            lw["norm_e"] = gain("norm_e", l)
            lw["norm_h"] = gain("norm_h", l)
        else:
            lw["norm_in"] = gain("norm_in", l)
        layers.append(lw)
    w["layers"] = layers
    return w


# --------------------------------------------------------------------------
# one step's batch
# --------------------------------------------------------------------------

@dataclasses.dataclass
class StepInputs:
    target_ids: np.ndarray     # int32 [T]
    target_pos: np.ndarray     # int32 [T]
    cu_in: np.ndarray          # int32 [B+1]
    num_accepted: np.ndarray   # int32 [B]
    sampled_ids: np.ndarray    # int32 [B]
    block_table: np.ndarray    # int32 [B, bt_stride]; unused entries -1
    num_blocks: int
    target_hidden: np.ndarray  # [T, 3d] bf16 bits or float32


def blocks_needed(wl: StepWorkload) -> np.ndarray:
    """Pages each request may touch: context + window + K - 1 MASK rows."""
    worst = wl.contexts + wl.window + wl.K - 1
    return (worst + wl.shape.page_size - 1) // wl.shape.page_size


def make_step_inputs(wl: StepWorkload) -> StepInputs:
    cid, sh = wl.config_id, wl.shape
    B = wl.B
    n = wl.window.astype(np.int64)
    cu_in = np.zeros(B + 1, np.int64)
    cu_in[1:] = np.cumsum(n)
    T = int(cu_in[-1])
    ids = rng_for(cid, "target_ids").integers(0, sh.vocab - 1, size=T)
    sampled = rng_for(cid, "sampled_ids").integers(0, sh.vocab - 1, size=B)
    pos = np.empty(T, np.int64)
    for r in range(B):
        # the verify window starts at the last cached position C_r - 1
        pos[cu_in[r]:cu_in[r + 1]] = wl.contexts[r] - 1 + np.arange(n[r])
    nblk = blocks_needed(wl)
    num_blocks = int(nblk.sum())
    stride = int(nblk.max())
    if wl.block_order == "identity":
        phys = np.arange(num_blocks)
    else:
        phys = rng_for(cid, "block_perm").permutation(num_blocks)
    bt = np.full((B, stride), -1, np.int64)
    off = 0
    for r in range(B):
        bt[r, :nblk[r]] = phys[off:off + nblk[r]]
        off += nblk[r]
    hid = normal(cid, "target_hidden", (T, sh.hidden3), 1.0, sh.dtype)
    return StepInputs(ids.astype(np.int32), pos.astype(np.int32),
                      cu_in.astype(np.int32), wl.accepted.astype(np.int32),
                      sampled.astype(np.int32), bt.astype(np.int32),
                      num_blocks, hid)


def make_kv_cache(wl: StepWorkload, inp: StepInputs):
    """Paged KV cache per layer, layout [num_blocks, Hkv, page, head_dim].

    Positions < C_r of request r hold N(0,1) draws; every other slot of the
    pool holds a NaN sentinel so that any out-of-range read shows up.
    Returns (k_cache, v_cache) lists of host arrays.
    """
    sh = wl.shape
    P = sh.page_size
    shp = (inp.num_blocks, sh.n_kv_heads, P, sh.head_dim)
    valid = np.zeros((inp.num_blocks, P), bool)
    for r in range(wl.B):
        C = int(wl.contexts[r])
        full, rem = divmod(C, P)
        valid[inp.block_table[r, :full]] = True
        if rem:
            valid[inp.block_table[r, full], :rem] = True
    sentinel = BF16_NAN_BITS if sh.dtype == "bf16" else np.float32(np.nan)
    ks, vs = [], []
    for l in range(sh.n_layers):
        for name, lst in (("k_cache", ks), ("v_cache", vs)):
            vals = normal(wl.config_id, name, shp, 1.0, sh.dtype, l)
            vals.transpose(0, 2, 1, 3)[~valid] = sentinel
            lst.append(vals)
    return ks, vs


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------

def tiny_fp32() -> StepWorkload:
    """Tiny fp32 drafter, batch 1, context 64, K=4, no rejected rows."""
    K = 4
    return StepWorkload("tiny-f32-b1-k4", 1, TINY, K,
                        contexts=np.array([64]), window=np.array([K + 1]),
                        accepted=np.array([K]), block_order="identity")


def gpt_oss_b1() -> StepWorkload:
    """GPT-OSS-20B-shaped drafter, bf16, one request, K=7, context 4096."""
    K = 7
    return StepWorkload("gpt-oss-20b-drafter-b1-k7-ctx4096", 2, GPT_OSS_20B, K,
                        contexts=np.array([4096]), window=np.array([K + 1]),
                        accepted=np.array([K]))


def lognormal_contexts(config_id: int, B: int, median=3891.0, p90=10800.0,
                       cap=20000) -> np.ndarray:
    sigma = math.log(p90 / median) / 1.2815515655446004
    g = rng_for(config_id, "contexts")
    c = np.exp(g.normal(math.log(median), sigma, size=B))
    return np.clip(np.rint(c), 1, cap).astype(np.int64)


def gpt_oss_b64(B: int = 64) -> StepWorkload:
    """GPT-OSS-20B-shaped drafter at batch 64, K=7, lognormal contexts."""
    K, cid = 7, 3
    acc = rng_for(cid, "accepted").integers(0, K + 1, size=B)
    return StepWorkload(f"gpt-oss-20b-drafter-b{B}-k7-lognormal", cid,
                        GPT_OSS_20B, K, contexts=lognormal_contexts(cid, B),
                        window=np.full(B, K + 1), accepted=acc)


def qwen_b16(K: int, B: int = 16) -> StepWorkload:
    """Qwen3-Coder-30B-shaped drafter, bf16, batch 16, contexts U[1K,16K]."""
    cid = 4
    ctx = rng_for(cid, "contexts").integers(1024, 16384 + 1, size=B)
    acc = rng_for(cid, "accepted", K).integers(0, K + 1, size=B)
    return StepWorkload(f"qwen3-coder-30b-drafter-b{B}-k{K}", cid,
                        QWEN3_CODER_30B, K, contexts=ctx,
                        window=np.full(B, K + 1), accepted=acc)


def expand_b256() -> StepWorkload:
    """Batch-expansion microbench: 256 requests, K=7, hidden width 8640."""
    K, cid, B = 7, 5, 256
    ctx = rng_for(cid, "contexts").integers(512, 20000 + 1, size=B)
    acc = rng_for(cid, "accepted").integers(0, K + 1, size=B)
    return StepWorkload("expand-b256-k7-h8640", cid, GPT_OSS_20B, K,
                        contexts=ctx, window=np.full(B, K + 1), accepted=acc)


def custom(name: str, config_id: int, shape: DrafterShape, K: int,
           contexts, window, accepted, block_order="random",
           gains="random") -> StepWorkload:
    return StepWorkload(name, config_id, shape, K, np.asarray(contexts),
                        np.asarray(window), np.asarray(accepted),
                        block_order, gains)


# --------------------------------------------------------------------------
# device-side draws for timing-only runs (no oracle comparison): the same
# distributions, seeded, generated on the GPU so that large pools cost no
# host time.  torch is imported lazily (the CPU tests never call these).
# --------------------------------------------------------------------------

def device_weights(shape: DrafterShape, seed: int, std: float = 0.02, device="cuda"):
    """Random-init drafter weights as device tensors (bf16), unit norm gains;
    the same keys and layouts as make_weights."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    d, F, V = shape.d, shape.ffn, shape.vocab
    qd = shape.n_heads * shape.head_dim

    def mat(*s):
        return (torch.randn(*s, generator=g, device=device) * std).to(dt)

    ones = lambda: torch.ones(d, dtype=dt, device=device)
    w = {"emb": mat(V, d), "fc": mat(d, shape.hidden3), "h_shared": mat(shape.hidden3),
         "norm_final": ones(), "lm_head": mat(V, d)}
    layers = []
    for l in range(shape.n_layers):
        lw = {"qkv": mat(shape.qkv_rows, 2 * d if l == 0 else d), "o": mat(d, qd),
              "gate": mat(F, d), "up": mat(F, d), "down": mat(d, F), "norm_post": ones()}
        if l == 0:
            lw["norm_e"], lw["norm_h"] = ones(), ones()
        else:
            lw["norm_in"] = ones()
        layers.append(lw)
    w["layers"] = layers
    return w


def device_kv_pools(shape: DrafterShape, num_blocks: int, seed: int, device="cuda"):
    """Paged KV pools [num_blocks, Hkv, page, head_dim] per layer, N(0,1)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    shp = (num_blocks, shape.n_kv_heads, shape.page_size, shape.head_dim)
    ks = [torch.randn(*shp, generator=g, device=device).to(dt) for _ in range(shape.n_layers)]
    vs = [torch.randn(*shp, generator=g, device=device).to(dt) for _ in range(shape.n_layers)]
    return ks, vs
