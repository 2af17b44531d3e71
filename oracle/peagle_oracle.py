"""CPU oracle for the P-EAGLE parallel drafting step -- TEST INFRASTRUCTURE.

A plain, slow, fp64 statement of what the drafting step computes.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it.  It shares no code with the CUDA library: the only thing both
use is the seeded input module ``synthetic``.

Sources (web pages on P-EAGLE), cited by title and section:
  [paper]  "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training"
           (summary page): section 2 "P-EAGLE architecture", Fig. 2,
           Fig. 3 (position-invariant causal mask).
  [blog]   "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding
           in vLLM" (summary page): the input formula (Input_i cases),
           "prompt position handling" (shift by one), and the engineering
           section: fused batch-expansion kernel, hidden-state management,
           KV-cache slot mapping (-1 for rejected tokens).
  [abstract page] ScienceStack page for the paper: Theorem 2.1 (RoPE
           injectivity), figure captions.

Readings taken where the pages are silent (each one is listed with its
reason in the design notes of the repository):
  R1 shift: the drafter row at position P carries the token x_P and the
     target hidden state h_{P-1} (EAGLE convention); so a target row at
     position q yields a drafter row at position q+1.
  R2 layout: per request, the n target-window rows followed by K-1 MASK rows.
     Rows after the accepted prefix (j > a) are kept but rejected: slot -1,
     no query, no KV write.
  R3 ids of target-derived rows: shift left by one, the last row takes the
     sampled token s, then row a (the next-token row) takes s.
  R4 MASK rows continue the positions after the next-token row.
  R5 h_shared is 3d wide and replaces the target hidden row before fc.
  R6 "emb (+) projected hidden" is the EAGLE-3 first-layer form:
     layer 0 input = [RMSNorm_e(emb) ; RMSNorm_h(fc h)] (2d wide),
     residual = fc h.  Later layers are pre-norm LLaMA layers.  No biases.
  R7 RMSNorm eps = 1e-5; RoPE is rotate-half with inv_freq_i = theta^(-2i/dh).
  R8 draft token = argmax of the logits, lowest index on ties.

Hidden-state rows are copied bit for bit; all other arithmetic is fp64 on
the exact values of the (bf16 or fp32) inputs.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# value conversion (inputs are bf16 bit patterns or float32)
# ---------------------------------------------------------------------------


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 value of a bf16-bits (uint16) or float32 array."""
    if dtype == "bf16":
        u = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def linear(x: np.ndarray, w: np.ndarray, dtype: str,
           rows_per_chunk: int = 16384) -> np.ndarray:
    """y = x W^T for W stored row-major [out, in] (converted chunk by chunk)."""
    out = np.empty((x.shape[0], w.shape[0]), np.float64)
    for lo in range(0, w.shape[0], rows_per_chunk):
        hi = min(w.shape[0], lo + rows_per_chunk)
        out[:, lo:hi] = x @ to_f64(w[lo:hi], dtype).T
    return out


# ---------------------------------------------------------------------------
# a1: batch expansion metadata
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Expanded:
    ids: np.ndarray          # int32 [T']
    pos: np.ndarray          # int32 [T']
    slot: np.ndarray         # int32 [T'], -1 for rejected rows
    is_rejected: np.ndarray  # uint8 [T']
    is_masked: np.ndarray    # uint8 [T']
    new_idx: np.ndarray      # int32 [B*K]
    hidden_map: np.ndarray   # int32 [T]
    cu_out: np.ndarray       # int32 [B+1]
    seq_lens: np.ndarray     # int32 [B]
    request_of_row: np.ndarray  # int32 [T'] (oracle bookkeeping only)


def expand_batch(K: int, target_ids, target_pos, cu_in, num_accepted,
                 sampled_ids, block_table, page_size: int,
                 mask_token_id: int) -> Expanded:
    """Expand the verified target batch into the parallel-drafting batch.

    [blog] engineering section, fused-kernel bullet: copy the previous ids
    and positions into the new slots, insert each request's sampled token,
    fill the extra parallel-drafting slots with the MASK id, and emit the
    rejected-token mask, the MASK-token mask, the new-token indices and the
    hidden-state map; [blog] "KV cache" bullet: slot mapping recomputed from
    the new positions, rejected tokens get -1.  Readings R1-R4.
    """
    B = len(num_accepted)
    T = int(cu_in[B])
    T_out = T + B * (K - 1)
    ids = np.zeros(T_out, np.int64)
    pos = np.zeros(T_out, np.int64)
    slot = np.zeros(T_out, np.int64)
    rej = np.zeros(T_out, np.uint8)
    msk = np.zeros(T_out, np.uint8)
    req = np.zeros(T_out, np.int64)
    new_idx = np.zeros(B * K, np.int64)
    hmap = np.zeros(T, np.int64)
    cu_out = np.zeros(B + 1, np.int64)
    seq_lens = np.zeros(B, np.int64)

    for r in range(B):
        start_in, end_in = int(cu_in[r]), int(cu_in[r + 1])
        n = end_in - start_in
        a = int(num_accepted[r])
        if not (1 <= n and 0 <= a <= n - 1):
            raise ValueError("accepted count outside the verify window")
        s = int(sampled_ids[r])
        out = start_in + r * (K - 1)
        cu_out[r] = out
        rows_of_r = n + K - 1
        req[out:out + rows_of_r] = r
        # target-derived rows: row j carries h at target position q_j, so its
        # own position is q_j + 1 and its token is the one at q_j + 1.
        for j in range(n):
            if j + 1 < n:
                ids[out + j] = target_ids[start_in + j + 1]
            else:
                ids[out + j] = s
            pos[out + j] = int(target_pos[start_in + j]) + 1
            rej[out + j] = 1 if j > a else 0
            hmap[start_in + j] = out + j
        ids[out + a] = s  # the next-token (NTP) row takes the sampled token
        q_a = int(target_pos[start_in + a])
        for k in range(1, K):
            row = out + n - 1 + k
            ids[row] = mask_token_id
            pos[row] = q_a + 1 + k
            msk[row] = 1
        for j in range(rows_of_r):
            row = out + j
            if rej[row]:
                slot[row] = -1
            else:
                p = int(pos[row])
                blk = int(block_table[r][p // page_size])
                slot[row] = blk * page_size + p % page_size
        new_idx[r * K] = out + a
        for k in range(1, K):
            new_idx[r * K + k] = out + n - 1 + k
        seq_lens[r] = q_a + K + 1
    cu_out[B] = T_out

    i32 = lambda v: v.astype(np.int32)
    return Expanded(i32(ids), i32(pos), i32(slot), rej, msk, i32(new_idx),
                    i32(hmap), i32(cu_out), i32(seq_lens), i32(req))


# ---------------------------------------------------------------------------
# a2: hidden scatter + h_shared broadcast
# ---------------------------------------------------------------------------


def expand_hidden(target_hidden: np.ndarray, hidden_map: np.ndarray,
                  is_masked: np.ndarray, h_shared: np.ndarray) -> np.ndarray:
    """[blog] hidden-state management: first copy every target hidden row to
    its new row through the map, then, where the MASK-token mask is set,
    replace the row by the learned shared hidden state (a masked select).
    Rows are copied bit for bit (reading R5: the rows are 3d wide)."""
    T_out = is_masked.shape[0]
    out = np.zeros((T_out, target_hidden.shape[1]), target_hidden.dtype)
    out[hidden_map] = target_hidden
    out[is_masked.astype(bool)] = h_shared
    return out


# ---------------------------------------------------------------------------
# drafter building blocks (LLaMA 3 layers: [paper] section 2)
# ---------------------------------------------------------------------------


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding (reading R7).

    x: [R, H, dh]; dimension i < dh/2 is paired with i + dh/2 and rotated by
    the angle position * theta^(-2i/dh).
    """
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / dh)
    ang = positions.astype(np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def attention_one_row(q: np.ndarray, k_seq: np.ndarray, v_seq: np.ndarray,
                      P: int) -> np.ndarray:
    """Causal attention of one query row at position P.

    q: [Hq, dh]; k_seq, v_seq: [S, Hkv, dh] by position.  Query head h reads
    kv head h // (Hq / Hkv) over positions 0..P; scores scaled by 1/sqrt(dh).
    """
    Hq, dh = q.shape
    Hkv = k_seq.shape[1]
    group = Hq // Hkv
    out = np.empty((Hq, dh), np.float64)
    for h in range(Hq):
        g = h // group
        keys = k_seq[: P + 1, g, :]
        s = keys @ q[h] / np.sqrt(dh)
        s = s - s.max()
        p = np.exp(s)
        p /= p.sum()
        out[h] = p @ v_seq[: P + 1, g, :]
    return out


# ---------------------------------------------------------------------------
# a3..a8: the drafter body over an explicit list of rows
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class DrafterRows:
    """Rows fed to the drafter: each row is one (token, hidden, position)."""

    tokens: np.ndarray        # [R] int
    hidden3: np.ndarray       # [R, 3d] raw dtype (bf16 bits or float32)
    positions: np.ndarray     # [R] int
    request: np.ndarray       # [R] int (which request's cache the row uses)


@dataclasses.dataclass
class DrafterOut:
    residual: np.ndarray                 # [R, d] fp64 after the last layer
    kv_writes: List[Dict[str, np.ndarray]]  # per layer: slot, k, v
    layer_residuals: List[np.ndarray]
    layer_attn: List[np.ndarray]         # per layer: attention output [R, Hq, dh]


def gather_request_cache(cache_layer: np.ndarray, block_table_row,
                         seq_len: int, page_size: int,
                         dtype: str, scale: Optional[float] = None) -> np.ndarray:
    """Dense fp64 [S, Hkv, dh] copy of one request's paged cache.

    cache_layer layout [num_blocks, Hkv, page, dh]; position p lives in block
    block_table_row[p // page] at offset p % page.  With a scale the pool
    holds e4m3 codes and the value is code * scale (oracle/fp8_kv.py).
    """
    nblk = (seq_len + page_size - 1) // page_size
    blocks = [int(b) for b in block_table_row[:nblk]]
    if scale is None:
        pages = to_f64(cache_layer[blocks], dtype)     # [nblk, Hkv, page, dh]
    else:
        from . import fp8_kv
        pages = fp8_kv.dequantize(cache_layer[blocks], scale)
    dense = pages.transpose(0, 2, 1, 3).reshape(nblk * page_size,
                                                pages.shape[1], pages.shape[3])
    return dense[:seq_len].copy()


def drafter_forward_rows(shape, weights, rows: DrafterRows, block_table,
                         seq_lens: Dict[int, int], k_cache, v_cache,
                         kv_scales=None) -> DrafterOut:
    """Run the N drafter layers on explicit rows ([paper] section 2, Fig. 2).

    Every row writes its k, v at its own position before the layer's
    attention; each row then attends positions 0..P of its request.
    kv_scales: None (the cache holds the model dtype) or one (k_scale,
    v_scale) pair per layer for an fp8 e4m3 cache: the pools hold codes, a
    new row is written as the code of k / k_scale, and attention reads
    code * scale (oracle/fp8_kv.py, readings F1-F3).
    """
    dt = shape.dtype
    d, Hq, Hkv, dh = shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim
    eps, P = shape.rms_eps, shape.page_size
    R = rows.tokens.shape[0]
    W = weights

    e = to_f64(W["emb"][rows.tokens], dt)                       # [R, d]
    h = linear(to_f64(rows.hidden3, dt), W["fc"], dt)           # [R, d]
    residual = h
    kv_writes, layer_res, layer_attn = [], [], []
    requests = sorted(set(int(r) for r in rows.request))
    for l, lw in enumerate(W["layers"]):
        if l == 0:
            x = np.concatenate([rms_norm(e, to_f64(lw["norm_e"], dt), eps),
                                rms_norm(h, to_f64(lw["norm_h"], dt), eps)],
                               axis=1)
        else:
            x = rms_norm(residual, to_f64(lw["norm_in"], dt), eps)
        qkv = linear(x, lw["qkv"], dt)
        q = qkv[:, : Hq * dh].reshape(R, Hq, dh)
        k = qkv[:, Hq * dh: (Hq + Hkv) * dh].reshape(R, Hkv, dh)
        v = qkv[:, (Hq + Hkv) * dh:].reshape(R, Hkv, dh)
        q = rope(q, rows.positions, shape.rope_theta)
        k = rope(k, rows.positions, shape.rope_theta)

        attn = np.zeros((R, Hq, dh), np.float64)
        slots = np.zeros(R, np.int64)
        ks, vs = (None, None) if kv_scales is None else kv_scales[l]
        if kv_scales is not None:
            from . import fp8_kv
            k_codes, v_codes = fp8_kv.quantize(k, ks), fp8_kv.quantize(v, vs)
        for r in requests:
            sel = np.nonzero(rows.request == r)[0]
            S = int(seq_lens[r])
            kd = gather_request_cache(k_cache[l], block_table[r], S, P, dt, ks)
            vd = gather_request_cache(v_cache[l], block_table[r], S, P, dt, vs)
            for i in sel:                     # writes first ...
                p = int(rows.positions[i])
                if kv_scales is None:
                    kd[p] = k[i]
                    vd[p] = v[i]
                else:
                    kd[p] = fp8_kv.dequantize(k_codes[i], ks)
                    vd[p] = fp8_kv.dequantize(v_codes[i], vs)
                slots[i] = int(block_table[r][p // P]) * P + p % P
            for i in sel:                     # ... then attention
                attn[i] = attention_one_row(q[i], kd, vd, int(rows.positions[i]))
        kv_writes.append({"slot": slots, "k": k, "v": v} if kv_scales is None else
                         {"slot": slots, "k": k, "v": v, "k_codes": k_codes,
                          "v_codes": v_codes})
        layer_attn.append(attn)

        residual = residual + linear(attn.reshape(R, Hq * dh), lw["o"], dt)
        n = rms_norm(residual, to_f64(lw["norm_post"], dt), eps)
        act = silu(linear(n, lw["gate"], dt)) * linear(n, lw["up"], dt)
        residual = residual + linear(act, lw["down"], dt)
        layer_res.append(residual)
    return DrafterOut(residual, kv_writes, layer_res, layer_attn)


# ---------------------------------------------------------------------------
# a9: final norm + LM head + argmax
# ---------------------------------------------------------------------------


def final_norm(shape, weights, residual_rows: np.ndarray) -> np.ndarray:
    return rms_norm(residual_rows, to_f64(weights["norm_final"], shape.dtype),
                    shape.rms_eps)


def lm_head_argmax(shape, weights, y: np.ndarray):
    """logits = y W_lm^T; draft token = argmax, lowest index on ties (R8)."""
    logits = linear(y, weights["lm_head"], shape.dtype)
    return logits, np.argmax(logits, axis=1).astype(np.int32)


# ---------------------------------------------------------------------------
# the whole parallel drafting step
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class StepResult:
    expanded: Expanded
    hidden: np.ndarray            # [T', 3d] raw dtype (expanded hidden)
    requests: List[int]           # requests computed
    new_rows: np.ndarray          # expanded row indices of the outputs
    out_hidden: np.ndarray        # [len(requests)*K, d] fp64, final-normed
    logits: np.ndarray            # [len(requests)*K, V] fp64
    tokens: np.ndarray            # [len(requests)*K] int32
    drafter: DrafterOut
    row_index: np.ndarray         # expanded row of each drafter row


def draft_step(shape, weights, K: int, inp, k_cache, v_cache,
               requests: Optional[Sequence[int]] = None, kv_scales=None) -> StepResult:
    """One parallel drafting step: all K draft tokens from one pass.

    [blog] input formula: row 1 is emb(new) (+) h_context and rows 2..K are
    emb(mask) (+) h_shared; [paper] section 2: every row goes through the N
    layers at once, then the LM head.  Only non-rejected rows are computed
    (rejected rows produce nothing and write nothing).  ``requests`` selects
    a subset of the batch (requests are independent).  ``kv_scales`` selects
    the fp8 (e4m3) KV cache: one (k_scale, v_scale) per layer, the pools
    holding e4m3 codes (oracle/fp8_kv.py).
    """
    ex = expand_batch(K, inp.target_ids, inp.target_pos, inp.cu_in,
                      inp.num_accepted, inp.sampled_ids, inp.block_table,
                      shape.page_size, shape.mask_token_id)
    hid = expand_hidden(inp.target_hidden, ex.hidden_map, ex.is_masked,
                        weights["h_shared"])
    B = len(inp.num_accepted)
    reqs = list(range(B)) if requests is None else [int(r) for r in requests]
    rowsel = np.array([i for i in range(ex.ids.shape[0])
                       if ex.request_of_row[i] in set(reqs)
                       and not ex.is_rejected[i]], np.int64)
    rows = DrafterRows(ex.ids[rowsel].astype(np.int64), hid[rowsel],
                       ex.pos[rowsel].astype(np.int64),
                       ex.request_of_row[rowsel].astype(np.int64))
    seq = {r: int(ex.seq_lens[r]) for r in reqs}
    dout = drafter_forward_rows(shape, weights, rows, inp.block_table, seq,
                                k_cache, v_cache, kv_scales)
    new_rows = np.concatenate([ex.new_idx[r * K:(r + 1) * K] for r in reqs])
    where = {int(e): i for i, e in enumerate(rowsel)}
    take = np.array([where[int(e)] for e in new_rows], np.int64)
    y = final_norm(shape, weights, dout.residual[take])
    logits, tokens = lm_head_argmax(shape, weights, y)
    return StepResult(ex, hid, reqs, new_rows, y, logits, tokens, dout, rowsel)


def ar_eagle_step(shape, weights, inp, k_cache, v_cache):
    """One autoregressive EAGLE drafting step (one draft token per request).

    Built directly, without the expansion machinery: for each request keep
    the accepted prefix of the verify window, shift its tokens left by one
    and put the sampled token last ([blog] prompt-position handling: the row
    at position i gets the hidden state of i-1), run the drafter, and read the
    last row.  With K=1 the parallel step must agree with it.
    """
    toks, hids, poss, reqs, last = [], [], [], [], []
    B = len(inp.num_accepted)
    for r in range(B):
        lo = int(inp.cu_in[r])
        a = int(inp.num_accepted[r])
        window_ids = list(inp.target_ids[lo:lo + a + 1])
        shifted = window_ids[1:] + [int(inp.sampled_ids[r])]
        for j in range(a + 1):
            toks.append(int(shifted[j]))
            hids.append(inp.target_hidden[lo + j])
            poss.append(int(inp.target_pos[lo + j]) + 1)
            reqs.append(r)
        last.append(len(toks) - 1)
    rows = DrafterRows(np.array(toks), np.stack(hids), np.array(poss),
                       np.array(reqs))
    seq = {r: int(inp.target_pos[int(inp.cu_in[r]) + int(inp.num_accepted[r])]) + 2
           for r in range(B)}
    dout = drafter_forward_rows(shape, weights, rows, inp.block_table, seq,
                                k_cache, v_cache)
    y = final_norm(shape, weights, dout.residual[np.array(last)])
    logits, tokens = lm_head_argmax(shape, weights, y)
    return logits, tokens
