"""Brute-force restatement of the drafter for tiny inputs (tests only).

Written independently of ``oracle/``: rotary embedding through complex
multiplication, attention through an explicit dense mask matrix over whole
sequences, products through ``einsum`` with named indices.  It is used to pin
the oracle, never the CUDA path directly.
"""

import numpy as np
from scipy.special import expit, softmax


def f64(a, dtype):
    if dtype == "bf16":
        return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, np.float32).astype(np.float64)


def lin(x, w):
    # w is [out, in]
    return np.einsum("ri,oi->ro", x, w)


def rmsnorm(x, g, eps):
    ms = np.einsum("ri,ri->r", x, x) / x.shape[1]
    return x * g[None, :] / np.sqrt(ms + eps)[:, None]


def rope_complex(x, pos, theta):
    # x [R, H, dh]; pair i with i + dh/2 as the real/imaginary parts
    dh = x.shape[-1]
    half = dh // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = np.array([theta ** (-2.0 * i / dh) for i in range(half)])
    rot = np.exp(1j * np.outer(pos, freq))[:, None, :]
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


def dense_cache(cache, bt_row, S, page, dtype):
    out = np.zeros((S,) + (cache.shape[1], cache.shape[3]))
    for p in range(S):
        out[p] = f64(cache[bt_row[p // page], :, p % page, :], dtype)
    return out


def drafter(shape, W, tokens, hidden3, positions, request, block_table,
            seq_lens, k_cache, v_cache):
    """Returns the last-layer residual [R, d] for the given rows."""
    dt = shape.dtype
    d, Hq, Hkv, dh = shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim
    eps = shape.rms_eps
    R = len(tokens)
    emb = np.stack([f64(W["emb"][t], dt) for t in tokens])
    h = lin(f64(hidden3, dt), f64(W["fc"], dt))
    res = h.copy()
    reqs = sorted(set(int(r) for r in request))
    for l, lw in enumerate(W["layers"]):
        g = lambda k: f64(lw[k], dt)
        if l == 0:
            x = np.concatenate([rmsnorm(emb, g("norm_e"), eps),
                                rmsnorm(h, g("norm_h"), eps)], axis=1)
        else:
            x = rmsnorm(res, g("norm_in"), eps)
        qkv = lin(x, f64(lw["qkv"], dt))
        q = rope_complex(qkv[:, :Hq * dh].reshape(R, Hq, dh), positions, shape.rope_theta)
        k = rope_complex(qkv[:, Hq * dh:(Hq + Hkv) * dh].reshape(R, Hkv, dh), positions, shape.rope_theta)
        v = qkv[:, (Hq + Hkv) * dh:].reshape(R, Hkv, dh)
        attn = np.zeros((R, Hq, dh))
        for r in reqs:
            idx = [i for i in range(R) if request[i] == r]
            S = seq_lens[r]
            Kd = dense_cache(k_cache[l], block_table[r], S, shape.page_size, dt)
            Vd = dense_cache(v_cache[l], block_table[r], S, shape.page_size, dt)
            for i in idx:
                Kd[positions[i]] = k[i]
                Vd[positions[i]] = v[i]
            mask = np.array([[t <= positions[i] for t in range(S)] for i in idx])
            for hq in range(Hq):
                kv = hq * Hkv // Hq
                sc = np.einsum("id,td->it", q[idx, hq, :], Kd[:, kv, :]) / np.sqrt(dh)
                sc = np.where(mask, sc, -np.inf)
                p = softmax(sc, axis=1)
                attn[idx, hq, :] = np.einsum("it,td->id", p, Vd[:, kv, :])
        res = res + lin(attn.reshape(R, Hq * dh), f64(lw["o"], dt))
        n = rmsnorm(res, g("norm_post"), eps)
        gate = lin(n, f64(lw["gate"], dt))
        up = lin(n, f64(lw["up"], dt))
        res = res + lin(gate * expit(gate) * up, f64(lw["down"], dt))
    return res
