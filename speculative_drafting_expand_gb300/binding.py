"""ctypes binding of libpeagle.so (include/peagle.h): argument marshalling only.

Every step of the drafting path runs in the library's CUDA kernels; PyTorch
is used here for device memory and streams.  Importing this module does not
need a GPU, but calling into the library does; if the library has not been
built the import fails loudly (there is no fallback path).
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpeagle.so")

PE_OK = 0
PE_ERR_INVALID_ARGUMENT = 1
PE_ERR_UNSUPPORTED = 2
PE_ERR_CUDA = 3
PE_ERR_OUT_OF_MEMORY = 4
PE_ERR_DEVICE = 5
PE_DTYPE_BF16 = 0
PE_DTYPE_F32 = 1

PE_MASK_BOOL_U8 = 0
PE_MASK_ADDITIVE_BF16 = 1

# include/peagle.h and include/peagle_train.h (pe_status_string last: it is
# the one that does not return a pe_status)
EXPORTED = ("pe_create", "pe_destroy", "pe_expand_batch", "pe_draft_forward",
            "pe_lmhead_argmax", "pe_get_device_error", "pe_set_trace", "pe_set_phase_events",
            "pe_set_small_batch_stream", "pe_set_stream_prefetch", "pe_set_stream_timeline",
            "pe_set_fusions", "pe_set_split_reduce", "pe_set_tuning", "pe_set_gemm_timeline",
            "pe_linear",
            "pe_get_launch_count", "pe_check_bounded_wait", "pe_linear_static",
            "pe_linear_static_error",
            "pe_set_kv_cache_fp8",
            "pe_train_build_mask",
            "pe_train_mask_view", "pe_train_partition", "pe_status_string")

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class pe_model_desc(ctypes.Structure):
    _fields_ = [("d", _i32), ("n_layers", _i32), ("n_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("ffn", _i32), ("vocab", _i32), ("hidden3", _i32),
                ("page_size", _i32), ("mask_token_id", _i32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("dtype", _i32)]


class pe_layer_weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("qkv", "o", "gate", "up", "down", "norm_e", "norm_h",
                                   "norm_in", "norm_post")]


class pe_weights(ctypes.Structure):
    _fields_ = [("emb", _vp), ("fc", _vp), ("h_shared", _vp), ("norm_final", _vp),
                ("lm_head", _vp), ("layers", ctypes.POINTER(pe_layer_weights))]


class pe_expanded(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("ids", "pos", "slot", "is_rejected", "is_masked",
                                   "new_idx", "hidden_map", "cu_out", "seq_lens", "hidden")] + \
               [("B", _i32), ("K", _i32), ("T", _i32), ("T_out", _i32),
                ("target_hidden", _vp)]


class PeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "speculative_drafting_expand_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.pe_create.argtypes = [P(pe_model_desc), P(pe_weights), _i32, _i32, P(_vp)]
    lib.pe_destroy.argtypes = [_vp]
    lib.pe_expand_batch.argtypes = [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                    _i32, _vp, P(pe_expanded), _vp]
    lib.pe_draft_forward.argtypes = [_vp, P(pe_expanded), _i32, _i32, _vp, _i32, P(_vp), P(_vp),
                                     _i32, _vp, _vp]
    lib.pe_lmhead_argmax.argtypes = [_vp, _vp, _i32, _vp, _vp, _vp]
    lib.pe_get_device_error.argtypes = [_vp, P(_i32), _vp]
    lib.pe_set_trace.argtypes = [_vp, _vp, _vp]
    lib.pe_linear.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp]
    lib.pe_get_launch_count.argtypes = [_vp, P(ctypes.c_int64)]
    lib.pe_linear_static.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp]
    lib.pe_check_bounded_wait.argtypes = [_vp, _vp, _vp]
    lib.pe_set_phase_events.argtypes = [_vp, P(_vp), _i32]
    lib.pe_set_small_batch_stream.argtypes = [_vp, _i32]
    lib.pe_set_stream_timeline.argtypes = [_vp, _vp]
    lib.pe_set_fusions.argtypes = [_vp, _i32]
    lib.pe_set_split_reduce.argtypes = [_vp, _i32]
    lib.pe_set_tuning.argtypes = [_vp, _i32, _i32]
    lib.pe_set_gemm_timeline.argtypes = [_vp, _vp, _i32]
    lib.pe_set_stream_prefetch.argtypes = [_vp, _i32, _i32]
    lib.pe_linear_static_error.argtypes = [P(_i32), _vp]
    lib.pe_set_kv_cache_fp8.argtypes = [_vp, P(ctypes.c_float), P(ctypes.c_float)]
    lib.pe_train_build_mask.argtypes = [_i32, _i32, _i32, _vp, ctypes.c_int64, _vp]
    lib.pe_train_mask_view.argtypes = [_vp, ctypes.c_int64, _i32, _i32, _i32, P(_vp),
                                       P(ctypes.c_int64), P(ctypes.c_int64)]
    lib.pe_train_partition.argtypes = [_i32, _i32, ctypes.c_float, _vp, _i32, P(_i32), _vp, _vp,
                                       _vp, _vp, _vp, _vp, ctypes.c_int64, _vp]
    lib.pe_status_string.argtypes = [_i32]
    lib.pe_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = _i32
    return lib


_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def status_string(s: int) -> str:
    return lib().pe_status_string(s).decode()


def _check(fn: str, s: int):
    if s != PE_OK:
        raise PeError(fn, s)


# ---------------------------------------------------------------------------
# tensors
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def stream_ptr(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def to_device(a: np.ndarray, dtype: str, device="cuda"):
    """Host array (bf16 bits as uint16, or float32 / int32 / uint8) -> tensor
    (a tensor is moved as it is)."""
    torch = _torch()
    if isinstance(a, torch.Tensor):
        return a.to(device)
    if dtype == "bf16" and a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def to_host(t) -> np.ndarray:
    """Tensor -> host array (bf16 as uint16 bits)."""
    torch = _torch()
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def model_desc(shape) -> pe_model_desc:
    return pe_model_desc(shape.d, shape.n_layers, shape.n_heads, shape.n_kv_heads,
                         shape.head_dim, shape.ffn, shape.vocab, shape.hidden3,
                         shape.page_size, shape.mask_token_id, shape.rope_theta,
                         shape.rms_eps, PE_DTYPE_BF16 if shape.dtype == "bf16" else PE_DTYPE_F32)


class Drafter:
    """Owns the device copies of the weights and a pe_handle."""

    def __init__(self, shape, host_weights: Dict, max_tokens: int, max_reqs: int,
                 device="cuda"):
        self.shape = shape
        self.device = device
        dt = shape.dtype
        W = host_weights
        self.w = {k: to_device(W[k], dt, device) for k in
                  ("emb", "fc", "h_shared", "norm_final", "lm_head")}
        self.layers = [{k: to_device(v, dt, device) for k, v in lw.items()}
                       for lw in W["layers"]]
        arr = (pe_layer_weights * shape.n_layers)()
        for l, lw in enumerate(self.layers):
            arr[l] = pe_layer_weights(*(ptr(lw.get(f[0])) for f in pe_layer_weights._fields_))
        self._layer_arr = arr
        self._weights = pe_weights(ptr(self.w["emb"]), ptr(self.w["fc"]),
                                   ptr(self.w["h_shared"]), ptr(self.w["norm_final"]),
                                   ptr(self.w["lm_head"]), arr)
        self._desc = model_desc(shape)
        h = _vp()
        _check("pe_create", lib().pe_create(ctypes.byref(self._desc), ctypes.byref(self._weights),
                                            max_tokens, max_reqs, ctypes.byref(h)))
        self.handle = h
        self.max_tokens = max_tokens

    def close(self):
        if getattr(self, "handle", None):
            lib().pe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------------------
# the entry points, same names as the C ABI
# ---------------------------------------------------------------------------

class Expanded:
    """Caller-owned device buffers of one expanded batch (pe_expanded)."""

    def __init__(self, T_out: int, T: int, B: int, K: int, hidden3: int, dtype: str,
                 device="cuda"):
        torch = _torch()
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.empty(T_out, **i32)
        self.pos = torch.empty(T_out, **i32)
        self.slot = torch.empty(T_out, **i32)
        self.is_rejected = torch.empty(T_out, dtype=torch.uint8, device=device)
        self.is_masked = torch.empty(T_out, dtype=torch.uint8, device=device)
        self.new_idx = torch.empty(B * K, **i32)
        self.hidden_map = torch.empty(T, **i32)
        self.cu_out = torch.empty(B + 1, **i32)
        self.seq_lens = torch.empty(B, **i32)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.hidden = torch.empty(T_out, hidden3, dtype=tdt, device=device)
        self.struct = pe_expanded(*(ptr(getattr(self, f)) for f in
                                    ("ids", "pos", "slot", "is_rejected", "is_masked",
                                     "new_idx", "hidden_map", "cu_out", "seq_lens", "hidden")),
                                  0, 0, 0, 0, None)


def pe_expand_batch(dr: Drafter, K: int, target_ids, target_pos, cu_in, num_accepted,
                    sampled_ids, block_table, num_blocks: int, target_hidden,
                    out: Expanded, stream=None):
    B = num_accepted.shape[0]
    T = target_ids.shape[0]
    _check("pe_expand_batch", lib().pe_expand_batch(
        dr.handle, B, K, T, ptr(target_ids), ptr(target_pos), ptr(cu_in), ptr(num_accepted),
        ptr(sampled_ids), ptr(block_table), block_table.shape[1], num_blocks,
        ptr(target_hidden), ctypes.byref(out.struct), stream_ptr(stream)))
    return out


def pe_draft_forward(dr: Drafter, ex: Expanded, block_table, k_cache: Sequence,
                     v_cache: Sequence, num_blocks: int, out_hidden, stream=None):
    L = len(k_cache)
    kc = (_vp * L)(*[ptr(t) for t in k_cache])
    vc = (_vp * L)(*[ptr(t) for t in v_cache])
    _check("pe_draft_forward", lib().pe_draft_forward(
        dr.handle, ctypes.byref(ex.struct), ex.struct.B, ex.struct.K, ptr(block_table),
        block_table.shape[1], kc, vc, num_blocks, ptr(out_hidden), stream_ptr(stream)))
    return out_hidden


def pe_lmhead_argmax(dr: Drafter, hidden, out_tokens, out_logits=None, stream=None):
    _check("pe_lmhead_argmax", lib().pe_lmhead_argmax(
        dr.handle, ptr(hidden), hidden.shape[0], ptr(out_tokens), ptr(out_logits),
        stream_ptr(stream)))
    return out_tokens


def pe_get_device_error(dr: Drafter, stream=None) -> int:
    code = _i32(0)
    _check("pe_get_device_error", lib().pe_get_device_error(dr.handle, ctypes.byref(code),
                                                            stream_ptr(stream)))
    return code.value


def pe_check_bounded_wait(dr: Drafter, out, stream=None) -> None:
    """Launch the bounded-wait self-check (out: device int32[2])."""
    _check("pe_check_bounded_wait", lib().pe_check_bounded_wait(dr.handle, ptr(out),
                                                                stream_ptr(stream)))


def pe_set_small_batch_stream(dr: Drafter, enable: bool) -> None:
    _check("pe_set_small_batch_stream", lib().pe_set_small_batch_stream(dr.handle, int(enable)))


PE_FUSE_ROPE_KV = 1
PE_FUSE_NORM = 2
PE_FUSE_ALL = 3


def pe_set_gemm_timeline(dr: Drafter, stamps=None, launches: int = 0) -> None:
    """stamps: int64 device tensor of launches * 512 * 16 entries, or None."""
    _check("pe_set_gemm_timeline",
           lib().pe_set_gemm_timeline(dr.handle, ptr(stamps), int(launches) if stamps is not None else 0))


def pe_set_fusions(dr: Drafter, mask: int) -> None:
    _check("pe_set_fusions", lib().pe_set_fusions(dr.handle, int(mask)))


PE_REDUCE_PULL = 0
PE_REDUCE_PUSH = 1


def pe_set_split_reduce(dr: Drafter, mode: int) -> None:
    _check("pe_set_split_reduce", lib().pe_set_split_reduce(dr.handle, int(mode)))


PE_TUNE_GEMM_PRE_STAGES = 1
PE_TUNE_ATTN_L2_AHEAD = 2
PE_TUNE_GEMM_MAX_SPLIT = 3
PE_TUNE_ATTN_MIN_CHUNKS = 4
PE_TUNE_ATTN_MAX_CHUNKS = 5
PE_TUNE_GEMM_TILE_ORDER = 6


def pe_set_tuning(dr: Drafter, key: int, value: int) -> None:
    _check("pe_set_tuning", lib().pe_set_tuning(dr.handle, int(key), int(value)))


def pe_set_stream_prefetch(dr: Drafter, tiles: int, boundary_tiles: int = -1) -> None:
    _check("pe_set_stream_prefetch",
           lib().pe_set_stream_prefetch(dr.handle, int(tiles), int(boundary_tiles)))


def pe_set_stream_timeline(dr: Drafter, stamps=None) -> None:
    """stamps: int64 device tensor of sm_count * 64 entries, or None."""
    _check("pe_set_stream_timeline", lib().pe_set_stream_timeline(dr.handle, ptr(stamps)))


def pe_set_phase_events(dr: Drafter, events=None) -> None:
    """events: torch.cuda.Event objects (2 + 2 n_layers, timing enabled), or
    None to turn phase timing off."""
    events = list(events or [])
    for e in events:
        if e.cuda_event == 0:      # torch creates the event on first record
            e.record()
    arr = (_vp * max(1, len(events)))(*[e.cuda_event for e in events])
    dr._phase_events = events      # the library keeps the handles
    _check("pe_set_phase_events", lib().pe_set_phase_events(dr.handle, arr, len(events)))


def pe_set_trace(dr: Drafter, residual_trace=None, attn_trace=None) -> None:
    _check("pe_set_trace", lib().pe_set_trace(dr.handle, ptr(residual_trace), ptr(attn_trace)))


def pe_set_kv_cache_fp8(dr: Drafter, k_scales=None, v_scales=None) -> None:
    """Switch the drafter to e4m3 KV pools with per-layer scales (None, None:
    back to pools of the model dtype)."""
    if k_scales is None and v_scales is None:
        _check("pe_set_kv_cache_fp8", lib().pe_set_kv_cache_fp8(dr.handle, None, None))
        return
    ks = (ctypes.c_float * len(k_scales))(*[float(x) for x in k_scales])
    vs = (ctypes.c_float * len(v_scales))(*[float(x) for x in v_scales])
    _check("pe_set_kv_cache_fp8", lib().pe_set_kv_cache_fp8(dr.handle, ks, vs))


def pe_get_launch_count(dr: Drafter) -> int:
    n = ctypes.c_int64(0)
    _check("pe_get_launch_count", lib().pe_get_launch_count(dr.handle, ctypes.byref(n)))
    return n.value


def pe_linear(dr: Drafter, x, w, y, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check("pe_linear", lib().pe_linear(dr.handle, ptr(x), ptr(w), ptr(y), M, N, K,
                                        stream_ptr(stream)))
    return y


def pe_linear_static(x, w, y, stream=None):
    """y = x w^T (bf16 in, fp32 out) through the entry point that allocates
    nothing: its scratch is a static device array inside the library."""
    M, K = x.shape
    N = w.shape[0]
    _check("pe_linear_static", lib().pe_linear_static(ptr(x), ptr(w), ptr(y), M, N, K,
                                                      stream_ptr(stream)))
    return y


def pe_linear_static_error(stream=None) -> int:
    """Read and clear the device error word of pe_linear_static's static
    array (0: nothing recorded since the last read)."""
    code = _i32(0)
    _check("pe_linear_static_error", lib().pe_linear_static_error(ctypes.byref(code),
                                                                  stream_ptr(stream)))
    return code.value


# ---------------------------------------------------------------------------
# training-side index work (include/peagle_train.h)
# ---------------------------------------------------------------------------

def pe_train_build_mask(out, n_max: int, K: int, mask_type: int, stream=None):
    """Fill out [n_max*K, ld] (uint8 for PE_MASK_BOOL_U8, bfloat16 for
    PE_MASK_ADDITIVE_BF16; ld = out.shape[1]) with the amortized mask."""
    if out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a row-major 2-D tensor")
    _check("pe_train_build_mask", lib().pe_train_build_mask(
        n_max, K, mask_type, ptr(out), out.stride(0), stream_ptr(stream)))
    return out


def pe_train_mask_view(mask, n_max: int, K: int, n: int):
    """The mask of an n-token sample: a view of the top-left block of the mask
    built for n_max (no copy)."""
    v = _vp()
    rows = ctypes.c_int64(0)
    ld = ctypes.c_int64(0)
    _check("pe_train_mask_view", lib().pe_train_mask_view(
        ptr(mask), mask.stride(0), n_max, K, n, ctypes.byref(v), ctypes.byref(rows),
        ctypes.byref(ld)))
    if v.value != mask.data_ptr() or ld.value != mask.stride(0):
        raise RuntimeError("pe_train_mask_view returned an unexpected view")
    return mask[: rows.value, : rows.value]


def pe_train_partition(n: int, K: int, r: float, u, bounds: Sequence[int], stream=None):
    """COD sampling + sequence partitioning of one n-token sample; u is a
    [n, K] float32 device tensor of draws.  Returns device tensors keep,
    seg, offsets, rows, owned (rows / owned trimmed to offsets[-1] by the
    caller)."""
    torch = _torch()
    S = len(bounds) - 1
    hb = (_i32 * (S + 1))(*[int(b) for b in bounds])
    cap = int(sum(bounds[:-1])) + n * K
    dev = u.device
    out = dict(keep=torch.empty(n, K, dtype=torch.uint8, device=dev),
               seg=torch.empty(n, K, dtype=torch.int32, device=dev),
               counts=torch.empty(max(S, 1), dtype=torch.int32, device=dev),
               offsets=torch.empty(S + 1, dtype=torch.int32, device=dev),
               rows=torch.empty(cap, dtype=torch.int32, device=dev),
               owned=torch.empty(cap, dtype=torch.uint8, device=dev))
    _check("pe_train_partition", lib().pe_train_partition(
        n, K, ctypes.c_float(r), ptr(u), S, hb, ptr(out["keep"]), ptr(out["seg"]),
        ptr(out["counts"]), ptr(out["offsets"]), ptr(out["rows"]), ptr(out["owned"]), cap,
        stream_ptr(stream)))
    return out
