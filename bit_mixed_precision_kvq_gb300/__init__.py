"""Thin Python binding of the kvq C ABI (``include/kvq.h``).

Argument marshalling only: every step of the path runs in the CUDA library
``_lib/libkvq.so`` (built by ``build_native.build()``).  There is no Python
or CPU fallback -- if the library is missing, ``load()`` raises.

Functions take either torch tensors (device memory, the current torch stream
by default) or raw integer addresses.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

__all__ = [
    "KvqError", "load", "lib_path", "cache_layout", "quantize_append", "decode_attention",
    "kvq_cache_layout", "kvq_quantize_append", "kvq_decode_attention", "KVQ_MAX_HEADS",
    "decode_attention_static_ws", "kvq_decode_attention_static_ws", "STATIC_WS_BYTES",
    "decode_step", "kvq_decode_step", "decode_attention_ragged", "kvq_decode_attention_ragged",
    "decode_step_ragged", "kvq_decode_step_ragged", "sensitivity_probe", "kvq_sensitivity_probe",
    "probe_workspace_bytes", "kvq_probe_workspace_bytes", "decode_attention_mq",
    "kvq_decode_attention_mq", "decode_mq_workspace_bytes", "kvq_decode_mq_workspace_bytes",
    "KVQ_MAX_QUERY_TOKENS", "workspace_status", "kvq_workspace_status", "set_wait_limits",
    "kvq_set_wait_limits", "set_cache_preload", "kvq_set_cache_preload", "STATUS_TILE_WAIT", "STATUS_PEER_WAIT", "STATUS_COUNTER",
    "SEG_K_CODES", "SEG_K_SZ", "SEG_V_CODES", "SEG_V_SZ", "SEG_PROT_K", "SEG_PROT_V",
    "SEG_TEXT_K", "SEG_TEXT_V", "EXPORTED_SYMBOLS",
]

KVQ_MAX_HEADS = 128
KVQ_MAX_QUERY_TOKENS = 64
KVQ_NSEG = 8
(SEG_K_CODES, SEG_K_SZ, SEG_V_CODES, SEG_V_SZ, SEG_PROT_K, SEG_PROT_V, SEG_TEXT_K,
 SEG_TEXT_V) = range(8)
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED",
          3: "KVQ_ERR_CAPACITY", 4: "KVQ_ERR_CUDA"}
EXPORTED_SYMBOLS = ["kvq_cache_layout", "kvq_quantize_append", "kvq_decode_attention",
                    "kvq_decode_step", "kvq_decode_attention_ragged", "kvq_decode_step_ragged",
                    "kvq_sensitivity_probe", "kvq_probe_workspace_bytes", "kvq_decode_attention_mq",
                    "kvq_decode_mq_workspace_bytes",
                    "kvq_decode_attention_static_ws", "kvq_workspace_status", "kvq_set_wait_limits",
                    "kvq_set_cache_preload",
                    "kvq_last_cuda_error", "kvq_status_string"]
STATUS_TILE_WAIT, STATUS_PEER_WAIT, STATUS_COUNTER = 1, 2, 4  # KVQ_STATUS_* bits
STATIC_WS_BYTES = 16 * 1024 * 1024  # KVQ_STATIC_WS_BYTES

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "_lib", "libkvq.so")


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {STATUS.get(status, status)}"
        self.cuda_error = 0
        if status == 4 and _lib is not None:
            self.cuda_error = int(_lib.kvq_last_cuda_error())
            msg += f" (cudaError {self.cuda_error})"
        super().__init__(msg)
        self.status = status


class LayoutDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("T_cap", ctypes.c_int32), ("vis_start", ctypes.c_int32),
                ("vis_end", ctypes.c_int32), ("k_bits", ctypes.c_int32),
                ("v_bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("protected_heads", ctypes.c_uint8 * KVQ_MAX_HEADS)]


class Layout(ctypes.Structure):
    _fields_ = [("d", LayoutDesc), ("g", ctypes.c_int32), ("n_prot", ctypes.c_int32),
                ("n_packed", ctypes.c_int32), ("Tv", ctypes.c_int32), ("Tv_pad", ctypes.c_int32),
                ("T_text", ctypes.c_int32),
                ("units", ctypes.c_int32),
                ("slot", ctypes.c_int32 * KVQ_MAX_HEADS),
                ("prot_head", ctypes.c_uint8 * KVQ_MAX_HEADS),
                ("packed_head", ctypes.c_uint8 * KVQ_MAX_HEADS),
                ("row_bytes", ctypes.c_int64 * KVQ_NSEG), ("off", ctypes.c_int64 * KVQ_NSEG),
                ("bytes", ctypes.c_int64 * KVQ_NSEG), ("total_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("eff_bits_k", ctypes.c_double),
                ("eff_bits_v", ctypes.c_double), ("n_konly", ctypes.c_int32),
                ("konly_head", ctypes.c_uint8 * KVQ_MAX_HEADS)]


_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"kvq native library missing at {path}; build it with "
                           "bit_mixed_precision_kvq_gb300.build_native.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    lib.kvq_cache_layout.argtypes = [ctypes.POINTER(LayoutDesc), ctypes.POINTER(Layout)]
    lib.kvq_cache_layout.restype = ctypes.c_int
    lib.kvq_quantize_append.argtypes = [ctypes.POINTER(Layout), P, P, P, i64, i64, i64, i32, i32, P]
    lib.kvq_quantize_append.restype = ctypes.c_int
    lib.kvq_decode_attention.argtypes = [ctypes.POINTER(Layout), P, P, i32, f32, P, P, P, sz, P]
    lib.kvq_decode_attention.restype = ctypes.c_int
    lib.kvq_decode_step.argtypes = [ctypes.POINTER(Layout), P, P, P, P, i32, f32, P, P, P, sz, P]
    lib.kvq_decode_step.restype = ctypes.c_int
    lib.kvq_decode_attention_ragged.argtypes = [ctypes.POINTER(Layout), P, P, P, i32, f32, P, P, P, sz, P]
    lib.kvq_decode_attention_ragged.restype = ctypes.c_int
    lib.kvq_decode_step_ragged.argtypes = [ctypes.POINTER(Layout), P, P, P, P, P, i32, f32, P, P, P, sz,
                                           P]
    lib.kvq_decode_step_ragged.restype = ctypes.c_int
    lib.kvq_decode_mq_workspace_bytes.argtypes = [ctypes.POINTER(Layout), i32]
    lib.kvq_decode_mq_workspace_bytes.restype = sz
    lib.kvq_decode_attention_mq.argtypes = [ctypes.POINTER(Layout), P, P, i32, i32, f32, P, P, P, sz, P]
    lib.kvq_decode_attention_mq.restype = ctypes.c_int
    lib.kvq_probe_workspace_bytes.argtypes = [ctypes.POINTER(Layout), i32]
    lib.kvq_probe_workspace_bytes.restype = sz
    lib.kvq_sensitivity_probe.argtypes = [ctypes.POINTER(Layout), P, P, P, P, i64, i64, i64, i32, f32, P,
                                          i32, P, P, sz, P]
    lib.kvq_sensitivity_probe.restype = ctypes.c_int
    lib.kvq_decode_attention_static_ws.argtypes = [ctypes.POINTER(Layout), P, P, i32, f32, P, P, P]
    lib.kvq_decode_attention_static_ws.restype = ctypes.c_int
    lib.kvq_workspace_status.argtypes = [P, P, P]
    lib.kvq_workspace_status.restype = ctypes.c_int
    lib.kvq_set_wait_limits.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.kvq_set_wait_limits.restype = None
    lib.kvq_set_cache_preload.argtypes = [ctypes.c_int32]
    lib.kvq_set_cache_preload.restype = None
    lib.kvq_last_cuda_error.argtypes = []
    lib.kvq_last_cuda_error.restype = ctypes.c_int
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def cache_layout(B: int, H_q: int, H_kv: int, D: int, T_cap: int, vis_start: int, vis_end: int,
                 k_bits: int, v_bits: int, group_size: int,
                 protected: Sequence[int] = (), k_only: Sequence[int] = ()) -> Layout:
    """kvq_cache_layout: validate the per-layer description and derive the layout.
    ``protected`` lists the KV heads whose visual K and V stay bf16, ``k_only``
    those whose visual K alone stays bf16 (V quantised)."""
    d = LayoutDesc(B, H_q, H_kv, D, T_cap, vis_start, vis_end, k_bits, v_bits, group_size)
    for mode, heads in ((1, protected), (2, k_only)):
        for h in heads:
            if not 0 <= int(h) < KVQ_MAX_HEADS or d.protected_heads[int(h)] != 0:
                raise KvqError(1, "kvq_cache_layout")
            d.protected_heads[int(h)] = mode
    out = Layout()
    st = load().kvq_cache_layout(ctypes.byref(d), ctypes.byref(out))
    if st != 0:
        raise KvqError(st, "kvq_cache_layout")
    return out


def quantize_append(L: Layout, cache, k, v, t0: int, n_tok: Optional[int] = None,
                    strides: Optional[Sequence[int]] = None, stream=None) -> None:
    """kvq_quantize_append: write positions [t0, t0 + n_tok) of K and V
    ([B, H_kv, n_tok, D] bf16 on the device) into the cache."""
    if strides is None:
        if k.stride() != v.stride():
            raise ValueError("k and v must share strides")
        if k.stride(-1) != 1:
            raise ValueError("last dim must be contiguous")
        strides = k.stride()[:3]
        n_tok = k.shape[2] if n_tok is None else n_tok
    st = load().kvq_quantize_append(ctypes.byref(L), _addr(cache), _addr(k), _addr(v),
                                    int(strides[0]), int(strides[1]), int(strides[2]), int(t0),
                                    int(n_tok), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_quantize_append")


def decode_attention(L: Layout, cache, q, T: int, out, softmax_scale: Optional[float] = None,
                     lse=None, workspace=None, ws_bytes: Optional[int] = None,
                     stream=None) -> None:
    """kvq_decode_attention: out[b, hq] = softmax(scale q . k) v over positions [0, T)."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kvq_decode_attention(ctypes.byref(L), _addr(cache), _addr(q), int(T),
                                     float(softmax_scale), _addr(out), _addr(lse),
                                     _addr(workspace), int(ws_bytes), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_attention")


def decode_step(L: Layout, cache, q, k_new, v_new, t_new: int, out,
                softmax_scale: Optional[float] = None, lse=None, workspace=None,
                ws_bytes: Optional[int] = None, stream=None) -> None:
    """kvq_decode_step: one fused decode step.  Stores the new token's bf16 K/V
    rows ([B, H_kv, D]) at text position t_new and attends q over [0, t_new]
    in one cooperative launch.  The workspace's first 4 bytes must be zero
    before its first use (every call leaves them zero)."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kvq_decode_step(ctypes.byref(L), _addr(cache), _addr(q), _addr(k_new),
                                _addr(v_new), int(t_new), float(softmax_scale), _addr(out),
                                _addr(lse), _addr(workspace), int(ws_bytes), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_step")


def decode_attention_ragged(L: Layout, cache, q, seq_len, T_max: int, out,
                            softmax_scale: Optional[float] = None, lse=None, workspace=None,
                            ws_bytes: Optional[int] = None, stream=None) -> None:
    """kvq_decode_attention_ragged: sequence b attends positions
    [0, seq_len[b]) (seq_len: device int32 [B]; an entry outside [1, T_max]
    marks an inactive sequence, whose outputs are zero and lse -inf)."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kvq_decode_attention_ragged(ctypes.byref(L), _addr(cache), _addr(q), _addr(seq_len),
                                            int(T_max), float(softmax_scale), _addr(out), _addr(lse),
                                            _addr(workspace), int(ws_bytes), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_attention_ragged")


def decode_step_ragged(L: Layout, cache, q, k_new, v_new, t_new, T_max: int, out,
                       softmax_scale: Optional[float] = None, lse=None, workspace=None,
                       ws_bytes: Optional[int] = None, stream=None) -> None:
    """kvq_decode_step_ragged: sequence b stores its row at t_new[b] (device
    int32 [B]) and attends [0, t_new[b]]; an entry outside [0, T_max) or
    inside the visual range marks an inactive sequence (nothing stored,
    outputs zero, lse -inf).  Workspace rules as for decode_step."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kvq_decode_step_ragged(ctypes.byref(L), _addr(cache), _addr(q), _addr(k_new),
                                       _addr(v_new), _addr(t_new), int(T_max), float(softmax_scale),
                                       _addr(out), _addr(lse), _addr(workspace), int(ws_bytes),
                                       _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_step_ragged")


def decode_mq_workspace_bytes(L: Layout, n_q: int) -> int:
    """kvq_decode_mq_workspace_bytes: workspace bytes of decode_attention_mq."""
    return int(load().kvq_decode_mq_workspace_bytes(ctypes.byref(L), int(n_q)))


def decode_attention_mq(L: Layout, cache, q, T: int, out, softmax_scale: Optional[float] = None,
                        lse=None, workspace=None, ws_bytes: Optional[int] = None,
                        stream=None) -> None:
    """kvq_decode_attention_mq: q [B, n_q, H_q, D] bf16; token i attends
    positions [0, T - n_q + 1 + i); out [B, n_q, H_q, D], lse [B, n_q, H_q]."""
    n_q = int(q.shape[1])
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kvq_decode_attention_mq(ctypes.byref(L), _addr(cache), _addr(q), n_q, int(T),
                                        float(softmax_scale), _addr(out), _addr(lse),
                                        _addr(workspace), int(ws_bytes), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_attention_mq")


def probe_workspace_bytes(L: Layout, T: int) -> int:
    """kvq_probe_workspace_bytes: scratch bytes of sensitivity_probe over T positions."""
    return int(load().kvq_probe_workspace_bytes(ctypes.byref(L), int(T)))


def sensitivity_probe(L: Layout, cache, q, k, v, T: int, readout, result,
                      softmax_scale: Optional[float] = None, workspace=None,
                      ws_bytes: Optional[int] = None, strides: Optional[Sequence[int]] = None,
                      stream=None) -> None:
    """kvq_sensitivity_probe: per (b, hq), fp64 (kl_attn, kl_out, err) of
    the cache against the raw rows k, v ([B, H_kv, >= T, D] bf16 on the
    device) into result ([B, H_q, 3] float64); readout [n_out, D] float32."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    if strides is None:
        if k.stride() != v.stride():
            raise ValueError("k and v must share strides")
        if k.stride(-1) != 1:
            raise ValueError("last dim must be contiguous")
        strides = k.stride()[:3]
    n_out = readout.shape[0] if hasattr(readout, "shape") else 0
    if workspace is None:
        import torch
        workspace = torch.empty(max(1, probe_workspace_bytes(L, T)), dtype=torch.uint8,
                                device=result.device)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    st = load().kvq_sensitivity_probe(ctypes.byref(L), _addr(cache), _addr(q), _addr(k), _addr(v),
                                      int(strides[0]), int(strides[1]), int(strides[2]), int(T),
                                      float(softmax_scale), _addr(readout), int(n_out), _addr(result),
                                      _addr(workspace), int(ws_bytes), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_sensitivity_probe")


def decode_attention_static_ws(L: Layout, cache, q, T: int, out,
                               softmax_scale: Optional[float] = None, lse=None,
                               stream=None) -> None:
    """kvq_decode_attention_static_ws: same result as decode_attention, for
    callers that may not allocate device memory -- the scratch is a fixed
    array inside the library (STATIC_WS_BYTES per GPU).  Calls on one device
    share that array, so they must not overlap on the GPU."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(L.d.D)
    st = load().kvq_decode_attention_static_ws(ctypes.byref(L), _addr(cache), _addr(q), int(T),
                                               float(softmax_scale), _addr(out), _addr(lse),
                                               _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_decode_attention_static_ws")


def workspace_status(workspace, stream=None) -> int:
    """kvq_workspace_status: the KVQ_STATUS_* bits OR-ed into the
    workspace's status word (synchronises the stream to read them)."""
    import torch
    host = torch.zeros(1, dtype=torch.int32).pin_memory()
    st = load().kvq_workspace_status(_addr(workspace), _addr(host), _stream(stream))
    if st != 0:
        raise KvqError(st, "kvq_workspace_status")
    s = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(s, int):
        torch.cuda.synchronize()
    else:
        s.synchronize()
    return int(host.item()) & 0xFFFFFFFF


def set_wait_limits(tile_polls: int = 0, peer_polls: int = 0) -> None:
    """kvq_set_wait_limits: bounded-wait limits of later decode calls from
    this host thread (0 = default)."""
    load().kvq_set_wait_limits(int(tile_polls), int(peer_polls))


def set_cache_preload(enable: bool) -> None:
    """kvq_set_cache_preload: later uniform single-query decode calls from
    this host thread copy their first cache tiles before the previous
    kernel in the stream has finished (requires that no kernel outside this
    library writes the cache just before a call)."""
    load().kvq_set_cache_preload(1 if enable else 0)


# Same names as the C entry points.
kvq_cache_layout = cache_layout
kvq_quantize_append = quantize_append
kvq_decode_attention = decode_attention
kvq_decode_attention_static_ws = decode_attention_static_ws
kvq_decode_step = decode_step
kvq_decode_attention_ragged = decode_attention_ragged
kvq_decode_step_ragged = decode_step_ragged
kvq_sensitivity_probe = sensitivity_probe
kvq_decode_attention_mq = decode_attention_mq
kvq_decode_mq_workspace_bytes = decode_mq_workspace_bytes
kvq_probe_workspace_bytes = probe_workspace_bytes
kvq_workspace_status = workspace_status
kvq_set_wait_limits = set_wait_limits
kvq_set_cache_preload = set_cache_preload
