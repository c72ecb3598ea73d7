"""CPU oracle for the compressed-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product package never imports it
and shares no code with it.

The arithmetic lives in ``kvq_oracle.cpp`` (plain C++, fp32 quantiser spec,
fp64 attention); this module builds and loads that library with ctypes and
offers numpy-level wrappers.  The one computation written here is the K-vs-V
sensitivity reference (``sensitivity_reference``): fp64 divergences in numpy
over the library's reconstruction, attention weights and outputs.  ``build_oracle()`` compiles it with g++ and
``-ffp-contract=off`` so that no multiply-add is fused on any host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.cpp")
_LIBDIR = os.path.join(_HERE, "_lib")

_libs: dict = {}


def lib_path(plant: int = 0) -> str:
    name = "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so"
    return os.path.join(_LIBDIR, name)


def build_oracle(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle into ``oracle/_lib``.  ``plant`` > 0 builds a copy
    with one deliberate mistake (used only by the test that shows the pins
    catch mistakes)."""
    out = lib_path(plant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_LIBDIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_PLANT={plant}",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(plant: int = 0) -> ctypes.CDLL:
    if plant in _libs:
        return _libs[plant]
    path = build_oracle(plant)
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f32, f64, u16 = (ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_double, ctypes.c_uint16)
    lib.oracle_bf16_to_f32.argtypes = [u16]
    lib.oracle_bf16_to_f32.restype = f32
    lib.oracle_f16_to_f32.argtypes = [u16]
    lib.oracle_f16_to_f32.restype = f32
    lib.oracle_f32_to_f16.argtypes = [f32]
    lib.oracle_f32_to_f16.restype = u16
    lib.oracle_quantize_row.argtypes = [P, i32, i32, i32, P, P, P]
    lib.oracle_quantize_row.restype = i32
    lib.oracle_pack_row.argtypes = [P, i32, i32, P]
    lib.oracle_pack_row.restype = i32
    lib.oracle_quantize_pack_rows.argtypes = [P, i64, i32, i32, i32, P, P, P]
    lib.oracle_quantize_pack_rows.restype = i32
    lib.oracle_code_slot.argtypes = [i32, i32, i32]
    lib.oracle_code_slot.restype = i32
    lib.oracle_quantize_pack_rows_stored.argtypes = [P, i64, i32, i32, i32, i32, P, P]
    lib.oracle_quantize_pack_rows_stored.restype = i32
    lib.oracle_dequant_row.argtypes = [P, P, P, i32, i32, P]
    lib.oracle_dequant_row.restype = None
    lib.oracle_is_packed.argtypes = [i32, i32, i32, i32, i32]
    lib.oracle_is_packed.restype = i32
    lib.oracle_reconstruct.argtypes = [P, i32, i32, i32, i32, i32, i32, P, i32, i32, P, P]
    lib.oracle_reconstruct.restype = i32
    lib.oracle_online_cores.argtypes = []
    lib.oracle_online_cores.restype = i32
    lib.oracle_attention.argtypes = [P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32]
    lib.oracle_attention.restype = i32
    lib.oracle_attention_weights.argtypes = [P, P, i32, i32, i32, i32, i32, f64, P]
    lib.oracle_attention_weights.restype = i32
    _libs[plant] = lib
    return lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


# --------------------------------------------------------------------------
# numpy-level wrappers (inputs are uint16 bit patterns for bf16 data)
# --------------------------------------------------------------------------

def f32_to_f16_bits(x: float, plant: int = 0) -> int:
    return int(load(plant).oracle_f32_to_f16(float(x)))


def f16_bits_to_f32(h: int, plant: int = 0) -> float:
    return float(load(plant).oracle_f16_to_f32(int(h)))


def quantize_row(x_bf16: np.ndarray, G: int, bits: int, plant: int = 0):
    """x_bf16: uint16[D].  Returns (codes uint8[D], s uint16[D/G], z uint16[D/G])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[0]
    codes = np.zeros(D, np.uint8)
    s = np.zeros(D // G, np.uint16)
    z = np.zeros(D // G, np.uint16)
    rc = load(plant).oracle_quantize_row(_ptr(x), D, G, bits, _ptr(codes), _ptr(s), _ptr(z))
    if rc != 0:
        raise ValueError("oracle_quantize_row rejected its arguments")
    return codes, s, z


def pack_row(codes: np.ndarray, bits: int, plant: int = 0) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    words = np.zeros(c.shape[0] * bits // 32, np.uint32)
    if load(plant).oracle_pack_row(_ptr(c), c.shape[0], bits, _ptr(words)) != 0:
        raise ValueError("oracle_pack_row rejected its arguments")
    return words


def quantize_pack_rows(x_bf16: np.ndarray, G: int, bits: int, plant: int = 0):
    """x_bf16 uint16 [..., D] -> (words uint32 [n, D*bits/32], s uint16 [n, D/G], z uint16 [n, D/G])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[-1]
    n = x.size // D
    words = np.zeros((n, D * bits // 32), np.uint32)
    s = np.zeros((n, D // G), np.uint16)
    z = np.zeros((n, D // G), np.uint16)
    rc = load(plant).oracle_quantize_pack_rows(_ptr(x), n, D, G, bits, _ptr(words), _ptr(s), _ptr(z))
    if rc != 0:
        raise ValueError("oracle_quantize_pack_rows rejected its arguments")
    return words, s, z


def code_slot(kind: str, bits: int, d: int, plant: int = 0) -> int:
    """Storage slot of element d in a packed K ("k") or V ("v") row."""
    return int(load(plant).oracle_code_slot(0 if kind == "k" else 1, bits, d))


def quantize_pack_rows_stored(x_bf16: np.ndarray, G: int, bits: int, kind: str, plant: int = 0):
    """x_bf16 uint16 [..., 128] -> (words uint32 [n, 128*bits/32] in the cache's
    storage order, sz uint16 [n, 2*128/G] = [z_0.., s_0..])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[-1]
    n = x.size // D
    words = np.zeros((n, D * bits // 32), np.uint32)
    sz = np.zeros((n, 2 * (D // G)), np.uint16)
    rc = load(plant).oracle_quantize_pack_rows_stored(_ptr(x), n, D, G, bits,
                                                      0 if kind == "k" else 1, _ptr(words), _ptr(sz))
    if rc != 0:
        raise ValueError("oracle_quantize_pack_rows_stored rejected its arguments")
    return words, sz


def dequant_row(codes, s, z, G: int, plant: int = 0) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    z = np.ascontiguousarray(z, dtype=np.uint16)
    out = np.zeros(c.shape[0], np.float64)
    load(plant).oracle_dequant_row(_ptr(c), _ptr(s), _ptr(z), c.shape[0], G, _ptr(out))
    return out


def is_packed(p: int, vis_start: int, vis_end: int, head_protected: bool, bits: int,
              plant: int = 0) -> bool:
    return bool(load(plant).oracle_is_packed(p, vis_start, vis_end, int(head_protected), bits))


def reconstruct(x_bf16: np.ndarray, vis_start: int, vis_end: int, prot, bits: int, G: int,
                plant: int = 0):
    """x_bf16: uint16 [B, H, T, D] -> (fp64 [B, H, T, D], number of packed rows)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    B, H, T, D = x.shape
    pr = np.ascontiguousarray(np.asarray(prot, dtype=np.uint8).reshape(H))
    out = np.empty(x.shape, np.float64)
    n = ctypes.c_int64(0)
    rc = load(plant).oracle_reconstruct(_ptr(x), B, H, T, D, vis_start, vis_end, _ptr(pr), bits,
                                        G, _ptr(out), ctypes.byref(n))
    if rc != 0:
        raise ValueError("oracle_reconstruct rejected its arguments")
    return out, int(n.value)


def online_cores() -> int:
    return int(load().oracle_online_cores())


def attention(q_bf16: np.ndarray, khat: np.ndarray, vhat: np.ndarray, scale: float,
              threads: int = 0, plant: int = 0):
    """q_bf16 uint16 [B, Hq, D]; khat/vhat fp64 [B, Hkv, T, D].
    Returns (out fp64 [B, Hq, D], lse fp64 [B, Hq])."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    k = np.ascontiguousarray(khat, dtype=np.float64)
    v = np.ascontiguousarray(vhat, dtype=np.float64)
    B, Hq, D = q.shape
    _, Hkv, T, _ = k.shape
    out = np.empty((B, Hq, D), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = load(plant).oracle_attention(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, T, D, float(scale),
                                      _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return out, lse


def attention_weights(q_bf16: np.ndarray, khat: np.ndarray, hq: int, scale: float,
                      plant: int = 0) -> np.ndarray:
    """Softmax weights of query head hq of a single sequence (B == 1)."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    k = np.ascontiguousarray(khat, dtype=np.float64)
    _, Hq, D = q.shape
    _, Hkv, T, _ = k.shape
    w = np.empty(T, np.float64)
    rc = load(plant).oracle_attention_weights(_ptr(q), _ptr(k), Hq, Hkv, T, D, hq, float(scale),
                                              _ptr(w))
    if rc != 0:
        raise ValueError("oracle_attention_weights rejected its arguments")
    return w


def decode_reference(q_bf16, k_bf16, v_bf16, vis_start: int, vis_end: int, prot, k_bits: int,
                     v_bits: int, G: int, scale: float, threads: int = 0, plant: int = 0):
    """Whole decode step for one layer: reconstruct K and V under the policy,
    then exact fp64 attention.  Returns (out, lse, khat, vhat).  prot[h]: 0 =
    quantised, 1 = K and V of the head's visual rows kept bf16, 2 = only its
    K kept bf16 (HeadGuard brief: image Key, and Value as needed)."""
    pm = [int(m) for m in np.asarray(prot).reshape(-1)]
    k_prot = [1 if m in (1, 2) else 0 for m in pm]
    if plant == 11:  # planted: a K-only head keeps its V in bf16 too
        v_prot = [1 if m in (1, 2) else 0 for m in pm]
    else:
        v_prot = [1 if m == 1 else 0 for m in pm]
    khat, _ = reconstruct(k_bf16, vis_start, vis_end, k_prot, k_bits, G, plant)
    vhat, _ = reconstruct(v_bf16, vis_start, vis_end, v_prot, v_bits, G, plant)
    out, lse = attention(q_bf16, khat, vhat, scale, threads, plant)
    return out, lse, khat, vhat


def sensitivity_reference(q_bf16, k_bf16, v_bf16, vis_start: int, vis_end: int, prot, k_bits: int,
                          v_bits: int, G: int, scale: float, readout, plant: int = 0):
    """K-vs-V sensitivity of one layer's compressed cache, in fp64.

    "VLM_KV_Quantization" sections 3-4 measure quantisation damage as the
    KL divergence D_KL(P_fp || P_q) of the model's output distribution from
    the unquantised one, quantising visual K or visual V alone with the same
    tokens, bits and group size.  Without a model, per (b, hq):
      kl_attn = D_KL(p || p_hat): softmax weights over positions with the raw
                bf16 K (p) and with K as the decode reads it (p_hat);
      kl_out  = D_KL(P || P_hat): P = softmax(readout @ o) with o the
                attention output over the raw cache, P_hat the same over the
                cache as the decode reads it (readout [n_out, D] fp32 stands
                for the layers after attention);
      err     = ||o_hat - o||_2.
    The cache as read is decode_reference's policy (prot, k_bits, v_bits,
    G); the raw cache is the same inputs with nothing quantised.  Returns
    fp64 [B, Hq, 3] = (kl_attn, kl_out, err)."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    B, Hq, D = q.shape
    Hkv = k_bf16.shape[1]
    kb, vb = (v_bits, k_bits) if plant == 13 else (k_bits, v_bits)  # planted: K and V swapped
    o, _, kx, _ = decode_reference(q, k_bf16, v_bf16, vis_start, vis_end, [0] * Hkv, 16, 16, G, scale,
                                   plant=plant)
    oh, _, kh, _ = decode_reference(q, k_bf16, v_bf16, vis_start, vis_end, prot, kb, vb, G, scale,
                                    plant=plant)
    W = np.asarray(readout, dtype=np.float32).astype(np.float64)
    res = np.empty((B, Hq, 3), np.float64)

    def kl(a, b, log_a, log_b):
        if plant == 12:  # planted: divergence taken in the other direction
            a, b, log_a, log_b = b, a, log_b, log_a
        return float(np.sum(a * (log_a - log_b)))

    def log_softmax(z):
        m = np.max(z)
        return z - (m + np.log(np.sum(np.exp(z - m))))

    for b in range(B):
        for hq in range(Hq):
            p = attention_weights(q[b:b + 1], kx[b:b + 1], hq, scale, plant)
            ph = attention_weights(q[b:b + 1], kh[b:b + 1], hq, scale, plant)
            res[b, hq, 0] = kl(p, ph, np.log(p), np.log(ph))
            lz = log_softmax(W @ o[b, hq])
            lzh = log_softmax(W @ oh[b, hq])
            res[b, hq, 1] = kl(np.exp(lz), np.exp(lzh), lz, lzh)
            res[b, hq, 2] = float(np.sqrt(np.sum((oh[b, hq] - o[b, hq]) ** 2)))
    return res
