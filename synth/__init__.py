"""Seeded synthetic inputs for the compressed-KV decode path.

This module holds NO arithmetic of the method: it only draws random tensors
(q, K, V, protected-head masks) with the shapes, value distributions and
structure of the workloads the pages describe, and it is the only module that
both the CPU oracle's tests and the CUDA path's tests/bench use.

Generator (counter-based, so any slice can be drawn independently and the same
definition runs on CPU and GPU tensors):
  * key  = splitmix64(seed XOR splitmix64(stream id))
  * element i of a stream: z1 = splitmix64(key + 2i), z2 = splitmix64(key + 2i + 1)
  * u1 = ((z1 >> 11) + 1) / 2^53  in (0, 1],   u2 = (z2 >> 11) / 2^53  in [0, 1)
  * normal = sqrt(-2 ln u1) * cos(2 pi u2)     (Box-Muller, fp64), then -> bf16.
splitmix64 is Steele, Lea and Flood's 64-bit mixer (2014).

Workload shapes (from the pages):
  * LLaVA-OneVision-7B: GQA 28 query / 4 KV heads, D = 128, 32 frames x ~196
    visual tokens ~ 6,273, 14 historical text tokens before them, K stored
    after RoPE ("VLM_KV_Quantization", §2).
  * about 1/8 of KV heads protected in bf16 (HeadGuard brief, key ideas).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

MASK64 = (1 << 64) - 1
BASE_SEED = 20261202


def _s64(x: int) -> int:
    """Python int (mod 2^64) -> the int64 with the same bit pattern."""
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)


def splitmix64_int(x: int) -> int:
    """splitmix64 on a Python int (reference scalar form)."""
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _lsr(t: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor viewed as uint64."""
    return (t >> k) & ((1 << (64 - k)) - 1)


def splitmix64_t(x: torch.Tensor) -> torch.Tensor:
    """splitmix64 on an int64 tensor (wrapping two's-complement arithmetic)."""
    z = x + _GOLDEN
    z = (z ^ _lsr(z, 30)) * _M1
    z = (z ^ _lsr(z, 27)) * _M2
    return z ^ _lsr(z, 31)


def stream_key(*ids: int, seed: int = BASE_SEED) -> int:
    """Derive a 64-bit stream key from a tuple of small integers."""
    k = seed & MASK64
    for i in ids:
        k = splitmix64_int(k ^ splitmix64_int(i & MASK64))
    return k


_TWO53 = float(1 << 53)


def normal(n: int, key: int, device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """n standard normals (fp64 -> returned as fp32) of stream `key`."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    k = _s64(key)
    for start in range(0, n, chunk):
        m = min(chunk, n - start)
        idx = torch.arange(start, start + m, dtype=torch.int64, device=device)
        c = idx * 2 + k
        z1 = splitmix64_t(c)
        z2 = splitmix64_t(c + 1)
        u1 = (_lsr(z1, 11).to(torch.float64) + 1.0) / _TWO53
        u2 = _lsr(z2, 11).to(torch.float64) / _TWO53
        r = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        out[start:start + m] = r.to(torch.float32)
    return out


def uniform_ints(n: int, hi: int, key: int) -> List[int]:
    """n integers in [0, hi) (host side, for small choices such as head masks)."""
    return [splitmix64_int((key + i) & MASK64) % hi for i in range(n)]


def sample_without_replacement(k: int, n: int, key: int) -> List[int]:
    """k distinct values from range(n), seeded (partial Fisher-Yates)."""
    pool = list(range(n))
    for i in range(k):
        j = i + splitmix64_int((key + i) & MASK64) % (n - i)
        pool[i], pool[j] = pool[j], pool[i]
    return sorted(pool[:k])


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

@dataclass
class LayerSpec:
    k_bits: int
    v_bits: int
    protected: List[int]


@dataclass
class Workload:
    name: str
    n_layers: int
    B: int
    H_q: int
    H_kv: int
    D: int
    T: int            # historical positions (text + visual)
    n_text_prefix: int
    n_visual: int
    group_size: int
    layers: List[LayerSpec]
    k_structure: str  # "iid", "outliers_rope", "lognormal", "outliers8", "outliers"
    seed_id: int
    extra: dict = field(default_factory=dict)

    @property
    def vis_start(self) -> int:
        return self.n_text_prefix

    @property
    def vis_end(self) -> int:
        return self.n_text_prefix + self.n_visual

    @property
    def g(self) -> int:
        return self.H_q // self.H_kv


def _prot_sets(seed_id: int, n_layers: int, k: int, H: int) -> List[List[int]]:
    return [sample_without_replacement(k, H, stream_key(seed_id, l, 77)) for l in range(n_layers)]


def workload(name: str, T: Optional[int] = None) -> Workload:
    """The five workloads, by name:
    tiny, llava_ov_7b, llava15_7b, longctx (T in 1024..32768), llava_next_13b."""
    if name == "tiny":
        return Workload("tiny", 1, 1, 4, 1, 128, 256, 14, 242, 32,
                        [LayerSpec(4, 4, [])], "iid", 1)
    if name == "llava_ov_7b":
        L = 28
        return Workload("llava_ov_7b", L, 1, 28, 4, 128, 6287, 14, 6273, 64,
                        [LayerSpec(4, 2, [0]) for _ in range(L)], "outliers_rope", 2)
    if name == "llava15_7b":
        L = 32
        prot = _prot_sets(3, L, 4, 32)
        return Workload("llava15_7b", L, 16, 32, 32, 128, 616, 40, 576, 32,
                        [LayerSpec(8, 4, prot[l]) for l in range(L)], "lognormal", 3)
    if name == "longctx":
        T = 32768 if T is None else int(T)
        prot = _prot_sets(4, 1, 1, 8)
        return Workload(f"longctx_T{T}", 1, 8, 32, 8, 128, T, 32, T - 32, 32,
                        [LayerSpec(2, 2, prot[0])], "outliers8", 4 + 100 * T)
    if name == "llava_next_13b":
        L = 40
        prot = _prot_sets(5, L, 5, 40)
        layers = [LayerSpec(8, 8, prot[l]) if l < 4 else LayerSpec(4, 2, prot[l])
                  for l in range(L)]
        return Workload("llava_next_13b", L, 32, 40, 40, 128, 2940, 60, 2880, 64,
                        layers, "outliers", 5)
    raise KeyError(name)


def _outlier_channels(seed_id: int, layer: int, head: int, k: int, D: int) -> List[int]:
    return sample_without_replacement(k, D, stream_key(seed_id, layer, 88, head))


def _rope_(x: torch.Tensor, base: float = 1.0e6) -> torch.Tensor:
    """Rotate-half RoPE over the last dim, positions 0..T-1 along dim -2 (fp32)."""
    T, D = x.shape[-2], x.shape[-1]
    half = D // 2
    inv = base ** (-(torch.arange(half, dtype=torch.float64, device=x.device) * 2.0 / D))
    pos = torch.arange(T, dtype=torch.float64, device=x.device)
    ang = pos[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    x1, x2 = x[..., :half].clone(), x[..., half:].clone()
    x[..., :half] = x1 * cos - x2 * sin
    x[..., half:] = x2 * cos + x1 * sin
    return x


def make_kv(w: Workload, layer: int, which: str, device="cpu",
            b_range: Optional[Sequence[int]] = None,
            h_range: Optional[Sequence[int]] = None,
            T: Optional[int] = None) -> torch.Tensor:
    """K or V of one layer as bf16 [B', H', T, D] (optionally a slice of the
    batch / heads: each (b, h) row is its own stream, so slices match the full
    tensor exactly)."""
    T = w.T if T is None else T
    bs = list(range(w.B)) if b_range is None else list(b_range)
    hs = list(range(w.H_kv)) if h_range is None else list(h_range)
    tid = 1 if which == "k" else 2
    out = torch.empty((len(bs), len(hs), T, w.D), dtype=torch.bfloat16, device=device)
    for i, b in enumerate(bs):
        for j, h in enumerate(hs):
            x = normal(T * w.D, stream_key(w.seed_id, layer, tid, b, h), device).view(T, w.D)
            if which == "k":
                if w.k_structure in ("outliers_rope", "outliers"):
                    for c in _outlier_channels(w.seed_id, layer, h, 4, w.D):
                        x[:, c] *= 10.0
                    if w.k_structure == "outliers_rope":
                        _rope_(x)
                elif w.k_structure == "outliers8":
                    for c in _outlier_channels(w.seed_id, layer, h, round(0.02 * w.D), w.D):
                        x[:, c] *= 8.0
                elif w.k_structure == "lognormal":
                    mag = torch.exp(0.5 * normal(w.D, stream_key(w.seed_id, layer, 99, h), device))
                    x *= mag[None, :]
            out[i, j] = to_bf16(x)
    return out


def make_q(w: Workload, layer: int, step: int = 0, device="cpu") -> torch.Tensor:
    """Decode queries bf16 [B, H_q, D] ~ N(0, 1), no RoPE."""
    x = normal(w.B * w.H_q * w.D, stream_key(w.seed_id, layer, 3, step), device)
    return to_bf16(x.view(w.B, w.H_q, w.D))


def make_step_kv(w: Workload, layer: int, which: str, step: int = 0, device="cpu") -> torch.Tensor:
    """K or V of the current decode step: bf16 [B, H_kv, 1, D] ~ N(0, 1)."""
    tid = 4 if which == "k" else 5
    x = normal(w.B * w.H_kv * w.D, stream_key(w.seed_id, layer, tid, step), device)
    return to_bf16(x.view(w.B, w.H_kv, 1, w.D))


def random_case(seed: int, B: int, H_q: int, H_kv: int, D: int, T: int, device="cpu",
                scale_k: float = 1.0):
    """Small i.i.d. N(0,1) case for fuzz tests: (q, K, V) bf16."""
    q = to_bf16(normal(B * H_q * D, stream_key(seed, 11), device).view(B, H_q, D))
    k = to_bf16(scale_k * normal(B * H_kv * T * D, stream_key(seed, 12), device).view(B, H_kv, T, D))
    v = to_bf16(normal(B * H_kv * T * D, stream_key(seed, 13), device).view(B, H_kv, T, D))
    return q, k, v
