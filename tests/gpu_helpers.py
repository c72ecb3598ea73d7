"""Helpers for the GPU parity tests: build a cache through the C ABI, read
its segments back, and compare them with the CPU oracle."""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import oracle
import synth

TOL = 4e-3  # max |o_gpu - o_oracle| <= TOL * max|V_hat| of that (b, h)


@dataclass
class Case:
    B: int
    H_q: int
    H_kv: int
    T_cap: int
    vs: int
    ve: int
    kb: int
    vb: int
    G: int
    prot: List[int]
    D: int = 128
    konly: List[int] = field(default_factory=list)  # K-only protected heads

    def layout(self):
        return kvq.cache_layout(self.B, self.H_q, self.H_kv, self.D, self.T_cap, self.vs, self.ve,
                                self.kb, self.vb, self.G, self.prot, self.konly)

    def mask(self):
        """Protection mode per KV head: 1 K and V, 2 K only, 0 none."""
        return [1 if h in self.prot else (2 if h in self.konly else 0) for h in range(self.H_kv)]


def case_of(w: synth.Workload, layer: int, extra: int = 0) -> Case:
    ls = w.layers[layer]
    return Case(w.B, w.H_q, w.H_kv, w.T + extra, w.vis_start, w.vis_end, ls.k_bits, ls.v_bits,
                w.group_size, list(ls.protected))


def alloc_cache(L, device="cuda", fill: int = 0xA5) -> torch.Tensor:
    c = torch.full((int(L.total_bytes),), fill, dtype=torch.uint8, device=device)
    assert c.data_ptr() % 256 == 0
    return c


def append(L, cache, k: torch.Tensor, v: torch.Tensor, t0: int = 0) -> None:
    kvq.quantize_append(L, cache, k, v, t0)


def decode(L, cache, q: torch.Tensor, T: int, scale: Optional[float] = None, ws_fill=None):
    B, Hq, D = q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=q.device)
    if ws_fill is not None:
        ws.fill_(ws_fill)
    kvq.decode_attention(L, cache, q, T, out, scale, lse, ws)
    return out, lse


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def seg(L, cache_np: np.ndarray, s: int, dtype) -> np.ndarray:
    o, n = int(L.off[s]), int(L.bytes[s])
    return cache_np[o:o + n].view(dtype)


def check_append(L, c: Case, cache: torch.Tensor, k_np: np.ndarray, v_np: np.ndarray,
                 t_hi: int, b_sel: Optional[Sequence[int]] = None) -> int:
    """Every position in [0, t_hi) of the cache against the oracle:
    packed codes (in the cache's storage order), scales and zeros
    word-for-word, bf16 rows bit-identical.
    k_np/v_np: uint16 [B', H_kv, >= t_hi, D] for the batch entries b_sel.
    Returns the number of packed rows compared."""
    cn = cache.cpu().numpy()
    B, H, D, Tv, Tt = c.B, c.H_kv, c.D, int(L.Tv), int(L.T_text)
    Tvp = int(L.Tv_pad)
    b_sel = list(range(B)) if b_sel is None else list(b_sel)
    prot = [h for h in range(H) if h in c.prot]
    konly = [h for h in range(H) if h in c.konly]
    pack = [h for h in range(H) if h not in c.prot and h not in c.konly]
    nvis = max(0, min(t_hi, c.ve) - c.vs)
    n_rows = 0
    for which, x_np, nbits, sc, ssz, sp, stx in (
            ("k", k_np, c.kb, kvq.SEG_K_CODES, kvq.SEG_K_SZ, kvq.SEG_PROT_K, kvq.SEG_TEXT_K),
            ("v", v_np, c.vb, kvq.SEG_V_CODES, kvq.SEG_V_SZ, kvq.SEG_PROT_V, kvq.SEG_TEXT_V)):
        text = seg(L, cn, stx, np.uint16).reshape(B, H, Tt, D)
        pre = min(t_hi, c.vs)
        post = max(0, t_hi - c.ve)
        for i, b in enumerate(b_sel):
            assert np.array_equal(text[b, :, :pre], x_np[i, :, :pre]), f"{which} text prefix b={b}"
            if post:
                assert np.array_equal(text[b, :, c.vs:c.vs + post], x_np[i, :, c.ve:c.ve + post]), \
                    f"{which} text suffix b={b}"
        if nvis == 0:
            continue
        # bf16 visual rows: K of protected then K-only heads; V of protected heads
        bf = prot + konly if which == "k" else prot
        # packed visual rows: K of packed heads; V of packed then K-only heads
        pk = pack if which == "k" else pack + konly
        if bf:
            pr = seg(L, cn, sp, np.uint16).reshape(B, len(bf), Tv, D)
            for i, b in enumerate(b_sel):
                assert np.array_equal(pr[b, :, :nvis], x_np[i][bf][:, c.vs:c.vs + nvis]), \
                    f"{which} protected rows b={b}"
        if not pk:
            continue
        if nbits == 16:
            raw = seg(L, cn, sc, np.uint16).reshape(B, len(pk), Tvp, D)
            for i, b in enumerate(b_sel):
                assert np.array_equal(raw[b, :, :nvis], x_np[i][pk][:, c.vs:c.vs + nvis])
            continue
        W = D * nbits // 32
        ng = D // c.G
        words = seg(L, cn, sc, np.uint32).reshape(B, len(pk), Tvp, W)
        sz = seg(L, cn, ssz, np.uint16).reshape(B, len(pk), Tvp, 2 * ng)
        for i, b in enumerate(b_sel):
            xin = np.ascontiguousarray(x_np[i][pk][:, c.vs:c.vs + nvis])
            w_ref, sz_ref = oracle.quantize_pack_rows_stored(xin, c.G, nbits, which)
            got_w = words[b, :, :nvis].reshape(-1, W)
            got_sz = sz[b, :, :nvis].reshape(-1, 2 * ng)
            if not np.array_equal(got_w, w_ref):
                bad = np.argwhere(got_w != w_ref)[:4]
                raise AssertionError(f"{which} codes differ b={b} at {bad.tolist()}")
            assert np.array_equal(got_sz[:, ng:], sz_ref[:, ng:]), f"{which} scales differ b={b}"
            assert np.array_equal(got_sz[:, :ng], sz_ref[:, :ng]), f"{which} zeros differ b={b}"
            n_rows += got_w.shape[0]
    return n_rows


def oracle_decode(c: Case, q_np, k_np, v_np, T: int, scale: float, prot_mask=None):
    """fp64 oracle over positions [0, T) of the given (possibly batch-sliced)
    inputs.  Returns (out, lse, max|V_hat| per (b, h))."""
    mask = c.mask() if prot_mask is None else prot_mask
    out, lse, kh, vh = oracle.decode_reference(q_np, np.ascontiguousarray(k_np[:, :, :T]),
                                               np.ascontiguousarray(v_np[:, :, :T]), c.vs, c.ve,
                                               mask, c.kb, c.vb, c.G, scale)
    vmax = np.abs(vh).max(axis=(2, 3))
    return out, lse, vmax


def check_decode(c: Case, out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref, lse_ref, vmax,
                 b_sel: Optional[Sequence[int]] = None) -> float:
    """Element-wise bar: |o_gpu - o_ref| <= TOL * max|V_hat| of (b, h).
    Returns the worst ratio err / (max|V_hat|)."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.cpu().numpy().astype(np.float64)
    b_sel = list(range(o.shape[0])) if b_sel is None else list(b_sel)
    o = o[b_sel]
    l = l[b_sel]
    g = c.H_q // c.H_kv
    worst = 0.0
    for hq in range(c.H_q):
        h = hq // g
        err = np.abs(o[:, hq] - out_ref[:, hq]).max(axis=1)
        ratio = err / vmax[:, h]
        worst = max(worst, float(ratio.max()))
        assert np.all(ratio <= TOL), f"hq={hq}: err/max|V| = {ratio.max():.3e}"
        lerr = np.abs(l[:, hq] - lse_ref[:, hq])
        assert np.all(lerr <= 2e-3 + 1e-4 * np.abs(lse_ref[:, hq])), f"lse hq={hq}: {lerr.max()}"
    assert np.all(np.isfinite(o))
    return worst
