"""kvq_decode_step (the fused decode step) against the CPU oracle and against
the two-call path it fuses (kvq_quantize_append of the step's row, then
kvq_decode_attention over [0, t_new]).

Bar: the step's bf16 row lands in the cache bit-identically; outputs within
4e-3 * max|V_hat| of the fp64 oracle.  Both paths use the same work plan and
split arithmetic and differ only in the summation order of the cross-split
combine, so they agree to a few fp32 rounding steps: at most one bf16 ulp
of the output apart (asserted as 2^-7 |o| + 1e-5 max|V_hat|).
"""
import math

import numpy as np
import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import synth
from gpu_helpers import Case, alloc_cache, append, bits, check_append, check_decode, decode, oracle_decode

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


HEAD = 256  # workspace head: the status word, then padding


def _cnt_bytes(L):
    return (4 * int(L.units) + 255) // 256 * 256


def _ws(L, dev):
    ws = torch.full((int(L.workspace_bytes),), 0x5A, dtype=torch.uint8, device=dev)
    ws[:HEAD + _cnt_bytes(L)] = 0  # status word and the per-unit arrival counters
    return ws


def _counters_zero(L, ws) -> bool:
    return bool((ws[HEAD:HEAD + _cnt_bytes(L)] == 0).all().item())


def _step(L, cache, q, ks, vs, t_new, ws):
    B, Hq, D = q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    kvq.decode_step(L, cache, q, ks, vs, t_new, out, SCALE, lse, ws)
    return out, lse


def _rows(c: Case, seed: int, n: int, dev):
    """n step rows of K and V, [B, H_kv, n, D] bf16 each."""
    k = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 1), dev)
                      .view(c.B, c.H_kv, n, c.D))
    v = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 2), dev)
                      .view(c.B, c.H_kv, n, c.D))
    return k, v


def _q(c: Case, seed: int, i: int, dev):
    return synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(seed, 100 + i), dev)
                         .view(c.B, c.H_q, c.D))


CASES = [
    # B, H_q, H_kv, T_cap, vs, ve, kb, vb, G, protected
    Case(1, 28, 4, 660, 14, 640, 4, 2, 64, [0]),        # LLaVA-OV-like heads, short history
    Case(2, 32, 2, 400, 5, 300, 8, 4, 32, [1]),         # g = 16: two head chunks per KV head
    Case(3, 8, 8, 300, 30, 250, 2, 8, 128, []),         # g = 1, B = 3
    Case(1, 40, 40, 320, 10, 290, 16, 16, 32, [3, 7]),  # MHA, bf16 "packed" segments
    Case(2, 28, 4, 700, 14, 690, 4, 2, 64, [2], konly=[0]),  # K-only protected head
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_steps_match_oracle_and_two_call_path(cuda_dev, kvq, ci):
    c = CASES[ci]
    n_steps = 4
    L = c.layout()
    hist = c.T_cap - n_steps
    _, k, v = synth.random_case(700 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    k, v = k[:, :, :hist].contiguous(), v[:, :, :hist].contiguous()
    ks, vs_ = _rows(c, 710 + ci, n_steps, cuda_dev)
    fused = alloc_cache(L)
    split = alloc_cache(L)
    append(L, fused, k, v, 0)
    append(L, split, k, v, 0)
    ws = _ws(L, cuda_dev)
    for i in range(n_steps):
        t = hist + i
        q = _q(c, 720 + ci, i, cuda_dev)
        kr, vr = ks[:, :, i].contiguous(), vs_[:, :, i].contiguous()
        out_f, lse_f = _step(L, fused, q, kr, vr, t, ws)
        kvq.quantize_append(L, split, kr.unsqueeze(2), vr.unsqueeze(2), t)
        out_s, lse_s = decode(L, split, q, t + 1)
        torch.cuda.synchronize()
        kf = torch.cat([k, ks[:, :, :i + 1]], 2)
        vf = torch.cat([v, vs_[:, :, :i + 1]], 2)
        ref, lr, vmax = oracle_decode(c, bits(q), bits(kf), bits(vf), t + 1, SCALE)
        check_decode(c, out_f, lse_f, ref, lr, vmax)
        g = c.H_q // c.H_kv
        a = out_f.float().cpu().numpy()
        b = out_s.float().cpu().numpy()
        for hq in range(c.H_q):
            bar = 2.0 ** -7 * np.maximum(np.abs(a[:, hq]), np.abs(b[:, hq])) + \
                1e-5 * vmax[:, hq // g][:, None]
            assert np.all(np.abs(a[:, hq] - b[:, hq]) <= bar), (ci, i, hq)
        assert np.allclose(lse_f.cpu().numpy(), lse_s.cpu().numpy(), rtol=0, atol=1e-4), (ci, i)
    assert torch.equal(fused, split)  # same cache bytes after the steps
    kf, vf = torch.cat([k, ks], 2), torch.cat([v, vs_], 2)
    check_append(L, c, fused, bits(kf), bits(vf), c.T_cap)
    assert _counters_zero(L, ws)  # every call leaves the arrival counters at zero


def test_step_before_visual_span(cuda_dev, kvq):
    """Steps whose position lies in the text prefix (T <= vis_start): no
    visual position is attended yet."""
    c = Case(2, 16, 4, 200, 40, 180, 4, 4, 32, [2])
    L = c.layout()
    ks, vs_ = _rows(c, 800, 40, cuda_dev)
    fused = alloc_cache(L)
    ws = _ws(L, cuda_dev)
    for t in (0, 1, 17, 39):
        if t:
            append(L, fused, ks[:, :, :t].contiguous(), vs_[:, :, :t].contiguous(), 0)
        q = _q(c, 801, t, cuda_dev)
        out, lse = _step(L, fused, q, ks[:, :, t].contiguous(), vs_[:, :, t].contiguous(), t, ws)
        torch.cuda.synchronize()
        ref, lr, vmax = oracle_decode(c, bits(q), bits(ks), bits(vs_), t + 1, SCALE)
        check_decode(c, out, lse, ref, lr, vmax)
        check_append(L, c, fused, bits(ks), bits(vs_), t + 1)


def test_step_at_capacity_and_in_graph(cuda_dev, kvq):
    """The last slot of the cache (t_new = T_cap - 1), run eagerly and as a
    replayed CUDA graph (the arrival counters return to zero every call)."""
    c = Case(1, 28, 4, 1000, 14, 990, 4, 2, 64, [0])
    L = c.layout()
    _, k, v = synth.random_case(900, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    t = c.T_cap - 1
    cache = alloc_cache(L)
    append(L, cache, k[:, :, :t].contiguous(), v[:, :, :t].contiguous(), 0)
    kr, vr = k[:, :, t].contiguous(), v[:, :, t].contiguous()
    q = _q(c, 901, 0, cuda_dev)
    ws = _ws(L, cuda_dev)
    out0, lse0 = _step(L, cache, q, kr, vr, t, ws)
    torch.cuda.synchronize()
    ref, lr, vmax = oracle_decode(c, bits(q), bits(k), bits(v), c.T_cap, SCALE)
    check_decode(c, out0, lse0, ref, lr, vmax)
    out = torch.empty_like(out0)
    lse = torch.empty_like(lse0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kvq.decode_step(L, cache, q, kr, vr, t, out, SCALE, lse, ws, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)
    assert _counters_zero(L, ws)


def test_single_unit_many_chunks_and_many_units_few_chunks(cuda_dev, kvq):
    """Both cut regimes: one unit split over many CTAs (B = 1, H_kv = 1,
    long history), and more units than CTAs (B = 24, MHA: units are
    combined inside the CTA that holds them)."""
    for ci, c in enumerate([Case(1, 8, 1, 20000, 16, 19990, 2, 2, 32, []),
                            Case(24, 48, 48, 96, 8, 90, 4, 4, 64, [5, 9])]):
        L = c.layout()
        t = c.T_cap - 1
        _, k, v = synth.random_case(950 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
        cache = alloc_cache(L)
        append(L, cache, k[:, :, :t].contiguous(), v[:, :, :t].contiguous(), 0)
        q = _q(c, 960 + ci, 0, cuda_dev)
        ws = _ws(L, cuda_dev)
        out, lse = _step(L, cache, q, k[:, :, t].contiguous(), v[:, :, t].contiguous(), t, ws)
        torch.cuda.synchronize()
        ref, lr, vmax = oracle_decode(c, bits(q), bits(k), bits(v), c.T_cap, SCALE)
        check_decode(c, out, lse, ref, lr, vmax)
        assert _counters_zero(L, ws)
