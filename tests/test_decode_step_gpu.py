"""kvq_decode_step (the fused decode step) against the CPU oracle and against
the two-call path it fuses (kvq_quantize_append of the step's row, then
kvq_decode_attention over [0, t_new]).

Bar: the step's bf16 row lands in the cache bit-identically; outputs within
4e-3 * max|V_hat| of the fp64 oracle; and, since both paths use the same
work plan and arithmetic, out and lse bit-identical to the two-call path.
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


def _ws(L, dev):
    ws = torch.full((int(L.workspace_bytes),), 0x5A, dtype=torch.uint8, device=dev)
    ws[:4] = 0  # the barrier's arrival counter
    return ws


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
    gen = int(ws[4:8].view(torch.int32).item())
    for i in range(n_steps):
        t = hist + i
        q = _q(c, 720 + ci, i, cuda_dev)
        kr, vr = ks[:, :, i].contiguous(), vs_[:, :, i].contiguous()
        out_f, lse_f = _step(L, fused, q, kr, vr, t, ws)
        kvq.quantize_append(L, split, kr.unsqueeze(2), vr.unsqueeze(2), t)
        out_s, lse_s = decode(L, split, q, t + 1)
        torch.cuda.synchronize()
        assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), (ci, i)
        assert torch.equal(lse_f, lse_s), (ci, i)
        kf = torch.cat([k, ks[:, :, :i + 1]], 2)
        vf = torch.cat([v, vs_[:, :, :i + 1]], 2)
        ref, lr, vmax = oracle_decode(c, bits(q), bits(kf), bits(vf), t + 1, SCALE)
        check_decode(c, out_f, lse_f, ref, lr, vmax)
    assert torch.equal(fused, split)  # same cache bytes after the steps
    kf, vf = torch.cat([k, ks], 2), torch.cat([v, vs_], 2)
    check_append(L, c, fused, bits(kf), bits(vf), c.T_cap)
    hdr = ws[:8].view(torch.int32).cpu().tolist()
    assert hdr[0] == 0                     # arrival counter left at zero
    assert (hdr[1] - gen) % (1 << 32) == n_steps  # one barrier generation per call


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
    replayed CUDA graph (the workspace counter survives replays)."""
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
    assert int(ws[:4].view(torch.int32).item()) == 0
