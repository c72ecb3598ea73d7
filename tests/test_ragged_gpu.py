"""Ragged batches: kvq_decode_attention_ragged and kvq_decode_step_ragged,
where each sequence has its own length in a device array.

Bar: per sequence, the oracle over that sequence's own positions (outputs
within 4e-3 * max|V_hat|), inactive entries give zero outputs and lse -inf
and store nothing, and a batch whose lengths are all equal gives the same
bits as the uniform entry point (same plan, same arithmetic).
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
    ws[:256 + (4 * int(L.units) + 255) // 256 * 256] = 0  # status word and the fused step's counters
    return ws


def _q(c: Case, seed: int, dev):
    return synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(seed, 3), dev)
                         .view(c.B, c.H_q, c.D))


def _check_inactive(out, lse, b):
    assert torch.all(out[b].float() == 0), b
    assert torch.all(torch.isneginf(lse[b])), b


def _check_seq(c, out, lse, q, k, v, b, T_b):
    ref, lr, vmax = oracle_decode(c, bits(q[b:b + 1]), bits(k[b:b + 1]), bits(v[b:b + 1]), T_b, SCALE)
    check_decode(c, out, lse, ref, lr, vmax, b_sel=[b])


RAGGED = [
    # layout, T_max, per-sequence lengths (0 and T_max + 1: inactive)
    (Case(6, 28, 4, 700, 14, 640, 4, 2, 64, [0]), 700, [700, 660, 300, 7, 1, 0]),
    (Case(4, 32, 8, 1200, 32, 1200, 2, 2, 32, [3]), 900, [900, 33, 901, 517]),
    (Case(3, 16, 4, 400, 20, 390, 4, 4, 32, [1], konly=[2]), 400, [395, 150, 21]),
    (Case(5, 8, 8, 300, 30, 250, 8, 4, 128, []), 290, [-3, 290, 250, 31, 100]),
]


@pytest.mark.parametrize("ci", range(len(RAGGED)))
def test_ragged_decode_matches_oracle_per_sequence(cuda_dev, kvq, ci):
    c, T_max, lens = RAGGED[ci]
    L = c.layout()
    _, k, v = synth.random_case(1100 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    q = _q(c, 1110 + ci, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    sl = torch.tensor(lens, dtype=torch.int32, device=cuda_dev)
    out = torch.full((c.B, c.H_q, c.D), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    lse = torch.zeros((c.B, c.H_q), dtype=torch.float32, device=cuda_dev)
    ws = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=cuda_dev)
    kvq.decode_attention_ragged(L, cache, q, sl, T_max, out, SCALE, lse, ws)
    torch.cuda.synchronize()
    for b, T_b in enumerate(lens):
        if 1 <= T_b <= T_max:
            _check_seq(c, out, lse, q, k, v, b, T_b)
        else:
            _check_inactive(out, lse, b)


def test_ragged_decode_equal_lengths_is_the_uniform_call(cuda_dev, kvq):
    c = Case(2, 28, 4, 2000, 14, 1900, 4, 2, 64, [0])
    L = c.layout()
    _, k, v = synth.random_case(1150, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    q = _q(c, 1151, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    for T in (1950, 1000, 12):
        out_u, lse_u = decode(L, cache, q, T, SCALE)
        out_r = torch.empty_like(out_u)
        lse_r = torch.empty_like(lse_u)
        ws = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=cuda_dev)
        sl = torch.full((c.B,), T, dtype=torch.int32, device=cuda_dev)
        kvq.decode_attention_ragged(L, cache, q, sl, T, out_r, SCALE, lse_r, ws)
        torch.cuda.synchronize()
        assert torch.equal(out_u.view(torch.int16), out_r.view(torch.int16)), T
        assert torch.equal(lse_u, lse_r), T


def _step_rows(c: Case, seed: int, n: int, dev):
    k = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 1), dev)
                      .view(c.B, c.H_kv, n, c.D))
    v = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 2), dev)
                      .view(c.B, c.H_kv, n, c.D))
    return k, v


STEPS = [
    # layout, T_max, first step position per sequence (-1 and visual: inactive)
    (Case(5, 28, 4, 700, 14, 640, 4, 2, 64, [0], konly=[2]), 700, [650, 690, 5, -1, 100]),
    (Case(3, 32, 8, 1300, 32, 1232, 2, 2, 32, [3]), 1300, [1240, 10, 1290]),
    (Case(4, 40, 40, 200, 10, 150, 8, 8, 64, [1, 7]), 180, [160, 2, 175, 178]),
]


@pytest.mark.parametrize("ci", range(len(STEPS)))
def test_ragged_steps_match_oracle_per_sequence(cuda_dev, kvq, ci):
    c, T_max, first = STEPS[ci]
    n_steps = 3
    L = c.layout()
    _, k, v = synth.random_case(1200 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    ks, vs_ = _step_rows(c, 1210 + ci, n_steps, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    kf, vf = k.clone(), v.clone()  # what the cache must hold
    ws = _ws(L, cuda_dev)
    out = torch.empty((c.B, c.H_q, c.D), dtype=torch.bfloat16, device=cuda_dev)
    lse = torch.empty((c.B, c.H_q), dtype=torch.float32, device=cuda_dev)

    def active(t):
        return 0 <= t < T_max and not (c.vs <= t < c.ve)

    for i in range(n_steps):
        tn = [t + i if t >= 0 else t for t in first]
        t_dev = torch.tensor(tn, dtype=torch.int32, device=cuda_dev)
        q = _q(c, 1220 + 10 * ci + i, cuda_dev)
        kr, vr = ks[:, :, i].contiguous(), vs_[:, :, i].contiguous()
        kvq.decode_step_ragged(L, cache, q, kr, vr, t_dev, T_max, out, SCALE, lse, ws)
        torch.cuda.synchronize()
        for b, t in enumerate(tn):
            if active(t):
                kf[b, :, t] = kr[b]
                vf[b, :, t] = vr[b]
                _check_seq(c, out, lse, q, kf, vf, b, t + 1)
            else:
                _check_inactive(out, lse, b)
    # every sequence's cache rows: the step rows where active, untouched elsewhere
    for b in range(c.B):
        check_append(L, c, cache, bits(kf[b:b + 1]), bits(vf[b:b + 1]), c.T_cap, b_sel=[b])
    assert bool((ws[:(4 * int(L.units) + 255) // 256 * 256] == 0).all().item())


def test_ragged_step_equal_positions_is_the_uniform_step(cuda_dev, kvq):
    c = Case(2, 28, 4, 800, 14, 700, 4, 2, 64, [0])
    L = c.layout()
    _, k, v = synth.random_case(1300, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    ks, vs_ = _step_rows(c, 1301, 1, cuda_dev)
    kr, vr = ks[:, :, 0].contiguous(), vs_[:, :, 0].contiguous()
    q = _q(c, 1302, cuda_dev)
    t = 750
    caches = []
    outs = []
    for ragged in (False, True):
        cache = alloc_cache(L)
        append(L, cache, k, v, 0)
        ws = _ws(L, cuda_dev)
        out = torch.empty((c.B, c.H_q, c.D), dtype=torch.bfloat16, device=cuda_dev)
        lse = torch.empty((c.B, c.H_q), dtype=torch.float32, device=cuda_dev)
        if ragged:
            t_dev = torch.full((c.B,), t, dtype=torch.int32, device=cuda_dev)
            kvq.decode_step_ragged(L, cache, q, kr, vr, t_dev, t + 1, out, SCALE, lse, ws)
        else:
            kvq.decode_step(L, cache, q, kr, vr, t, out, SCALE, lse, ws)
        torch.cuda.synchronize()
        caches.append(cache)
        outs.append((out, lse))
    assert torch.equal(caches[0], caches[1])
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


def test_ragged_step_graph_advances_positions_on_device(cuda_dev, kvq):
    """A decode loop captured once: the graph runs the ragged step and then
    advances every sequence's position on the device; each replay is the
    next step (the host never sees the positions)."""
    c = Case(3, 28, 4, 900, 14, 800, 4, 2, 64, [0])
    L = c.layout()
    _, k, v = synth.random_case(1400, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    n_steps = 4
    ks, vs_ = _step_rows(c, 1401, n_steps, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    kf, vf = k.clone(), v.clone()
    first = [810, 850, 5]
    t_dev = torch.tensor(first, dtype=torch.int32, device=cuda_dev)
    q = _q(c, 1402, cuda_dev)
    kr = torch.zeros((c.B, c.H_kv, c.D), dtype=torch.bfloat16, device=cuda_dev)
    vr = torch.empty_like(kr)
    out = torch.empty((c.B, c.H_q, c.D), dtype=torch.bfloat16, device=cuda_dev)
    lse = torch.empty((c.B, c.H_q), dtype=torch.float32, device=cuda_dev)
    ws = _ws(L, cuda_dev)
    # one eager call on scratch copies first (per-kernel set-up happens outside the capture)
    kvq.decode_step_ragged(L, cache.clone(), q, kr, vr, t_dev.clone(), c.T_cap, out.clone(), SCALE,
                           lse.clone(), _ws(L, cuda_dev))
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kvq.decode_step_ragged(L, cache, q, kr, vr, t_dev, c.T_cap, out, SCALE, lse, ws, stream=s)
        t_dev.add_(1)
    torch.cuda.synchronize()
    assert t_dev.tolist() == first  # capturing ran nothing
    for i in range(n_steps):
        kr.copy_(ks[:, :, i])
        vr.copy_(vs_[:, :, i])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for b in range(c.B):
            t = first[b] + i
            kf[b, :, t] = ks[b, :, i]
            vf[b, :, t] = vs_[b, :, i]
            _check_seq(c, out, lse, q, kf, vf, b, t + 1)
    assert t_dev.tolist() == [t + n_steps for t in first]
    for b in range(c.B):
        check_append(L, c, cache, bits(kf[b:b + 1]), bits(vf[b:b + 1]), c.T_cap, b_sel=[b])
