"""Early cache-tile copies (kvq_set_cache_preload) against the CPU oracle and
against the same calls without them.

With preload on, a decode kernel copies its first cache tiles before the
previous kernel in the stream has finished.  These tests chain calls on one
stream with no host synchronisation in between, so that the previous kernel
is the one that wrote the rows being copied early: fused steps of two
layers interleaved, steps back to back on one cache (the step row of call t
is history for call t + 1, across a text-tile boundary), a bulk append
followed at once by a decode, and the same chain replayed as a CUDA graph.
Bar: outputs bit-identical to the calls without preload (same plan, same
arithmetic), and within 4e-3 * max|V_hat| of the fp64 oracle.
"""
import math

import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import synth
from gpu_helpers import Case, alloc_cache, append, bits, check_append, check_decode, oracle_decode

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)
HEAD = 256  # workspace head before the arrival counters


@pytest.fixture
def preload():
    """Turns preload on for this host thread and back off afterwards."""
    kvq.set_cache_preload(True)
    try:
        yield
    finally:
        kvq.set_cache_preload(False)


def _ws(L, dev):
    ws = torch.full((int(L.workspace_bytes),), 0x5A, dtype=torch.uint8, device=dev)
    ws[:HEAD + (4 * int(L.units) + 255) // 256 * 256] = 0
    return ws


def _rows(c: Case, seed: int, n: int, dev):
    k = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 1), dev)
                      .view(c.B, c.H_kv, n, c.D))
    v = synth.to_bf16(synth.normal(c.B * c.H_kv * n * c.D, synth.stream_key(seed, 2), dev)
                      .view(c.B, c.H_kv, n, c.D))
    return k, v


def _qs(c: Case, seed: int, n: int, dev):
    return [synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(seed, 100 + i), dev)
                          .view(c.B, c.H_q, c.D)) for i in range(n)]


class _Layer:
    """One layer's cache, history and step rows."""

    def __init__(self, c: Case, seed: int, hist: int, n_steps: int, dev):
        self.c, self.hist = c, hist
        self.L = c.layout()
        _, k, v = synth.random_case(seed, c.B, c.H_q, c.H_kv, c.D, c.T_cap, dev)
        self.k, self.v = k[:, :, :hist].contiguous(), v[:, :, :hist].contiguous()
        self.ks, self.vs = _rows(c, seed + 1, n_steps, dev)
        self.qs = _qs(c, seed + 2, n_steps, dev)
        self.cache = alloc_cache(self.L)
        append(self.L, self.cache, self.k, self.v, 0)
        self.ws = _ws(self.L, dev)
        self.outs = [torch.empty((c.B, c.H_q, c.D), dtype=torch.bfloat16, device=dev) for _ in range(n_steps)]
        self.lses = [torch.empty((c.B, c.H_q), dtype=torch.float32, device=dev) for _ in range(n_steps)]

    def step(self, i, stream=None):
        kvq.decode_step(self.L, self.cache, self.qs[i], self.ks[:, :, i].contiguous(),
                        self.vs[:, :, i].contiguous(), self.hist + i, self.outs[i], SCALE, self.lses[i],
                        self.ws, stream=stream)

    def check(self, n_steps):
        c = self.c
        for i in range(n_steps):
            t = self.hist + i
            kf = torch.cat([self.k, self.ks[:, :, :i + 1]], 2)
            vf = torch.cat([self.v, self.vs[:, :, :i + 1]], 2)
            ref, lr, vmax = oracle_decode(c, bits(self.qs[i]), bits(kf), bits(vf), t + 1, SCALE)
            check_decode(c, self.outs[i], self.lses[i], ref, lr, vmax)
        kf = torch.cat([self.k, self.ks[:, :, :n_steps]], 2)
        vf = torch.cat([self.v, self.vs[:, :, :n_steps]], 2)
        check_append(self.L, c, self.cache, bits(kf), bits(vf), self.hist + n_steps)


def _run_chain(cases, n_steps, dev, seed):
    """Steps of every layer interleaved (layer 0 step i, layer 1 step i, ...)
    on the current stream, no host synchronisation until the end."""
    layers = [_Layer(c, seed + 10 * j, hist, n_steps, dev) for j, (c, hist) in enumerate(cases)]
    torch.cuda.synchronize()
    for i in range(n_steps):
        for ly in layers:
            ly.step(i)
    torch.cuda.synchronize()
    return layers


# (Case, history length): the history ends 3 rows before a 64-row text-tile
# boundary after the visual span, so the steps' rows cross it.
CHAIN = [
    (Case(1, 28, 4, 760, 14, 640, 4, 2, 64, [0]), 640 + 61),   # LLaVA-OV heads (cluster mode)
    (Case(3, 16, 4, 520, 20, 400, 2, 4, 32, [1]), 400 + 61),   # B = 3, g = 4
]


@pytest.mark.parametrize("ci", range(len(CHAIN)))
def test_preload_steps_back_to_back(cuda_dev, kvq, preload, ci):
    """One layer, steps t, t + 1, ... with nothing in between: each step's
    rows are history for the next call, which copies tiles early."""
    n = 6
    on = _run_chain([CHAIN[ci]], n, cuda_dev, 3000 + 100 * ci)[0]
    on.check(n)
    kvq.set_cache_preload(False)
    off = _run_chain([CHAIN[ci]], n, cuda_dev, 3000 + 100 * ci)[0]
    for i in range(n):
        assert torch.equal(on.outs[i].view(torch.int16), off.outs[i].view(torch.int16)), (ci, i)
        assert torch.equal(on.lses[i], off.lses[i]), (ci, i)
    assert torch.equal(on.cache, off.cache)


def test_preload_two_layers_interleaved(cuda_dev, kvq, preload):
    """Two layers' steps interleaved (the decode of a model): each call's
    previous kernel writes the other layer's cache."""
    n = 5
    layers = _run_chain(CHAIN, n, cuda_dev, 3500)
    for ly in layers:
        ly.check(n)


def test_preload_append_then_decode(cuda_dev, kvq, preload):
    """A bulk append (two calls) followed at once by a decode over its rows."""
    for ci, c in enumerate([Case(1, 28, 4, 900, 14, 880, 4, 2, 64, [0]),
                            Case(2, 32, 8, 700, 10, 650, 2, 2, 32, [3], konly=[5])]):
        L = c.layout()
        _, k, v = synth.random_case(3600 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
        q = _qs(c, 3610 + ci, 1, cuda_dev)[0]
        cache = alloc_cache(L)
        ws = torch.zeros((int(L.workspace_bytes),), dtype=torch.uint8, device=cuda_dev)
        out = torch.empty((c.B, c.H_q, c.D), dtype=torch.bfloat16, device=cuda_dev)
        lse = torch.empty((c.B, c.H_q), dtype=torch.float32, device=cuda_dev)
        torch.cuda.synchronize()
        half = c.T_cap // 2
        append(L, cache, k[:, :, :half].contiguous(), v[:, :, :half].contiguous(), 0)
        append(L, cache, k[:, :, half:].contiguous(), v[:, :, half:].contiguous(), half)
        kvq.decode_attention(L, cache, q, c.T_cap, out, SCALE, lse, ws)
        torch.cuda.synchronize()
        ref, lr, vmax = oracle_decode(c, bits(q), bits(k), bits(v), c.T_cap, SCALE)
        check_decode(c, out, lse, ref, lr, vmax)


def test_preload_graph_replay(cuda_dev, kvq, preload):
    """Two layers' steps captured in a CUDA graph (programmatic edges between
    the kernels) and replayed: bit-identical to the eager calls without
    preload every replay."""
    n = 3
    ref_layers = None
    kvq.set_cache_preload(False)
    ref_layers = _run_chain(CHAIN, n, cuda_dev, 3700)
    kvq.set_cache_preload(True)
    layers = [_Layer(c, 3700 + 10 * j, hist, n, cuda_dev) for j, (c, hist) in enumerate(CHAIN)]
    base = [ly.cache.clone() for ly in layers]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(n):
            for ly in layers:
                ly.step(i, stream=s)
    for _ in range(3):
        for ly, b0 in zip(layers, base):
            ly.cache.copy_(b0)
            for o in ly.outs:
                o.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for ly, rl in zip(layers, ref_layers):
            for i in range(n):
                assert torch.equal(ly.outs[i].view(torch.int16), rl.outs[i].view(torch.int16)), i
                assert torch.equal(ly.lses[i], rl.lses[i]), i
            assert torch.equal(ly.cache, rl.cache)
