"""Failure detection of the decode kernels without a GPU fault.

Every wait of the kernels is bounded; a wait that gives up, or an arrival
counter of the fused step found non-zero at entry, sets a KVQ_STATUS_* bit in
the workspace's status word and turns the affected output rows into NaN, and
the call still returns.  These tests make that happen on purpose in the
host-visible state only -- they seed the workspace's counters (a workspace
that was not zeroed, or that overlapping calls share) and shorten the wait
limits -- and check the status word, the NaN rows, and that a later call on
a re-zeroed workspace is correct again.
"""
import math

import numpy as np
import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import synth
from gpu_helpers import TOL, Case, alloc_cache, append, bits, oracle_decode

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)
HEAD = 256

# 16 units of 64 text positions each: more units than 16-CTA clusters fit on
# the GPU at once, so the fused step runs in global mode (workspace partials
# and per-unit arrival counters); each unit's cost (64 positions x 768) is 6
# chunks of the plan's 8 Ki minimum, so every unit is split over n = 6 CTAs
# and combined by its last min(6, g = 4) arrivals.
CASE = Case(4, 16, 4, 64, 0, 0, 4, 2, 64, [])
N_CHUNKS = 6
N_COMB = 4


def _setup(dev):
    c = CASE
    L = c.layout()
    _, k, v = synth.random_case(900, c.B, c.H_q, c.H_kv, c.D, c.T_cap, dev)
    cache = alloc_cache(L)
    append(L, cache, k[:, :, :c.T_cap - 1].contiguous(), v[:, :, :c.T_cap - 1].contiguous(), 0)
    q = synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(901, 1), dev).view(c.B, c.H_q, c.D))
    ks = k[:, :, c.T_cap - 1:].contiguous()
    vs = v[:, :, c.T_cap - 1:].contiguous()
    return L, cache, q, k, v, ks, vs


def _ws(L, dev, seed_counters=None):
    ws = torch.zeros(int(L.workspace_bytes), dtype=torch.uint8, device=dev)
    if seed_counters is not None:
        cnt = ws[HEAD:HEAD + 4 * int(L.units)].view(torch.int32)
        cnt.fill_(seed_counters)
    return ws


def _step(L, cache, q, ks, vs, ws):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    kvq.decode_step(L, cache, q, ks, vs, CASE.T_cap - 1, out, SCALE, lse, ws)
    return out, lse


def _check_correct(L, q, k, v, out):
    ref, _, vmax = oracle_decode(CASE, bits(q), bits(k), bits(v), CASE.T_cap, SCALE)
    got = out.float().cpu().numpy().astype(np.float64)
    g = CASE.H_q // CASE.H_kv
    for hq in range(CASE.H_q):
        assert np.all(np.abs(got[:, hq] - ref[:, hq]).max(axis=1) <= TOL * vmax[:, hq // g]), hq


def test_corrupt_counter_sets_status_and_nan_rows(cuda_dev):
    """Counters far above the unit's chunk count: every arrival sees the
    corruption, reports KVQ_STATUS_COUNTER and writes NaN rows."""
    L, cache, q, k, v, ks, vs = _setup(cuda_dev)
    assert L.units == 16
    ws = _ws(L, cuda_dev, seed_counters=1 << 30)
    out, lse = _step(L, cache, q, ks, vs, ws)
    torch.cuda.synchronize()
    st = kvq.workspace_status(ws)
    assert st & kvq.STATUS_COUNTER
    assert torch.isnan(out.float()).all()
    assert torch.isnan(lse).all()
    # a re-zeroed workspace gives the right answer and a clean status
    ws.zero_()
    out, lse = _step(L, cache, q, ks, vs, ws)
    torch.cuda.synchronize()
    assert kvq.workspace_status(ws) == 0
    _check_correct(L, q, k, v, out)


def test_peer_wait_gives_up(cuda_dev):
    """Counters seeded at n - 1: the first arrival of each unit takes itself
    for the last, combines row n_comb - 1 from incomplete partials and
    resets the counter.  Whoever arrives before that reset finds the counter
    at n or more (KVQ_STATUS_COUNTER: NaN into every row of the unit);
    whoever arrives after it with a combining role waits for a reset that
    never comes and, with a short wait limit, gives up
    (KVQ_STATUS_PEER_WAIT: NaN into its row).  Which of the two happens
    depends on the arrival order, but in every order rows 0 .. n_comb - 2 of
    every unit end up NaN, the status word says so, and the call returns."""
    L, cache, q, k, v, ks, vs = _setup(cuda_dev)
    ws = _ws(L, cuda_dev, seed_counters=N_CHUNKS - 1)
    kvq.set_wait_limits(0, 2000)
    try:
        out, _ = _step(L, cache, q, ks, vs, ws)
        torch.cuda.synchronize()
    finally:
        kvq.set_wait_limits(0, 0)
    st = kvq.workspace_status(ws)
    assert st & (kvq.STATUS_PEER_WAIT | kvq.STATUS_COUNTER)
    assert not st & kvq.STATUS_TILE_WAIT
    g = CASE.H_q // CASE.H_kv
    o = out.float().view(CASE.B, CASE.H_kv, g, CASE.D)
    assert torch.isnan(o[:, :, :N_COMB - 1]).all()
    # recovery after zeroing the workspace
    ws.zero_()
    out, _ = _step(L, cache, q, ks, vs, ws)
    torch.cuda.synchronize()
    assert kvq.workspace_status(ws) == 0
    _check_correct(L, q, k, v, out)


def test_status_clean_on_normal_calls(cuda_dev):
    """Normal calls leave the status word zero (fused step and two-call
    decode; cluster and global mode)."""
    for c in (CASE, Case(1, 28, 4, 300, 14, 290, 4, 2, 64, [0])):
        L = c.layout()
        _, k, v = synth.random_case(910, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
        cache = alloc_cache(L)
        append(L, cache, k, v, 0)
        q = synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(911, 1), cuda_dev)
                          .view(c.B, c.H_q, c.D))
        ws = torch.zeros(int(L.workspace_bytes), dtype=torch.uint8, device=cuda_dev)
        out = torch.empty_like(q)
        kvq.decode_attention(L, cache, q, c.T_cap, out, SCALE, None, ws)
        torch.cuda.synchronize()
        assert kvq.workspace_status(ws) == 0
