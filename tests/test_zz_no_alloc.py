"""kvq_decode_attention_static_ws: decoding for callers that may not allocate.

Some users of this library cannot call cudaMalloc (a plug-in whose host
framework owns all device memory, a serving loop that must never allocate).
The static-workspace entry point gives them the same decode without a
caller-provided workspace: its scratch is a fixed array inside the library.
These tests call it through the C ABI and check it against the regular entry
point (which takes a workspace) on two calls in a row, and check that an
over-large layout is refused before any CUDA work.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq_mod
import synth
from gpu_helpers import TOL, Case, alloc_cache, append, bits, decode, oracle_decode

SCALE = 1.0 / math.sqrt(128)


def _static_decode(L, cache, q, T):
    B, Hq, D = q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    kvq_mod.decode_attention_static_ws(L, cache, q, T, out, SCALE, lse)
    return out, lse


@pytest.mark.gpu
def test_static_workspace_matches_workspace_entry_point(cuda_dev, kvq):
    cases = [
        Case(1, 28, 4, 700, 14, 690, 4, 2, 64, [0]),     # GQA 7, one protected head (cluster merge)
        Case(3, 16, 8, 300, 20, 280, 8, 4, 32, [1, 6]),  # several sequences and units (workspace partials)
    ]
    for i, c in enumerate(cases):
        _, k, v = synth.random_case(500 + i, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
        L = c.layout()
        assert L.workspace_bytes <= kvq_mod.STATIC_WS_BYTES
        cache = alloc_cache(L)
        append(L, cache, k, v, 0)
        # two calls in a row, with different queries and lengths; the array
        # keeps the first call's partials when the second one starts
        for call, T in enumerate((c.T_cap, c.T_cap - 37)):
            q = synth.to_bf16(synth.normal(c.B * c.H_q * c.D, synth.stream_key(600 + i, call),
                                           cuda_dev).view(c.B, c.H_q, c.D))
            out_ref, lse_ref = decode(L, cache, q, T, SCALE)
            out_s, lse_s = _static_decode(L, cache, q, T)
            torch.cuda.synchronize()
            ref, lr, vmax = oracle_decode(c, bits(q), bits(k), bits(v), T, SCALE)
            # same plan and kernels as the workspace entry point, only the
            # scratch differs: the results must be identical bit for bit (a
            # stale partial read from the shared array would show here)
            assert torch.equal(out_s, out_ref), (i, call)
            assert torch.equal(lse_s, lse_ref), (i, call)
            a = out_s.float().cpu().numpy().astype(np.float64)
            g = c.H_q // c.H_kv
            for hq in range(c.H_q):
                bar = TOL * vmax[:, hq // g]
                assert np.all(np.abs(a[:, hq] - ref[:, hq]).max(axis=1) <= bar), (i, call, hq)


def test_static_workspace_refuses_oversize_layout():
    """A layout whose scratch exceeds the fixed array is refused with
    KVQ_ERR_CAPACITY before any CUDA call (runs without a GPU)."""
    kvq_mod.load()
    L = kvq_mod.cache_layout(32, 128, 128, 128, 64, 8, 56, 4, 4, 32, [])
    assert L.workspace_bytes > kvq_mod.STATIC_WS_BYTES
    fake = 1 << 40  # never dereferenced: the call must return first
    with pytest.raises(kvq_mod.KvqError) as e:
        kvq_mod.load().kvq_decode_attention_static_ws  # symbol present
        kvq_mod.decode_attention_static_ws(L, fake, fake, 64, fake, SCALE, None, stream=0)
    assert e.value.status == 3


def test_static_workspace_capacity_boundary():
    """The fixed array holds the scratch of layouts up to 3007 units
    (B * H_kv * ceil(g/8)); one unit more is refused before any CUDA call
    (runs without a GPU)."""
    kvq_mod.load()
    fits = kvq_mod.cache_layout(31, 97, 97, 128, 64, 8, 56, 4, 4, 32, [])
    over = kvq_mod.cache_layout(32, 94, 94, 128, 64, 8, 56, 4, 4, 32, [])
    assert (fits.units, over.units) == (3007, 3008)
    assert fits.workspace_bytes == kvq_mod.STATIC_WS_BYTES
    assert over.workspace_bytes > kvq_mod.STATIC_WS_BYTES
    fake = 1 << 40
    with pytest.raises(kvq_mod.KvqError) as e:
        kvq_mod.decode_attention_static_ws(over, fake, fake, 64, fake, SCALE, None, stream=0)
    assert e.value.status == 3
