"""kvq_sensitivity_probe against the CPU oracle's sensitivity reference.

Both sides are fp64 and differ only in summation order (the kernel uses the
one-pass identity D_KL(p || p_hat) = sum p (s - s_hat) - lse + lse_hat, the
oracle sums p log(p / p_hat) term by term), so they agree to a few hundred
fp64 ulps of the O(10) log-sum-exp values: |gpu - ref| <= 1e-11 + 1e-9 |ref|.
The softmax scale is the fp32 value the entry point takes, given to the
oracle as that same value.
Where the exact and the read cache coincide (V-only quantisation for
kl_attn, nothing quantised for all three) the kernel's two sides run the
same arithmetic, so the result is exactly 0.
"""
import math

import numpy as np
import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import oracle
import synth
from gpu_helpers import Case, alloc_cache, append, bits

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)
SCALE32 = float(np.float32(SCALE))  # the fp32 value the entry point receives


def _readout(seed, n_out, dev):
    g = np.random.default_rng(seed).standard_normal((n_out, 128)).astype(np.float32)
    return torch.from_numpy(g).to(dev)


def _probe(L, cache, q, k, v, T, R):
    B, Hq, _ = q.shape
    res = torch.full((B, Hq, 3), float("nan"), dtype=torch.float64, device=q.device)
    ws = torch.full((max(1, kvq.probe_workspace_bytes(L, T)),), 0x7F, dtype=torch.uint8, device=q.device)
    kvq.sensitivity_probe(L, cache, q, k, v, T, R, res, SCALE, ws)
    torch.cuda.synchronize()
    return res.cpu().numpy()


def _ref(c: Case, q, k, v, T, R):
    return oracle.sensitivity_reference(bits(q), np.ascontiguousarray(bits(k)[:, :, :T]),
                                        np.ascontiguousarray(bits(v)[:, :, :T]), c.vs, c.ve, c.mask(),
                                        c.kb, c.vb, c.G, SCALE32, R.cpu().numpy())


def _close(got, ref):
    err = np.abs(got - ref)
    bar = 1e-11 + 1e-9 * np.abs(ref)
    assert np.all(err <= bar), f"worst {np.max(err / bar):.3g} x bar at {np.unravel_index(np.argmax(err / bar), err.shape)}"


CASES = [
    # layout (bits of the probed cache), T
    (Case(1, 28, 4, 700, 14, 640, 4, 16, 64, [0]), 700),    # K quantised, V raw
    (Case(1, 28, 4, 700, 14, 640, 16, 4, 64, [0]), 700),    # V quantised, K raw
    (Case(2, 32, 8, 600, 32, 600, 2, 2, 32, [3]), 450),     # both, T inside the visual range
    (Case(3, 16, 4, 300, 20, 290, 8, 4, 128, [1], konly=[2]), 297),
    (Case(2, 8, 8, 200, 10, 150, 2, 8, 32, []), 180),       # MHA
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_probe_matches_oracle(cuda_dev, kvq, ci):
    c, T = CASES[ci]
    L = c.layout()
    q, k, v = synth.random_case(1500 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    R = _readout(1510 + ci, 257, cuda_dev)
    got = _probe(L, cache, q, k, v, T, R)
    ref = _ref(c, q, k, v, T, R)
    _close(got, ref)
    if c.kb == 16:  # K read as stored: the softmax weights cannot move
        assert np.all(got[..., 0] == 0.0)
    assert np.all(got >= 0)


def test_probe_nothing_quantised_is_exactly_zero(cuda_dev, kvq):
    c = Case(2, 8, 2, 300, 20, 280, 16, 16, 32, [])
    L = c.layout()
    q, k, v = synth.random_case(1550, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    got = _probe(L, cache, q, k, v, 300, _readout(1551, 64, cuda_dev))
    assert np.array_equal(got, np.zeros_like(got))


def test_probe_strided_rows_and_single_position(cuda_dev, kvq):
    """Raw rows passed as a strided view (a slice of a longer buffer), and
    T = 1 (one text position: everything exactly 0)."""
    c = Case(1, 4, 2, 400, 5, 380, 2, 2, 64, [])
    L = c.layout()
    q, k, v = synth.random_case(1560, c.B, c.H_q, c.H_kv, c.D, c.T_cap + 40, cuda_dev)
    k, v = k[:, :, :c.T_cap], v[:, :, :c.T_cap]  # non-contiguous views
    cache = alloc_cache(L)
    append(L, cache, k.contiguous(), v.contiguous(), 0)
    R = _readout(1561, 100, cuda_dev)
    for T in (400, 1):
        got = _probe(L, cache, q, k, v, T, R)
        ref = _ref(c, q, k, v, T, R)
        _close(got, ref)
    assert np.array_equal(got, np.zeros_like(got))  # T = 1
