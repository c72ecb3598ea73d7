"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: packed codes, scales and zeros bit-exact, bf16 rows bit-identical;
attention outputs within 4e-3 * max|V_hat| of the fp64 oracle (per (b, h)),
lse within 2e-3 + 1e-4 |lse|.
"""
import math

import numpy as np
import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import synth
from gpu_helpers import (Case, alloc_cache, append, bits, case_of, check_append, check_decode,
                         decode, oracle_decode)

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


def _run_full(c: Case, q, k, v, T, check_bits=True, b_sel=None):
    """Build the cache from k/v (all T_cap positions appended in one call),
    decode, compare.  q/k/v are device tensors."""
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    out, lse = decode(L, cache, q, T)
    torch.cuda.synchronize()
    sel = list(range(c.B)) if b_sel is None else list(b_sel)
    k_np, v_np, q_np = bits(k[sel]), bits(v[sel]), bits(q[sel])
    n = check_append(L, c, cache, k_np, v_np, c.T_cap, sel) if check_bits else 0
    ref, lse_ref, vmax = oracle_decode(c, q_np, k_np, v_np, T, SCALE)
    worst = check_decode(c, out[sel], lse[sel], ref, lse_ref, vmax)
    return n, worst


def test_tiny(cuda_dev, kvq):
    w = synth.workload("tiny")
    c = case_of(w, 0)
    k = synth.make_kv(w, 0, "k", cuda_dev)
    v = synth.make_kv(w, 0, "v", cuda_dev)
    q = synth.make_q(w, 0, device=cuda_dev)
    n, worst = _run_full(c, q, k, v, w.T)
    assert n == 2 * 242  # K and V, one unprotected head
    print(f"tiny: worst err/max|V| = {worst:.2e}")


def test_tiny_decode_step_appends_current_token(cuda_dev, kvq):
    """A decode step: history appended once, then the step's own K/V is
    appended as a text position and attended together with the history."""
    w = synth.workload("tiny")
    c = case_of(w, 0, extra=1)
    L = c.layout()
    k = synth.make_kv(w, 0, "k", cuda_dev)
    v = synth.make_kv(w, 0, "v", cuda_dev)
    ks = synth.make_step_kv(w, 0, "k", 0, cuda_dev)
    vs_ = synth.make_step_kv(w, 0, "v", 0, cuda_dev)
    q = synth.make_q(w, 0, device=cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    append(L, cache, ks, vs_, w.T)
    out, lse = decode(L, cache, q, w.T + 1)
    torch.cuda.synchronize()
    kf, vf = torch.cat([k, ks], 2), torch.cat([v, vs_], 2)
    check_append(L, c, cache, bits(kf), bits(vf), w.T + 1)
    ref, lr, vmax = oracle_decode(c, bits(q), bits(kf), bits(vf), w.T + 1, SCALE)
    check_decode(c, out, lse, ref, lr, vmax)


@pytest.mark.parametrize("layer", [0, 27])
def test_llava_ov_7b_layer(cuda_dev, kvq, layer):
    w = synth.workload("llava_ov_7b")
    c = case_of(w, layer)
    k = synth.make_kv(w, layer, "k", cuda_dev)
    v = synth.make_kv(w, layer, "v", cuda_dev)
    q = synth.make_q(w, layer, device=cuda_dev)
    n, worst = _run_full(c, q, k, v, w.T)
    assert n == 2 * 3 * 6273
    print(f"llava_ov_7b layer {layer}: worst err/max|V| = {worst:.2e}")


def test_llava15_7b_layer(cuda_dev, kvq):
    w = synth.workload("llava15_7b")
    c = case_of(w, 0)
    k = synth.make_kv(w, 0, "k", cuda_dev)
    v = synth.make_kv(w, 0, "v", cuda_dev)
    q = synth.make_q(w, 0, device=cuda_dev)
    n, worst = _run_full(c, q, k, v, w.T)
    assert n == 2 * 16 * 28 * 576
    print(f"llava15_7b: worst err/max|V| = {worst:.2e}")


@pytest.mark.parametrize("T", [1024, 4096, 16384, 32768])
def test_longctx(cuda_dev, kvq, T):
    w = synth.workload("longctx", T)
    c = case_of(w, 0)
    k = synth.make_kv(w, 0, "k", cuda_dev)
    v = synth.make_kv(w, 0, "v", cuda_dev)
    q = synth.make_q(w, 0, device=cuda_dev)
    n, worst = _run_full(c, q, k, v, w.T)  # every sequence, every head
    print(f"longctx T={T}: worst err/max|V| = {worst:.2e}")


@pytest.mark.parametrize("layer", [0, 4])
def test_llava_next_13b_layer(cuda_dev, kvq, layer):
    """Full-size layer (B = 32, 40 heads, T = 2940) built by one prefill
    append and decoded whole; every sequence compared."""
    w = synth.workload("llava_next_13b")
    c = case_of(w, layer)
    k = synth.make_kv(w, layer, "k", cuda_dev)
    v = synth.make_kv(w, layer, "v", cuda_dev)
    q = synth.make_q(w, layer, device=cuda_dev)
    n, worst = _run_full(c, q, k, v, w.T)
    assert n == 2 * 32 * 35 * 2880
    print(f"llava_next_13b layer {layer}: worst err/max|V| = {worst:.2e}")


def _fuzz_cases(n=40, seed=99):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.choice([1, 3]))
        H_kv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 4, 7, 8, 9, 16]))
        T = int(rng.choice([1, 17, 64, 65, 300, 1000]))
        kb, vb = (int(x) for x in rng.choice([2, 4, 8, 16], 2))
        G = int(rng.choice([32, 64, 128]))
        kind = i % 5
        if kind == 0:
            vs, ve = 0, 0            # no visual range
        elif kind == 1:
            vs, ve = 0, T            # all visual
        elif kind == 2:
            vs, ve = min(5, T), T    # text prefix
        elif kind == 3:
            vs, ve = 0, max(0, T - 3)  # text suffix
        else:
            vs = min(T, int(rng.integers(0, 20)))
            ve = vs + int(rng.integers(0, T - vs + 1))
        prot = [h for h in range(H_kv) if rng.random() < 0.3]
        # every other case also has K-only protected heads
        konly = [h for h in range(H_kv) if h not in prot and (h + i) % 3 == 1] if i % 2 == 0 else []
        out.append((i, Case(B, g * H_kv, H_kv, T, vs, ve, kb, vb, G, prot, konly=konly)))
    return out


@pytest.mark.parametrize("i,c", _fuzz_cases(), ids=lambda x: str(x) if isinstance(x, int) else "")
def test_fuzz(cuda_dev, kvq, i, c):
    q, k, v = synth.random_case(1000 + i, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev,
                                scale_k=float(1 + (i % 3)))
    _run_full(c, q, k, v, c.T_cap)


KONLY_CASES = [
    # B, H_q, H_kv, T_cap, vs, ve, kb, vb, G, protected, K-only
    Case(1, 28, 4, 6288, 14, 6287, 4, 2, 64, [], konly=[0]),        # LLaVA-OV shape, head 0 K-only
    Case(2, 32, 8, 1500, 32, 1500, 2, 2, 32, [3], konly=[0, 5]),    # both kinds, long visual tail
    Case(3, 16, 16, 300, 10, 290, 8, 4, 32, [1], konly=[2, 3, 9]),  # MHA
    Case(1, 8, 2, 500, 0, 500, 4, 16, 128, [], konly=[1]),          # bf16 V segment
]


@pytest.mark.parametrize("ci", range(len(KONLY_CASES)))
def test_konly_heads(cuda_dev, kvq, ci):
    """HeadGuard's "K, and V as needed": K-only protected heads keep their
    visual K in bf16 and quantise their V; storage bit-exact, attention
    within the bar."""
    c = KONLY_CASES[ci]
    q, k, v = synth.random_case(1200 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    n, worst = _run_full(c, q, k, v, c.T_cap)
    assert n > 0
    print(f"konly {ci}: worst err/max|V| = {worst:.2e}")


def test_chunked_appends_equal_one_append(cuda_dev, kvq):
    """Appending in pieces (prefill chunks, then one token at a time) writes
    the same bytes as one append of everything."""
    c = Case(2, 8, 4, 300, 20, 250, 4, 2, 64, [2])
    q, k, v = synth.random_case(7, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    L = c.layout()
    a = alloc_cache(L, fill=0)
    b = alloc_cache(L, fill=0)
    append(L, a, k, v, 0)
    bounds = [0, 7, 20, 21, 100, 249, 250, 251, 260, 300]
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        append(L, b, k[:, :, t0:t1], v[:, :, t0:t1], t0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_strided_inputs(cuda_dev, kvq):
    """K/V given as a strided view ([B, T, H, D] storage permuted)."""
    c = Case(2, 8, 4, 100, 10, 90, 8, 4, 32, [1])
    q, k, v = synth.random_case(8, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    ks = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vs_ = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert not ks.is_contiguous()
    L = c.layout()
    a = alloc_cache(L, fill=0)
    b = alloc_cache(L, fill=0)
    append(L, a, k, v, 0)
    append(L, b, ks, vs_, 0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [1, 5, 37, 200, 301])
def test_partial_T(cuda_dev, kvq, T):
    """Attend to a prefix of the cache: T before, inside and after the visual range."""
    c = Case(2, 12, 3, 301, 30, 240, 4, 4, 32, [0])
    q, k, v = synth.random_case(9, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    out, lse = decode(L, cache, q, T)
    torch.cuda.synchronize()
    ref, lr, vmax = oracle_decode(c, bits(q), bits(k), bits(v), T, SCALE)
    check_decode(c, out, lse, ref, lr, vmax)


def test_decode_writes_only_its_outputs(cuda_dev, kvq):
    """Decode never writes the cache (no dequantised K/V written back), and
    ignores the workspace's previous contents."""
    c = Case(3, 16, 4, 500, 14, 480, 2, 4, 32, [3])
    q, k, v = synth.random_case(10, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    before = cache.clone()
    o1, l1 = decode(L, cache, q, 500, ws_fill=0xFF)  # NaN bytes in the workspace
    o2, l2 = decode(L, cache, q, 500, ws_fill=0x00)
    torch.cuda.synchronize()
    assert torch.equal(cache, before)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_repeatable(cuda_dev, kvq):
    c = Case(1, 28, 4, 2000, 14, 1990, 4, 2, 64, [0])
    q, k, v = synth.random_case(11, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    outs = [decode(L, cache, q, 2000)[0] for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_quantiser_edge_rows(cuda_dev, kvq):
    """Constant groups, signed-zero minima, tiny ranges near binary16
    underflow, large outliers: codes/scales/zeros still bit-exact."""
    c = Case(1, 4, 2, 64, 0, 64, 4, 8, 32, [])
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 2, 64, 128)).astype(np.float32)
    x[0, 0, 0, :] = 1.25                     # constant row
    x[0, 0, 1, :32] = 0.0
    x[0, 0, 1, 5] = -0.0                     # signed-zero minimum
    x[0, 0, 1, 7] = 3.0
    x[0, 0, 2, :] *= 1e-6                    # scale underflows binary16
    x[0, 0, 3, :] *= 1e-3
    x[0, 1, 4, 9] = 60000.0                  # large outlier (inside fp16 range)
    x[0, 1, 5, :] = np.float32(2.0) ** -20   # zero below binary16 normal range
    x[0, 1, 6, 32:64] = 0.75                 # one constant group inside a varying row
    x[0, 0, 7, 96:] = -2.5                   # (both tensors, other lanes of the row)
    k = torch.tensor(x).to(torch.bfloat16).to(cuda_dev)
    v = k.flip(2).contiguous()
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    torch.cuda.synchronize()
    check_append(L, c, cache, bits(k), bits(v), 64)


def test_quantiser_ties_and_near_ties(cuda_dev, kvq):
    """Values whose quotient (x - z) / s is exactly k + 1/2 (ties, rounded
    half to even) or one bf16 step beside it: the codes must match the
    correctly rounded definition bit for bit."""
    c = Case(1, 4, 2, 64, 0, 64, 4, 2, 32, [])
    rows = []
    rng = np.random.default_rng(17)
    for r in range(64):
        g = np.zeros(128, np.float32)
        for grp in range(4):
            base = grp * 32
            # INT4 (K): min 0, max 15/16 -> s = 1/16; ties at (k + 1/2)/16
            vals = np.array([(k + 0.5) / 16 for k in range(15)] * 2 + [0.0, 15 / 16], np.float32)
            if r % 3 == 1:  # one bf16 step up from each tie
                vals[:30] = np.nextafter(torch.tensor(vals[:30]).to(torch.bfloat16).float().numpy(),
                                         np.float32(2.0))
            vals = vals * np.float32(2.0) ** int(rng.integers(-6, 6))
            g[base:base + 32] = vals
        rows.append(g)
    x = np.stack(rows).reshape(1, 1, 64, 128)
    k = torch.tensor(np.concatenate([x, x[:, :, ::-1]], axis=1)).to(torch.bfloat16).to(cuda_dev)
    v = k.clone()
    L = c.layout()
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    torch.cuda.synchronize()
    check_append(L, c, cache, bits(k), bits(v), 64)
