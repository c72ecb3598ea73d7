"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (optionally a
copy built with one planted mistake) disagrees with a fact fixed by the pages
or by mathematics: a library routine for a special case, brute force on tiny
inputs, a closed form, an invariant, or a hand-computed worked example.
``test_oracle_pins.py`` runs them on the real oracle and checks that every
planted mistake is caught by at least one of them.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16_bits_from_float(x) -> np.ndarray:
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _f16_value(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------------------
# Number formats: the oracle's binary16 conversion against numpy's.
# ---------------------------------------------------------------------------

def pin_f16_conversion(plant: int = 0, n: int = 20000):
    rng = np.random.default_rng(7)
    mags = np.exp(rng.uniform(np.log(1e-9), np.log(1e6), n)).astype(np.float32)
    xs = np.concatenate([
        mags * rng.choice([-1.0, 1.0], n).astype(np.float32),
        np.float32([0.0, -0.0, 65504.0, 65519.99, 65520.0, 70000.0, 6.1035156e-05,
                    5.9604645e-08, 2.9802322e-08, 2.9802326e-08, 1.0, 1.00048828125,
                    1.000732421875, 2049.0, 2051.0]),
        # exact ties between two binary16 neighbours (round half to even)
        (np.arange(1, 400, dtype=np.float32) + 0.5) * np.float32(2.0 ** -24),
        (np.float32(1024.0) + np.arange(0, 64, dtype=np.float32) * np.float32(0.5)),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(float(x), plant) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"f32->f16 differs from numpy at {xs[bad[:5]]}: {got[bad[:5]]} vs {want[bad[:5]]}"
    # binary16 -> float: every finite pattern, exact
    pats = np.arange(0, 1 << 16, 97, dtype=np.uint32).astype(np.uint16)
    pats = pats[np.isfinite(pats.view(np.float16))]
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_bits_to_f32(int(p), plant) for p in pats], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------------------
# Quantiser
# ---------------------------------------------------------------------------

def _groups_for_quantiser(seed: int):
    rng = np.random.default_rng(seed)
    cases = []
    for bits in (2, 4, 8):
        for G in (32, 64, 128):
            for kind in range(5):
                D = 128
                if kind == 0:
                    x = rng.standard_normal(D)
                elif kind == 1:
                    x = rng.standard_normal(D) * 10.0 + 3.0
                elif kind == 2:
                    x = rng.standard_normal(D) * 1e-3
                elif kind == 3:
                    x = rng.uniform(-1, 1, D)
                    x[rng.integers(0, D, 4)] *= 40.0
                else:
                    x = rng.standard_normal(D) * 1e-6  # scale near binary16 underflow
                cases.append((bits, G, _bf16_bits_from_float(x)))
    return cases


def pin_quantiser_bruteforce(plant: int = 0):
    """Given the stored fp16 scale s and zero z of each group, every code the
    oracle picks is a nearest code over ALL 2^b candidates (exact rational
    distances); within a tiny tolerance of a half-way point either neighbour
    is accepted, because the spec divides in fp32."""
    for bits, G, x in _groups_for_quantiser(11):
        codes, s, z = oracle.quantize_row(x, G, bits, plant)
        qmax = (1 << bits) - 1
        assert codes.max() <= qmax
        xv = _bf16_value(x).astype(np.float64)
        for g in range(len(s)):
            sv = Fraction(float(_f16_value(s[g])))
            zv = Fraction(float(_f16_value(z[g])))
            for i in range(G):
                d = g * G + i
                xf = Fraction(float(xv[d]))
                if sv == 0:
                    assert codes[d] == 0
                    continue
                dists = [abs(xf - (c * sv + zv)) for c in range(qmax + 1)]
                best = min(dists)
                tol = sv * Fraction(1, 1 << 20) * max(1, abs((xf - zv) / sv))
                assert dists[codes[d]] <= best + tol, (bits, G, d, codes[d], dists.index(best))


def pin_quantiser_scale_zero(plant: int = 0):
    """z is the group minimum rounded to binary16 and s*(2^b-1) equals the
    group range up to the two roundings (fp32 division, then binary16)."""
    for bits, G, x in _groups_for_quantiser(12):
        codes, s, z = oracle.quantize_row(x, G, bits, plant)
        xv = _bf16_value(x)
        qmax = (1 << bits) - 1
        for g in range(len(s)):
            grp = xv[g * G:(g + 1) * G]
            mn, mx = float(grp.min()), float(grp.max())
            assert z[g] == np.float16(np.float32(mn) + np.float32(0.0)).view(np.uint16), "zero != fp16(min)"
            sv = float(_f16_value(s[g]))
            rng_ = mx - mn
            # |s - range/qmax| <= half an fp16 ulp of s (+ subnormal spacing) + fp32 rounding
            ideal = rng_ / qmax
            bound = abs(ideal) * (2.0 ** -11 + 2.0 ** -23) + 2.0 ** -25
            assert abs(sv - ideal) <= bound, (bits, G, sv, ideal)


def pin_quantiser_exact_grid(plant: int = 0):
    """A group whose values lie exactly on z + k*s with s a power of two and
    k covering 0..2^b-1 quantises to exactly those k, and dequantises back to
    the inputs bit for bit (closed form)."""
    with open(os.path.join(GOLDEN, "quantiser_worked_examples.json")) as f:
        ex = json.load(f)["exact_grid"]
    for case in ex:
        bits, G, z0, s0, ks = case["bits"], case["G"], case["z"], case["s"], case["codes"]
        vals = np.array([z0 + k * s0 for k in ks], dtype=np.float64)
        x = _bf16_bits_from_float(vals)
        assert np.array_equal(_bf16_value(x).astype(np.float64), vals), "fixture not bf16-exact"
        codes, s, z = oracle.quantize_row(x, G, bits, plant)
        assert list(codes) == ks, (bits, G)
        assert float(_f16_value(s[0])) == s0 and float(_f16_value(z[0])) == z0
        deq = oracle.dequant_row(codes, s, z, G, plant)
        assert np.array_equal(deq, vals)


def pin_quantiser_constant_group(plant: int = 0):
    for bits in (2, 4, 8):
        for val in (0.0, 1.5, -3.25, 1e-3):
            x = _bf16_bits_from_float(np.full(64, val))
            codes, s, z = oracle.quantize_row(x, 32, bits, plant)
            assert np.all(codes == 0) and np.all(s == 0)
            deq = oracle.dequant_row(codes, s, z, 32, plant)
            assert np.array_equal(deq, _bf16_value(x).astype(np.float64)
                                  if val != 1e-3 else _f16_value(z).repeat(32))


def pin_signed_zero_minimum(plant: int = 0):
    """A group whose minimum is a signed zero stores the zero as +0 whatever
    the order of -0 and +0 in the row (signed zeros compare equal)."""
    for order in ((-0.0, 0.0), (0.0, -0.0)):
        vals = np.full(32, 0.5)
        vals[3], vals[17] = order
        codes, s, z = oracle.quantize_row(_bf16_bits_from_float(vals), 32, 4, plant)
        assert int(z[0]) == 0, hex(int(z[0]))
        assert codes[3] == 0 and codes[17] == 0 and codes[0] == 15


def pin_round_trip_bound(plant: int = 0):
    """|x - deq(q(x))| <= s/2 + |min - z| + 2^-20 max(|x|, s) on every packed
    element of the tiny workload and a slice of the LLaVA-OV-shaped one."""
    for name, hs in (("tiny", [0]), ("llava_ov_7b", [1, 2])):
        w = synth.workload(name)
        for which, bits in (("k", w.layers[0].k_bits), ("v", w.layers[0].v_bits)):
            x = synth.bf16_bits(synth.make_kv(w, 0, which, h_range=hs, T=min(w.T, 1200)))
            G = w.group_size
            rows = x.reshape(-1, w.D)[::7]
            for r in rows:
                codes, s, z = oracle.quantize_row(r, G, bits, plant)
                deq = oracle.dequant_row(codes, s, z, G, plant)
                xv = _bf16_value(r).astype(np.float64)
                sv = _f16_value(s).repeat(G)
                zv = _f16_value(z).repeat(G)
                mn = xv.reshape(-1, G).min(axis=1).repeat(G)
                bound = sv / 2 + np.abs(mn - zv) + 2.0 ** -20 * np.maximum(np.abs(xv), sv)
                err = np.abs(xv - deq)
                assert np.all(err <= bound), (name, which, float((err - bound).max()))


# ---------------------------------------------------------------------------
# Packing
# ---------------------------------------------------------------------------

def pin_pack_worked_examples(plant: int = 0):
    with open(os.path.join(GOLDEN, "pack_worked_examples.json")) as f:
        ex = json.load(f)["examples"]
    for case in ex:
        words = oracle.pack_row(np.array(case["codes"], np.uint8), case["bits"], plant)
        assert [int(w) for w in words] == [int(h, 16) for h in case["words"]], case["bits"]


def pin_pack_roundtrip(plant: int = 0):
    rng = np.random.default_rng(3)
    for bits in (2, 4, 8):
        codes = rng.integers(0, 1 << bits, 128).astype(np.uint8)
        words = oracle.pack_row(codes, bits, plant)
        per = 32 // bits
        back = [(int(words[d // per]) >> (bits * (d % per))) & ((1 << bits) - 1) for d in range(128)]
        assert back == [int(c) for c in codes]


def pin_slot_worked_examples(plant: int = 0):
    """Storage slots of a few elements, derived by hand from the layout."""
    with open(os.path.join(GOLDEN, "slot_order_examples.json")) as f:
        ex = json.load(f)
    for bits, pairs in ex["k"].items():
        for d, slot in pairs:
            assert oracle.code_slot("k", int(bits), d, plant) == slot, ("k", bits, d)
    for bits in (2, 4, 8):
        for d, slot in ex["v"]:
            assert oracle.code_slot("v", bits, d, plant) == slot, ("v", bits, d)


def pin_slot_order_is_permutation(plant: int = 0):
    """Every element gets its own slot, and the stored words hold exactly the
    row's codes (read back through the slot order)."""
    rng = np.random.default_rng(5)
    for kind in ("k", "v"):
        for bits in (2, 4, 8):
            slots = [oracle.code_slot(kind, bits, d, plant) for d in range(128)]
            assert sorted(slots) == list(range(128)), (kind, bits)
            for G in (32, 64, 128):
                x = _bf16_bits_from_float(rng.standard_normal((3, 128)) * 3.0)
                words, sz = oracle.quantize_pack_rows_stored(x, G, bits, kind, plant)
                w_seq, s_seq, z_seq = oracle.quantize_pack_rows(x, G, bits, plant)
                per, mask = 32 // bits, (1 << bits) - 1
                for r in range(3):
                    seq = [(int(w_seq[r, d // per]) >> (bits * (d % per))) & mask for d in range(128)]
                    got = [(int(words[r, j // per]) >> (bits * (j % per))) & mask for j in slots]
                    assert got == seq, (kind, bits, G, r)
                    ng = 128 // G
                    assert list(sz[r, :ng]) == list(z_seq[r]) and list(sz[r, ng:]) == list(s_seq[r])


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _small_case(seed, B, Hq, Hkv, T, D):
    q, k, v = synth.random_case(seed, B, Hq, Hkv, D, T)
    return synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v)


def pin_attention_single_position(plant: int = 0):
    """T = 1: the only weight is 1, so the output is the (dequantised) value row."""
    q, k, v = _small_case(21, 2, 4, 2, 1, 64)
    kh, _ = oracle.reconstruct(k, 0, 1, [0, 0], 4, 32, plant)
    vh, _ = oracle.reconstruct(v, 0, 1, [0, 0], 4, 32, plant)
    out, lse = oracle.attention(q, kh, vh, 0.125, plant=plant)
    for hq in range(4):
        assert np.array_equal(out[:, hq], vh[:, hq // 2, 0]), hq


def pin_attention_uniform(plant: int = 0):
    """All scores equal (K = 0): the output is the plain mean of V."""
    q, _, v = _small_case(22, 1, 2, 1, 37, 32)
    kh = np.zeros((1, 1, 37, 32))
    vh = _bf16_value(v).astype(np.float64).reshape(1, 1, 37, 32)
    out, lse = oracle.attention(q, kh, vh, 0.3, plant=plant)
    mean = np.array([math.fsum(vh[0, 0, :, d]) / 37 for d in range(32)])
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-13)
    assert abs(lse[0, 0] - math.log(37)) < 1e-13


def pin_attention_weights_sum(plant: int = 0):
    q, k, _ = _small_case(23, 1, 4, 2, 300, 128)
    kh = _bf16_value(k).astype(np.float64).reshape(k.shape) * 3.0
    for hq in range(4):
        w = oracle.attention_weights(q, kh, hq, 1 / math.sqrt(128), plant)
        assert abs(math.fsum(w) - 1.0) < 1e-12 and np.all(w >= 0)


def pin_attention_bruteforce(plant: int = 0):
    """Exact rational dot products, exp without max-shift, fsum: tiny T and D."""
    B, Hq, Hkv, T, D = 1, 4, 2, 9, 16
    q, k, v = _small_case(24, B, Hq, Hkv, T, D)
    kh = _bf16_value(k).astype(np.float64).reshape(k.shape)
    vh = _bf16_value(v).astype(np.float64).reshape(v.shape)
    qv = _bf16_value(q).astype(np.float64).reshape(q.shape)
    scale = 0.25
    out, lse = oracle.attention(q, kh, vh, scale, plant=plant)
    for hq in range(Hq):
        h = hq // (Hq // Hkv)
        sc = [float(scale * sum(Fraction(qv[0, hq, d]) * Fraction(kh[0, h, t, d]) for d in range(D)))
              for t in range(T)]
        e = [math.exp(s) for s in sc]
        den = math.fsum(e)
        ref = [math.fsum(e[t] * vh[0, h, t, d] for t in range(T)) / den for d in range(D)]
        assert np.allclose(out[0, hq], ref, rtol=1e-12, atol=1e-14), hq
        assert abs(lse[0, hq] - math.log(den)) < 1e-12


def pin_all_protected_closed_form(plant: int = 0):
    """With every KV head protected (or bits = 16) nothing is quantised, so the
    decode output equals fp64 softmax attention on the raw bf16 inputs
    (computed here with numpy's matmul/exp)."""
    B, Hq, Hkv, T, D = 2, 8, 2, 80, 128
    q, k, v = _small_case(25, B, Hq, Hkv, T, D)
    scale = 1 / math.sqrt(D)
    qv = _bf16_value(q).astype(np.float64).reshape(q.shape)
    kv = _bf16_value(k).astype(np.float64).reshape(k.shape)
    vv = _bf16_value(v).astype(np.float64).reshape(v.shape)
    g = Hq // Hkv
    ref = np.empty((B, Hq, D))
    for b in range(B):
        for hq in range(Hq):
            s = scale * (kv[b, hq // g] @ qv[b, hq])
            w = np.exp(s - s.max())
            ref[b, hq] = (w / w.sum()) @ vv[b, hq // g]
    for prot, kb, vb in (([1, 1], 4, 2), ([0, 0], 16, 16)):
        out, _, _, _ = oracle.decode_reference(q, k, v, 10, 70, prot, kb, vb, 32, scale, plant=plant)
        assert np.allclose(out, ref, rtol=0, atol=1e-12), (prot, kb, vb)


# ---------------------------------------------------------------------------
# Invariants of the policy (the pages' sanity checklist)
# ---------------------------------------------------------------------------

def pin_text_rows_untouched(plant: int = 0):
    """Text positions and the current step (everything outside the visual
    range) are never quantised: reconstruct returns them bit-identical."""
    _, k, _ = _small_case(26, 2, 4, 4, 50, 128)
    vs, ve = 7, 40
    out, n = oracle.reconstruct(k, vs, ve, [0, 1, 0, 0], 2, 32, plant)
    raw = _bf16_value(k).astype(np.float64).reshape(k.shape)
    for p in list(range(0, vs)) + list(range(ve, 50)):
        assert np.array_equal(out[:, :, p], raw[:, :, p]), p
    assert np.array_equal(out[:, 1], raw[:, 1]), "protected head was quantised"
    assert not np.array_equal(out[:, 0, vs:ve], raw[:, 0, vs:ve])


def pin_packed_row_count(plant: int = 0):
    """Packed-row count = visual rows x unprotected heads x batch, and it is
    non-zero whenever both factors are."""
    _, k, _ = _small_case(27, 3, 4, 4, 40, 128)
    for prot, vs, ve, bits in (([0, 1, 0, 0], 5, 33, 4), ([1, 1, 1, 1], 5, 33, 4),
                               ([0, 0, 0, 0], 0, 40, 8), ([0, 1, 0, 0], 5, 33, 16),
                               ([0, 0, 0, 1], 12, 12, 2)):
        _, n = oracle.reconstruct(k, vs, ve, prot, bits, 32, plant)
        want = (ve - vs) * (4 - sum(prot)) * 3 if bits < 16 else 0
        assert n == want, (prot, vs, ve, bits, n, want)


def pin_gqa_grouping(plant: int = 0):
    """Query head hq reads KV head hq // (H_q / H_kv) (contiguous groups):
    with distinct constant V per KV head, each output row names its head."""
    B, Hq, Hkv, T, D = 1, 6, 3, 5, 32
    q, k, _ = _small_case(28, B, Hq, Hkv, T, D)
    kh = _bf16_value(k).astype(np.float64).reshape(k.shape)
    vh = np.zeros((B, Hkv, T, D))
    for h in range(Hkv):
        vh[0, h] = h + 1.0
    out, _ = oracle.attention(q, kh, vh, 0.2, plant=plant)
    for hq in range(Hq):
        assert np.allclose(out[0, hq], hq // 2 + 1.0, atol=1e-13), hq


def pin_konly_policy(plant: int = 0):
    """A K-only protected head (HeadGuard brief: image Key kept, Value as
    needed) keeps its visual K rows exactly and quantises its visual V rows
    like an unprotected head; other heads are unaffected."""
    rng = np.random.default_rng(11)
    B, H, T, D, vs, ve = 1, 3, 24, 128, 4, 20
    k = _bf16_bits_from_float(rng.standard_normal((B, H, T, D)))
    v = _bf16_bits_from_float(rng.standard_normal((B, H, T, D)))
    q = _bf16_bits_from_float(rng.standard_normal((B, H, D)))
    _, _, kh, vh = oracle.decode_reference(q, k, v, vs, ve, [2, 1, 0], 4, 4, 32, 0.1, plant=plant)
    kraw = _bf16_value(k).astype(np.float64)
    vraw = _bf16_value(v).astype(np.float64)
    assert np.array_equal(kh[:, 0], kraw[:, 0]) and np.array_equal(kh[:, 1], kraw[:, 1])
    assert np.array_equal(vh[:, 1], vraw[:, 1])
    # the K-only head's V and the packed head's K and V are quantised
    for x, xr in ((vh[:, 0], vraw[:, 0]), (kh[:, 2], kraw[:, 2]), (vh[:, 2], vraw[:, 2])):
        assert not np.array_equal(x[:, vs:ve], xr[:, vs:ve])
        assert np.array_equal(x[:, :vs], xr[:, :vs]) and np.array_equal(x[:, ve:], xr[:, ve:])
    vq, _ = oracle.reconstruct(v[:, :1], vs, ve, [0], 4, 32, plant)
    assert np.array_equal(vh[:, 0], vq[:, 0])


# ---------------------------------------------------------------------------
# K-vs-V sensitivity probe ("VLM_KV_Quantization" sections 3-4: KL of the
# distribution after quantising K or V alone, against the unquantised one)
# ---------------------------------------------------------------------------

def _readout(seed, n_out, D):
    return np.random.default_rng(seed).standard_normal((n_out, D)).astype(np.float32)


def pin_probe_nothing_quantised(plant: int = 0):
    """With nothing quantised (bits 16, or every head protected) the cache
    as read is the raw cache: every divergence and the error are exactly 0."""
    q, k, v = _small_case(41, 1, 4, 2, 60, 128)
    W = _readout(1, 16, 128)
    for prot, kb, vb in (([0, 0], 16, 16), ([1, 1], 2, 2)):
        r = oracle.sensitivity_reference(q, k, v, 5, 50, prot, kb, vb, 32, 0.1, W, plant=plant)
        assert np.array_equal(r, np.zeros_like(r)), (prot, kb, vb)


def pin_probe_v_only_leaves_weights(plant: int = 0):
    """Quantising V alone cannot move the softmax weights (kl_attn = 0
    exactly) but does move the output; quantising K alone moves both."""
    q, k, v = _small_case(42, 1, 4, 2, 60, 128)
    W = _readout(2, 16, 128)
    r = oracle.sensitivity_reference(q, k, v, 5, 50, [0, 0], 16, 2, 32, 0.1, W, plant=plant)
    assert np.all(r[..., 0] == 0.0)
    assert np.all(r[..., 1] > 0) and np.all(r[..., 2] > 0)
    r = oracle.sensitivity_reference(q, k, v, 5, 50, [0, 0], 2, 16, 32, 0.1, W, plant=plant)
    assert np.all(r[..., 0] > 0) and np.all(r[..., 1] > 0) and np.all(r[..., 2] > 0)


def pin_probe_two_positions_closed_form(plant: int = 0):
    """Two positions, q = e_0, scale 1.  Position 0 is text with k = e_0;
    position 1 is visual with k = (0.5, 3, 0, ...), whose 2-bit group has
    s = 1, z = 0 and sends 0.5 to code 0 (half to even): scores (1, 0.5)
    exact, (1, 0) as read.  v_0 = e_0, v_1 = 0 (V unquantised), readout rows
    (4 e_0, 0).  Every value below is a two-term formula."""
    D = 32
    k = np.zeros((1, 1, 2, D))
    k[0, 0, 0, 0] = 1.0
    k[0, 0, 1, 0], k[0, 0, 1, 1] = 0.5, 3.0
    v = np.zeros((1, 1, 2, D))
    v[0, 0, 0, 0] = 1.0
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    W = np.zeros((2, D), np.float32)
    W[0, 0] = 4.0
    r = oracle.sensitivity_reference(_bf16_bits_from_float(q), _bf16_bits_from_float(k),
                                     _bf16_bits_from_float(v), 1, 2, [0], 2, 16, 32, 1.0, W,
                                     plant=plant)

    def two(x0, x1):  # softmax of two scores
        e0, e1 = math.exp(x0), math.exp(x1)
        return e0 / (e0 + e1), e1 / (e0 + e1)

    p0, p1 = two(1.0, 0.5)
    h0, h1 = two(1.0, 0.0)
    kl_attn = p0 * math.log(p0 / h0) + p1 * math.log(p1 / h1)
    P0, P1 = two(4.0 * p0, 0.0)
    Q0, Q1 = two(4.0 * h0, 0.0)
    kl_out = P0 * math.log(P0 / Q0) + P1 * math.log(P1 / Q1)
    assert abs(r[0, 0, 0] - kl_attn) < 1e-14, (r[0, 0, 0], kl_attn)
    assert abs(r[0, 0, 1] - kl_out) < 1e-14, (r[0, 0, 1], kl_out)
    assert abs(r[0, 0, 2] - abs(p0 - h0)) < 1e-15


def pin_probe_nonnegative_and_ordered(plant: int = 0):
    """Divergences are >= 0 (Gibbs), and fewer bits do more damage: mean
    INT2 > mean INT4 > mean INT8 for each of K and V."""
    q, k, v = _small_case(43, 2, 4, 2, 120, 128)
    W = _readout(3, 32, 128)
    for which in ("k", "v"):
        means = []
        for bits in (2, 4, 8):
            kb, vb = (bits, 16) if which == "k" else (16, bits)
            r = oracle.sensitivity_reference(q, k, v, 8, 110, [0, 0], kb, vb, 32, 0.09, W, plant=plant)
            assert np.all(r >= 0), (which, bits)
            means.append(r[..., 1].mean())
        assert means[0] > means[1] > means[2] > 0, (which, means)


ALL_PINS = [
    pin_f16_conversion,
    pin_quantiser_bruteforce,
    pin_quantiser_scale_zero,
    pin_quantiser_exact_grid,
    pin_quantiser_constant_group,
    pin_signed_zero_minimum,
    pin_round_trip_bound,
    pin_pack_worked_examples,
    pin_pack_roundtrip,
    pin_slot_worked_examples,
    pin_slot_order_is_permutation,
    pin_attention_single_position,
    pin_attention_uniform,
    pin_attention_weights_sum,
    pin_attention_bruteforce,
    pin_all_protected_closed_form,
    pin_text_rows_untouched,
    pin_packed_row_count,
    pin_gqa_grouping,
    pin_konly_policy,
    pin_probe_nothing_quantised,
    pin_probe_v_only_leaves_weights,
    pin_probe_two_positions_closed_form,
    pin_probe_nonnegative_and_ordered,
]
