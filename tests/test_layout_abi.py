"""Host-side tests of the C ABI: layout arithmetic, exported symbols and the
argument checks that return before any launch (no GPU needed)."""
import ctypes
import re
import subprocess

import pytest

import bit_mixed_precision_kvq_gb300 as kvq
from bit_mixed_precision_kvq_gb300 import build_native

HEADER = __import__("os").path.join(build_native.ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    build_native.build()
    return kvq.load()


def test_header_declares_what_library_exports(lib):
    text = open(HEADER).read()
    declared = set(re.findall(r"^\s*(?:kvq_status|const char\*|int|size_t|void)\s+(kvq_\w+)\s*\(", text, re.M))
    assert declared == set(kvq.EXPORTED_SYMBOLS)
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(kvq_\w+)$", out, re.M))
    assert declared <= exported, declared - exported
    for name in declared:
        assert hasattr(lib, name)


def _align(x, a):
    return (x + a - 1) // a * a


def _expected(B, Hq, Hkv, D, Tcap, vs, ve, kb, vb, G, prot, konly):
    """Independent restatement of the documented segment shapes."""
    Tv = ve - vs
    Tvp = -(-Tv // 16) * 16
    npr = len(prot)
    nko = len(konly)
    npk = Hkv - npr - nko
    rb = [D * kb // 8, 4 * D // G if kb < 16 else 0, D * vb // 8, 4 * D // G if vb < 16 else 0,
          2 * D, 2 * D, 2 * D, 2 * D]
    # K-only heads: K with the protected heads' K, V with the packed heads' V
    rows = ([B * npk * Tvp] * 2 + [B * (npk + nko) * Tvp] * 2 + [B * (npr + nko) * Tv, B * npr * Tv]
            + [B * Hkv * (Tcap - Tv)] * 2)
    off, offs = 0, []
    for r, n in zip(rb, rows):
        offs.append(off)
        off = _align(off + r * n + 256, 256)
    return rb, rows, offs, off


CASES = [
    (1, 4, 1, 128, 257, 14, 256, 4, 4, 32, [], []),
    (1, 28, 4, 128, 6288, 14, 6287, 4, 2, 64, [0], []),
    (16, 32, 32, 128, 617, 40, 616, 8, 4, 32, [1, 5, 9, 30], []),
    (8, 32, 8, 128, 32769, 32, 32768, 2, 2, 32, [3], []),
    (32, 40, 40, 128, 2941, 60, 2940, 8, 8, 64, [0, 1, 2, 3, 39], []),
    (3, 12, 4, 128, 100, 0, 100, 16, 2, 128, [0, 1, 2, 3], []),
    (2, 2, 2, 128, 50, 10, 10, 4, 16, 32, [], []),
    (1, 28, 4, 128, 6288, 14, 6287, 4, 2, 64, [], [0]),          # K-only protection
    (4, 32, 8, 128, 1000, 8, 990, 2, 4, 32, [5], [1, 6, 7]),     # both kinds
]


@pytest.mark.parametrize("case", CASES)
def test_layout_matches_formula(lib, case):
    B, Hq, Hkv, D, Tcap, vs, ve, kb, vb, G, prot, konly = case
    L = kvq.cache_layout(B, Hq, Hkv, D, Tcap, vs, ve, kb, vb, G, prot, konly)
    rb, rows, offs, total = _expected(*case)
    assert list(L.row_bytes) == rb
    assert list(L.bytes) == [r * n for r, n in zip(rb, rows)]
    assert list(L.off) == offs and L.total_bytes == total
    assert all(o % 256 == 0 for o in L.off)
    assert L.g == Hq // Hkv and L.n_prot == len(prot) and L.n_konly == len(konly)
    assert L.n_packed == Hkv - len(prot) - len(konly)
    assert L.Tv == ve - vs and L.T_text == Tcap - (ve - vs) and L.Tv_pad == -(-(ve - vs) // 16) * 16
    nhc = -(-(Hq // Hkv) // 8)
    assert L.units == B * Hkv * nhc
    # head -> slot -> head round trip
    ps = pk = ko = 0
    for h in range(Hkv):
        if h in prot:
            assert L.slot[h] == ps and L.prot_head[ps] == h
            ps += 1
        elif h in konly:
            assert L.slot[h] == ko and L.konly_head[ko] == h
            ko += 1
        else:
            assert L.slot[h] == pk and L.packed_head[pk] == h
            pk += 1
    # "is INT2 really 2 bit/value": codes cost b bits, plus 32 bits of fp16
    # scale and zero per group of G ("VLM_KV_Quantization", intro checklist)
    assert L.eff_bits_k == (kb + 32.0 / G if kb < 16 else 16.0)
    assert L.eff_bits_v == (vb + 32.0 / G if vb < 16 else 16.0)
    if kb < 16:
        assert L.row_bytes[kvq.SEG_K_CODES] * 8 == kb * D
    slots = L.units + 1024 - 1
    # 256-byte head (status word), arrival counters, partial o and (m, l)
    assert L.workspace_bytes == (256 + _align(4 * L.units, 256) + _align(slots * 8 * D * 4, 256)
                                 + _align(slots * 8 * 8, 256))


BAD_DESCS = [
    dict(B=0), dict(H_kv=0), dict(H_q=6), dict(H_kv=129, H_q=129), dict(D=100), dict(T_cap=0),
    dict(vis_start=-1), dict(vis_end=300), dict(vis_start=20, vis_end=10), dict(k_bits=3),
    dict(v_bits=1), dict(k_bits=32), dict(group_size=16), dict(group_size=48),
]


@pytest.mark.parametrize("bad", BAD_DESCS, ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_layout_rejects_bad_desc(lib, bad):
    args = dict(B=1, H_q=8, H_kv=4, D=128, T_cap=256, vis_start=10, vis_end=200, k_bits=4,
                v_bits=4, group_size=32)
    args.update(bad)
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_layout(protected=[], **args)
    assert e.value.status == 1


def test_layout_unsupported_head_dim(lib):
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_layout(1, 8, 4, 64, 256, 10, 200, 4, 4, 32, [])
    assert e.value.status == 2


def test_layout_rejects_mask_beyond_heads(lib):
    with pytest.raises(kvq.KvqError):
        kvq.cache_layout(1, 8, 4, 128, 256, 10, 200, 4, 4, 32, [5])
    with pytest.raises(kvq.KvqError):
        kvq.cache_layout(1, 8, 4, 128, 256, 10, 200, 4, 4, 32, [], [4])


def test_layout_rejects_unknown_protection_mode(lib):
    d = kvq.LayoutDesc(1, 8, 4, 128, 256, 10, 200, 4, 4, 32)
    d.protected_heads[1] = 3
    out = kvq.Layout()
    assert lib.kvq_cache_layout(ctypes.byref(d), ctypes.byref(out)) == 1


# Fake, never-dereferenced device addresses: every case below must be rejected
# on the host before any CUDA call.
FAKE = 1 << 40


def test_append_argument_checks(lib):
    L = kvq.cache_layout(1, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ok = dict(cache=FAKE, k=FAKE, v=FAKE, t0=0, n_tok=4, strides=(4 * 256 * 128, 256 * 128, 128))
    for bad, code in ((dict(cache=0), 1), (dict(k=0), 1), (dict(cache=FAKE + 16), 1),
                      (dict(k=FAKE + 2), 1), (dict(strides=(1, 128, 128)), 1),
                      (dict(t0=-1), 1), (dict(n_tok=-2), 1), (dict(t0=250, n_tok=7), 3)):
        a = dict(ok)
        a.update(bad)
        with pytest.raises(kvq.KvqError) as e:
            kvq.quantize_append(L, a["cache"], a["k"], a["v"], a["t0"], a["n_tok"], a["strides"],
                                stream=0)
        assert e.value.status == code, bad
    # n_tok == 0 is a no-op and touches nothing
    kvq.quantize_append(L, FAKE, FAKE, FAKE, 256, 0, ok["strides"], stream=0)


def test_decode_argument_checks(lib):
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ws = L.workspace_bytes
    ok = dict(cache=FAKE, q=FAKE, T=100, out=FAKE, lse=0, ws=FAKE, ws_bytes=ws)
    for bad, code in ((dict(cache=0), 1), (dict(q=0), 1), (dict(out=0), 1), (dict(ws=0), 1),
                      (dict(T=0), 1), (dict(T=257), 1), (dict(q=FAKE + 8), 1),
                      (dict(ws=FAKE + 64), 1), (dict(lse=FAKE + 2), 1),
                      (dict(ws_bytes=ws - 1), 3)):
        a = dict(ok)
        a.update(bad)
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_attention(L, a["cache"], a["q"], a["T"], a["out"], 0.1, a["lse"], a["ws"],
                                 a["ws_bytes"], stream=0)
        assert e.value.status == code, bad
    with pytest.raises(kvq.KvqError):
        kvq.decode_attention(L, FAKE, FAKE, 10, FAKE, float("nan"), 0, FAKE, ws, stream=0)


def test_decode_step_argument_checks(lib):
    # text 0-9 and 200-255, visual 10-199
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ws = L.workspace_bytes
    ok = dict(cache=FAKE, q=FAKE, kn=FAKE, vn=FAKE, t=220, out=FAKE, lse=0, ws=FAKE, ws_bytes=ws)
    for bad, code in ((dict(kn=0), 1), (dict(vn=0), 1), (dict(kn=FAKE + 8), 1),
                      (dict(vn=FAKE + 2), 1), (dict(t=-1), 1), (dict(t=256), 1), (dict(t=10), 1),
                      (dict(t=199), 1), (dict(cache=0), 1), (dict(q=FAKE + 8), 1),
                      (dict(ws=0), 1), (dict(ws=FAKE + 64), 1), (dict(ws_bytes=ws - 1), 3)):
        a = dict(ok)
        a.update(bad)
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_step(L, a["cache"], a["q"], a["kn"], a["vn"], a["t"], a["out"], 0.1,
                            a["lse"], a["ws"], a["ws_bytes"], stream=0)
        assert e.value.status == code, bad
    with pytest.raises(kvq.KvqError):
        kvq.decode_step(L, FAKE, FAKE, FAKE, FAKE, 220, FAKE, float("inf"), 0, FAKE, ws, stream=0)


def test_ragged_argument_checks(lib):
    """The ragged entry points check what the host sees (the length array's
    pointer, T_max, the rest as for the uniform calls); the lengths
    themselves live on the device and are checked by the kernels."""
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ws = L.workspace_bytes
    ok = dict(cache=FAKE, q=FAKE, sl=FAKE, T=256, out=FAKE, lse=0, ws=FAKE, ws_bytes=ws)
    for bad, code in ((dict(sl=0), 1), (dict(sl=FAKE + 2), 1), (dict(T=0), 1), (dict(T=257), 1),
                      (dict(cache=0), 1), (dict(q=FAKE + 8), 1), (dict(ws=0), 1),
                      (dict(ws_bytes=ws - 1), 3)):
        a = dict(ok)
        a.update(bad)
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_attention_ragged(L, a["cache"], a["q"], a["sl"], a["T"], a["out"], 0.1,
                                        a["lse"], a["ws"], a["ws_bytes"], stream=0)
        assert e.value.status == code, bad
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_step_ragged(L, a["cache"], a["q"], FAKE, FAKE, a["sl"], a["T"], a["out"], 0.1,
                                   a["lse"], a["ws"], a["ws_bytes"], stream=0)
        assert e.value.status == code, bad
    for kn, vn in ((0, FAKE), (FAKE, 0), (FAKE + 8, FAKE)):
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_step_ragged(L, FAKE, FAKE, kn, vn, FAKE, 256, FAKE, 0.1, 0, FAKE, ws, stream=0)
        assert e.value.status == 1


def test_corrupted_layout_rejected(lib):
    L = kvq.cache_layout(1, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    for field, val in (("total_bytes", 1), ("n_prot", 2), ("Tv", 5)):
        bad = kvq.Layout.from_buffer_copy(L)
        setattr(bad, field, val)
        with pytest.raises(kvq.KvqError) as e:
            kvq.decode_attention(bad, FAKE, FAKE, 10, FAKE, 0.1, 0, FAKE, 1 << 40, stream=0)
        assert e.value.status == 1
    bad = kvq.Layout.from_buffer_copy(L)
    bad.off[3] += 256
    with pytest.raises(kvq.KvqError):
        kvq.quantize_append(bad, FAKE, FAKE, FAKE, 0, 1, (128, 128, 128), stream=0)


def test_status_strings(lib):
    for code, name in kvq.STATUS.items():
        assert lib.kvq_status_string(code).decode() == name


def test_probe_argument_checks(lib):
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ws = kvq.probe_workspace_bytes(L, 256)
    assert ws > 0 and ws % 8 == 0
    assert kvq.probe_workspace_bytes(L, 0) == 0
    ok = dict(cache=FAKE, q=FAKE, k=FAKE, v=FAKE, strides=(4 * 256 * 128, 256 * 128, 128), T=200,
              R=FAKE, n_out=64, res=FAKE, ws=FAKE, ws_bytes=ws)
    for bad, code in ((dict(cache=0), 1), (dict(k=0), 1), (dict(v=FAKE + 4), 1), (dict(R=0), 1),
                      (dict(res=FAKE + 4), 1), (dict(ws=0), 1), (dict(T=0), 1), (dict(T=257), 1),
                      (dict(n_out=0), 1), (dict(n_out=2049), 1), (dict(strides=(8, 4, 128)), 1),
                      (dict(k=FAKE + 8), 1), (dict(R=FAKE + 4), 1),
                      (dict(cache=FAKE + 128), 1), (dict(ws_bytes=ws - 1), 3)):
        a = dict(ok)
        a.update(bad)
        st = lib.kvq_sensitivity_probe(ctypes.byref(L), a["cache"], a["q"], a["k"], a["v"],
                                       *a["strides"], a["T"], 0.1, a["R"], a["n_out"], a["res"],
                                       a["ws"], a["ws_bytes"], None)
        assert st == code, (bad, st)


def test_mq_argument_checks(lib):
    # text 0-9 and 200-255, visual 10-199
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    assert kvq.decode_mq_workspace_bytes(L, 1) == L.workspace_bytes
    assert kvq.decode_mq_workspace_bytes(L, 8) > L.workspace_bytes
    assert kvq.decode_mq_workspace_bytes(L, 0) == 0
    assert kvq.decode_mq_workspace_bytes(L, kvq.KVQ_MAX_QUERY_TOKENS + 1) == 0
    ws4 = kvq.decode_mq_workspace_bytes(L, 4)
    ok = dict(n_q=4, T=256, ws_bytes=ws4)
    for bad, code in ((dict(n_q=0), 1), (dict(n_q=kvq.KVQ_MAX_QUERY_TOKENS + 1), 1),
                      (dict(T=3), 1), (dict(T=257), 1),
                      (dict(T=202), 1),   # token 0 would not see positions 199..201: 199 is visual
                      (dict(ws_bytes=ws4 - 1), 3)):
        a = dict(ok)
        a.update(bad)
        st = lib.kvq_decode_attention_mq(ctypes.byref(L), FAKE, FAKE, a["n_q"], a["T"], 0.1, FAKE, None,
                                         FAKE, a["ws_bytes"], None)
        assert st == code, (bad, st)
    # an empty visual range leaves every position text: no constraint on T
    L0 = kvq.cache_layout(2, 8, 4, 128, 256, 10, 10, 4, 4, 32, [])
    st = lib.kvq_decode_attention_mq(ctypes.byref(L0), FAKE, FAKE, 4, 12, 0.1, FAKE, None, FAKE,
                                     kvq.decode_mq_workspace_bytes(L0, 4) - 1, None)
    assert st == 3  # past the position check, stopped by the workspace size


def test_concurrent_argument_checks_from_two_threads(lib):
    """Decode entry points keep no process-wide state: calls from several
    host threads run at once (ctypes releases the GIL) and each gets its own
    status, with no lock between them."""
    import threading
    L = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
    ws = L.workspace_bytes
    errors = []

    def worker(kind, n):
        try:
            for i in range(n):
                if kind == 0:  # T out of range -> KVQ_ERR_INVALID_ARG
                    with pytest.raises(kvq.KvqError) as e:
                        kvq.decode_attention(L, FAKE, FAKE, 257, FAKE, 0.1, 0, FAKE, ws, stream=0)
                    assert e.value.status == 1
                elif kind == 1:  # workspace too small -> KVQ_ERR_CAPACITY
                    with pytest.raises(kvq.KvqError) as e:
                        kvq.decode_step(L, FAKE, FAKE, FAKE, FAKE, 220, FAKE, 0.1, 0, FAKE, ws - 1, stream=0)
                    assert e.value.status == 3
                else:  # layouts built concurrently agree with one built alone
                    L2 = kvq.cache_layout(2, 8, 4, 128, 256, 10, 200, 4, 4, 32, [1])
                    assert L2.workspace_bytes == ws and L2.total_bytes == L.total_bytes
        except BaseException as exc:  # noqa: BLE001 -- reported below
            errors.append((kind, repr(exc)))

    threads = [threading.Thread(target=worker, args=(k, 2000)) for k in (0, 1, 2, 0, 1)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors[:3]
