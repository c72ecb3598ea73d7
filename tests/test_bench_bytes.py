"""The algorithmic bytes bench.py divides by (its roofline and GB/s), against a
position-by-position count from the documented layout: every attended
position of every (b, KV head) costs the cache rows the decode must read --
bf16 K and V rows (2 x 256 B) for text positions and protected heads, bf16 K
plus the packed V row and its scale/zero for K-only heads, the packed K and V
rows and their scales/zeros for the other heads -- and q and out cost 2 x 256 B
per (b, token, query head).  No GPU needed."""
import pytest

import bench
import bit_mixed_precision_kvq_gb300 as kvq
from bit_mixed_precision_kvq_gb300 import build_native


@pytest.fixture(scope="module")
def lib():
    build_native.build()
    return kvq.load()


def _count(B, Hq, Hkv, T, vs, ve, kb, vb, G, prot, konly, n_q):
    D = 128
    packed_k = D * kb // 8 + (4 * D // G if kb < 16 else 0)
    packed_v = D * vb // 8 + (4 * D // G if vb < 16 else 0)
    total = 0
    for _b in range(B):
        for h in range(Hkv):
            for t in range(T):
                if not vs <= t < ve or h in prot:
                    total += 2 * 2 * D
                elif h in konly:
                    total += 2 * D + packed_v
                else:
                    total += packed_k + packed_v
    return total + 2 * B * n_q * Hq * D * 2


CASES = [
    # B, Hq, Hkv, T_cap, vs, ve, kb, vb, G, prot, konly, T, n_q
    (1, 28, 4, 700, 14, 640, 4, 2, 64, [0], [], 700, 1),
    (2, 16, 4, 300, 20, 290, 8, 4, 32, [1], [2], 297, 1),
    (3, 8, 8, 200, 10, 150, 2, 16, 128, [], [5, 6], 120, 4),   # T inside the visual range
    (2, 32, 8, 500, 32, 400, 16, 2, 32, [3], [], 31, 2),       # T inside the text prefix
]


@pytest.mark.parametrize("case", CASES)
def test_decode_bytes_match_position_count(lib, case):
    B, Hq, Hkv, Tc, vs, ve, kb, vb, G, prot, konly, T, n_q = case
    L = kvq.cache_layout(B, Hq, Hkv, 128, Tc, vs, ve, kb, vb, G, prot, konly)
    assert bench.decode_bytes(L, T, n_q) == _count(B, Hq, Hkv, T, vs, ve, kb, vb, G, prot, konly, n_q)


def test_append_bytes(lib):
    L = kvq.cache_layout(2, 8, 4, 128, 100, 10, 90, 4, 4, 32, [1])
    # the step's bf16 K and V rows are read and written once: 2 x (B H_kv n 2 x 256 B)
    assert bench.append_bytes(L, 3) == 2 * (2 * 4 * 3 * 2 * 256)
