"""kvq_decode_attention_mq (several query tokens per sequence) against the
CPU oracle: token i of sequence b is an ordinary decode query over positions
[0, T - n_q + 1 + i), so the oracle runs once per token.  Bar as for the
single-query decode (4e-3 * max|V_hat|); n_q = 1 gives the same bits as
kvq_decode_attention.  Calls run on the split-KV kernel (one pass per 8
(query head, token) columns of a KV head) unless there are at least 32
(sequence, KV head) pairs and >= 128 columns per KV head, or >= 32 columns
with T <= 2048 -- then on the tensor-core (tcgen05) kernel (one pass per 128
columns); the cases cover both."""
import math

import pytest
import torch

import bit_mixed_precision_kvq_gb300 as kvq
import synth
from gpu_helpers import Case, alloc_cache, append, bits, check_decode, decode, oracle_decode

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


def _q(c: Case, n_q: int, seed: int, dev):
    x = synth.normal(c.B * n_q * c.H_q * c.D, synth.stream_key(seed, 7), dev)
    return synth.to_bf16(x.view(c.B, n_q, c.H_q, c.D))


def _mq(L, cache, q, T):
    B, n_q, Hq, D = q.shape
    out = torch.full((B, n_q, Hq, D), 5.0, dtype=torch.bfloat16, device=q.device)
    lse = torch.zeros((B, n_q, Hq), dtype=torch.float32, device=q.device)
    ws = torch.full((kvq.decode_mq_workspace_bytes(L, n_q),), 0x3C, dtype=torch.uint8, device=q.device)
    kvq.decode_attention_mq(L, cache, q, T, out, SCALE, lse, ws)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # layout, n_q, T
    (Case(1, 28, 4, 700, 14, 640, 4, 2, 64, [0]), 2, 700),                # g = 7: 14 columns, 2 units
    (Case(1, 28, 4, 700, 14, 640, 4, 2, 64, [0]), 4, 690),
    (Case(2, 8, 8, 300, 10, 250, 8, 4, 32, [1], konly=[2]), 8, 300),      # MHA: 8 tokens fill N = 8
    (Case(2, 32, 8, 500, 32, 400, 2, 2, 32, [3]), 3, 480),                # g = 4: 12 columns
    (Case(3, 4, 2, 64, 20, 40, 4, 4, 64, []), 5, 5),                      # all in the text prefix
    (Case(1, 4, 4, 400, 16, 300, 2, 4, 32, [0]), 64, 400),                # g = 1, 64 tokens: 8 units
    (Case(2, 16, 2, 2500, 30, 2400, 4, 2, 64, [], konly=[1]), 6, 2450),   # long history, K-only head
    (Case(16, 16, 16, 130, 10, 120, 4, 2, 32, [3]), 8, 130),              # 256 units: stream-cut plan
    # tensor-core kernel: 64 (b, KV head) pairs, g = 4, 8 tokens = 32 columns, short history
    (Case(8, 32, 8, 600, 10, 560, 2, 2, 32, [3]), 8, 600),
    # tensor-core kernel: 32 pairs, 32 tokens = 128 columns, T > 2048, K-only head
    (Case(4, 32, 8, 2300, 16, 2200, 4, 2, 64, [1], konly=[5]), 32, 2300),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_mq_matches_oracle_per_token(cuda_dev, kvq, ci):
    c, n_q, T = CASES[ci]
    L = c.layout()
    _, k, v = synth.random_case(1700 + ci, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    q = _q(c, n_q, 1710 + ci, cuda_dev)
    out, lse = _mq(L, cache, q, T)
    kb, vb = bits(k), bits(v)
    for i in range(n_q):
        ref, lr, vmax = oracle_decode(c, bits(q[:, i].contiguous()), kb, vb, T - n_q + 1 + i, SCALE)
        check_decode(c, out[:, i], lse[:, i], ref, lr, vmax)


def test_mq_single_token_is_plain_decode(cuda_dev, kvq):
    c = Case(2, 28, 4, 900, 14, 850, 4, 2, 64, [0])
    L = c.layout()
    _, k, v = synth.random_case(1750, c.B, c.H_q, c.H_kv, c.D, c.T_cap, cuda_dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    q = _q(c, 1, 1751, cuda_dev)
    assert kvq.decode_mq_workspace_bytes(L, 1) == L.workspace_bytes
    for T in (900, 300):
        out, lse = _mq(L, cache, q, T)
        out1, lse1 = decode(L, cache, q[:, 0].contiguous(), T, SCALE)
        assert torch.equal(out[:, 0].view(torch.int16), out1.view(torch.int16)), T
        assert torch.equal(lse[:, 0], lse1), T


def _full_check(c, n_q, T, seed, dev, b_sel=None):
    L = c.layout()
    _, k, v = synth.random_case(seed, c.B, c.H_q, c.H_kv, c.D, c.T_cap, dev)
    cache = alloc_cache(L)
    append(L, cache, k, v, 0)
    q = _q(c, n_q, seed + 1, dev)
    ws = torch.zeros((kvq.decode_mq_workspace_bytes(L, n_q),), dtype=torch.uint8, device=dev)
    B, _, Hq, D = q.shape
    out = torch.full((B, n_q, Hq, D), 5.0, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((B, n_q, Hq), dtype=torch.float32, device=dev)
    kvq.decode_attention_mq(L, cache, q, T, out, SCALE, lse, ws)
    torch.cuda.synchronize()
    assert kvq.workspace_status(ws) == 0
    kb, vb = bits(k), bits(v)
    for i in range(n_q):
        ref, lr, vmax = oracle_decode(c, bits(q[:, i].contiguous()), kb, vb, T - n_q + 1 + i, SCALE)
        check_decode(c, out[:, i], lse[:, i], ref, lr, vmax)


def test_mq_llava_ov_4_tokens(cuda_dev, kvq):
    """The LLaVA-OneVision-7B layer shape (28/4 heads, 14 text + 6273 visual
    positions + 4 new text rows, K4/V2 G64, head 0 bf16) with 4 query
    tokens: 28 columns per KV head in one tensor-core pass."""
    T = 14 + 6273 + 4
    _full_check(Case(1, 28, 4, T, 14, 14 + 6273, 4, 2, 64, [0]), 4, T, 1800, cuda_dev)


def test_mq_llava_ov_64_tokens(cuda_dev, kvq):
    """64 query tokens on the same layout: 448 columns per KV head, four
    128-column units per head."""
    T = 14 + 1200 + 64
    _full_check(Case(1, 28, 4, T, 14, 14 + 1200, 4, 2, 64, [0]), 64, T, 1820, cuda_dev)
