"""The synthetic inputs against the five workload descriptions they stand in
for (shapes, bits, protected heads, the structure of K), and the property
the parity tests rely on: every (b, h) row is its own random stream, so a
slice of the batch or heads equals the same slice of the full tensor.  CPU."""
import numpy as np
import pytest
import torch

import synth

# name, layers, B, H_q, H_kv, text prefix, visual, G, (k_bits, v_bits) of layer 0 / of the last layer,
# protected heads per layer
SHAPES = [
    ("tiny", 1, 1, 4, 1, 14, 242, 32, (4, 4), (4, 4), 0),
    ("llava_ov_7b", 28, 1, 28, 4, 14, 6273, 64, (4, 2), (4, 2), 1),
    ("llava15_7b", 32, 16, 32, 32, 40, 576, 32, (8, 4), (8, 4), 4),
    ("llava_next_13b", 40, 32, 40, 40, 60, 2880, 64, (8, 8), (4, 2), 5),
]


@pytest.mark.parametrize("case", SHAPES, ids=[c[0] for c in SHAPES])
def test_workload_shapes(case):
    name, L, B, Hq, Hkv, n_text, n_vis, G, bits0, bits_last, n_prot = case
    w = synth.workload(name)
    assert (w.n_layers, w.B, w.H_q, w.H_kv, w.D) == (L, B, Hq, Hkv, 128)
    assert (w.vis_start, w.vis_end, w.T) == (n_text, n_text + n_vis, n_text + n_vis)
    assert w.group_size == G
    assert (w.layers[0].k_bits, w.layers[0].v_bits) == bits0
    assert (w.layers[-1].k_bits, w.layers[-1].v_bits) == bits_last
    for ls in w.layers:
        assert len(ls.protected) == n_prot and len(set(ls.protected)) == n_prot
        assert all(0 <= h < Hkv for h in ls.protected)
    if name == "llava_ov_7b":
        assert all(ls.protected == [0] for ls in w.layers)
    if name == "llava_next_13b":  # layers 0-3 K8/V8, the rest K4/V2
        assert all((ls.k_bits, ls.v_bits) == ((8, 8) if i < 4 else (4, 2)) for i, ls in enumerate(w.layers))


@pytest.mark.parametrize("T", [1024, 4096, 16384, 32768])
def test_longctx_shapes(T):
    w = synth.workload("longctx", T)
    assert (w.n_layers, w.B, w.H_q, w.H_kv, w.T, w.vis_start, w.vis_end) == (1, 8, 32, 8, T, 32, T)
    assert (w.layers[0].k_bits, w.layers[0].v_bits, w.group_size) == (2, 2, 32)
    assert len(w.layers[0].protected) == 1


def test_slices_equal_full_tensor():
    w = synth.workload("llava15_7b")
    full = synth.make_kv(w, 3, "k", T=40)
    part = synth.make_kv(w, 3, "k", b_range=[2, 7], h_range=[5, 0, 31], T=40)
    assert torch.equal(part, full[[2, 7]][:, [5, 0, 31]])
    again = synth.make_kv(w, 3, "k", T=40)
    assert torch.equal(full, again)  # seeded: the same call gives the same bits


def test_k_outlier_channels_without_rope():
    """LLaVA-Next-shaped K: 4 channels per (layer, head) scaled x10, the rest
    N(0, 1) (the outliers of the LLaVA-OV recipe without its RoPE)."""
    w = synth.workload("llava_next_13b")
    k = synth.make_kv(w, 0, "k", b_range=[0], h_range=[0, 1], T=2000).float()
    for h in range(2):
        rms = k[0, h].pow(2).mean(0).sqrt().numpy()
        big = np.sort(np.argsort(rms)[-4:])
        assert np.all(rms[big] > 7.0) and np.all(np.delete(rms, big) < 1.3), rms[big]
    v = synth.make_kv(w, 0, "v", b_range=[0], h_range=[0], T=2000).float()
    assert v[0, 0].pow(2).mean(0).sqrt().max() < 1.3  # V has no outliers


def test_k_outliers_rotate_with_rope():
    """LLaVA-OV-shaped K: RoPE mixes channel d with d + 64, so the outlier
    energy sits in up to 4 channel pairs (d, d + 64) whose summed mean
    square is ~100 per outlier."""
    w = synth.workload("llava_ov_7b")
    k = synth.make_kv(w, 0, "k", b_range=[0], h_range=[1], T=3000).float()
    ms = k[0, 0].pow(2).mean(0).numpy()
    pair = ms[:64] + ms[64:]
    big = np.argsort(pair)[-4:]
    assert pair[big].sum() > 300.0 and np.all(np.delete(pair, big) < 3.0), pair[big]


def test_lognormal_channel_magnitudes():
    """LLaVA-1.5-shaped K: per-channel magnitude exp(N(0, 0.5^2)) times N(0, 1):
    log of the channel RMS has standard deviation ~0.5 across channels."""
    w = synth.workload("llava15_7b")
    k = synth.make_kv(w, 0, "k", b_range=[0], h_range=[4], T=4000).float()
    lr = np.log(k[0, 0].pow(2).mean(0).sqrt().numpy())
    assert 0.35 < lr.std() < 0.65, lr.std()


def test_longctx_outliers_x8():
    """Long-context K: round(0.02 * 128) = 3 channels per head scaled x8."""
    w = synth.workload("longctx", 1024)
    k = synth.make_kv(w, 0, "k", b_range=[0], h_range=[2], T=1024).float()
    rms = k[0, 0].pow(2).mean(0).sqrt().numpy()
    big = np.argsort(rms)[-3:]
    assert np.all(rms[big] > 6.0) and np.all(np.delete(rms, big) < 1.3)
