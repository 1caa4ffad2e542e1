"""The synthetic inputs, on the CPU: the recipe the workloads are built from (structure the
pages fix: a (frame, row, column) token grid with neighbouring tokens numerically close,
keys reaching |x| ~ 1e2 and values ~ 1e3 through a few outlier channels) and the
properties the tests and the benchmark rely on (seeded, batch- and chunk-independent)."""
import numpy as np
import pytest
import torch

from video_kv_cache_gb300 import synth


@pytest.fixture(scope="module")
def kv():
    # one key and one value tensor of 3 frames of 30 x 52 tokens
    return synth.kv_tensor(7, [0, 1], 0, 3, 30, 52, torch.float32, "cpu")


def test_seeded_and_independent_of_batching():
    a = synth.kv_tensor(3, [0, 1, 2, 3], 0, 1, 8, 9, torch.bfloat16)
    b = synth.kv_tensor(3, [0, 1, 2, 3], 0, 1, 8, 9, torch.bfloat16, batch=1)
    c = synth.kv_tensor(3, [2], 0, 1, 8, 9, torch.bfloat16)
    assert torch.equal(a, b) and torch.equal(a[2:3], c)
    assert not torch.equal(a, synth.kv_tensor(4, [0, 1, 2, 3], 0, 1, 8, 9, torch.bfloat16))


def test_a_chunk_is_a_slice_of_the_whole_clip():
    whole = synth.kv_tensor(5, [0, 1], 0, 6, 10, 12, torch.float32)
    part = synth.kv_tensor(5, [0, 1], 3, 2, 10, 12, torch.float32)
    sl = whole[:, 3 * 120:5 * 120]
    # the noise is a counter hash (exact); the field is recomputed per token in fp32
    np.testing.assert_allclose(part.numpy(), sl.numpy(), rtol=0, atol=1e-3)


def test_outlier_channels(kv):
    for t, (lo, hi, clip) in enumerate(((60.0, 90.0, 100.0), (600.0, 900.0, 1000.0))):
        x = kv[t].double()
        m = x.mean(dim=0).abs()
        out = torch.nonzero(m > 20.0 * (10 if t else 1)).flatten()
        assert len(out) == synth.N_OUTLIERS, (t, m.topk(6))
        # A_k + 10 z_k: the mean sits near A_k within the field's spread
        assert ((m[out] > lo - 15 * (10 if t else 1)) & (m[out] < hi + 15 * (10 if t else 1))).all()
        assert x.abs().max() <= clip
        rest = torch.ones(128, dtype=torch.bool)
        rest[out] = False
        assert x[:, rest].abs().max() < 0.1 * clip


def test_ordinary_channels_are_unit_scale_and_smooth(kv):
    x = kv[0].double().reshape(3, 30, 52, 128)
    m = x.mean(dim=(0, 1, 2)).abs()
    ordinary = m < 20.0
    sd = x[..., ordinary].std(dim=(0, 1, 2))
    assert 0.5 < float(sd.mean()) < 1.5
    # neighbours along a row are close (squared-exponential length 6 tokens), tokens 20
    # columns apart far less so
    z = x[..., ordinary] - x[..., ordinary].mean(dim=(0, 1, 2))

    def corr(a, b):
        return float((a * b).sum() / torch.sqrt((a * a).sum() * (b * b).sum()))

    near = corr(z[:, :, :-1], z[:, :, 1:])
    far = corr(z[:, :, :-20], z[:, :, 20:])
    assert near > 0.9 and far < 0.5 * near


def test_values_are_keys_scaled_by_ten():
    # odd tensor ids are values: the key construction scaled by 10 and clipped at 1000
    k = synth.kv_tensor(9, [4], 0, 1, 6, 7, torch.float32)
    assert float(k.abs().max()) <= 100.0
    v = synth.kv_tensor(9, [5], 0, 1, 6, 7, torch.float32)
    assert 100.0 < float(v.abs().max()) <= 1000.0


def test_rounding_to_16_bits_is_nearest_even():
    x32 = synth.kv_tensor(11, [0, 1], 0, 1, 9, 10, torch.float32)
    for dt in (torch.bfloat16, torch.float16):
        x16 = synth.kv_tensor(11, [0, 1], 0, 1, 9, 10, dt)
        assert torch.equal(x16, x32.to(dt))


@pytest.mark.parametrize("name,H,N,C,T", [
    ("single_head_4x32x32", 1, 4096, 64, 1), ("layer_1p3b_32760", 24, 32760, 256, 2),
    ("dit13b_65536", 64, 65536, 256, 4), ("stream_30x12_60chunk", 720, 280800, 256, 2)])
def test_workload_shapes(name, H, N, C, T):
    w = synth.workload(name)
    assert (w.H, w.N, w.C, w.T) == (H, N, C, T)
    # tensor ids interleave keys and values: (layer, head, K/V) -> 2 (layer heads + head) + kv
    assert w.tids[:4] == list(range(min(4, w.H)))
    assert synth.tensor_id(1, 2, 1, w.heads) == 2 * (w.heads + 2) + 1


def test_stream_chunks():
    w = synth.workload("stream_30x12_60chunk")
    assert w.chunk_frames * w.gh * w.gw == 4680 and w.frames // w.chunk_frames == 60
    assert w.iters == 10 and w.warm_iters == 2
