"""The seeded input generator: published SplitMix64 values and moments of its laws."""
import numpy as np

import synth
from synth import workloads


def test_splitmix64_published_sequence():
    # SplitMix64 started from state 0 (Steele, Lea, Flood 2014): first three outputs.
    z = 0
    out = []
    for _ in range(3):
        z = (z + synth.GAMMA) & synth.MASK64
        out.append(synth.mix64_int(z))
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # the vectorised finaliser agrees with the scalar one
    zs = np.array([synth.GAMMA, 2 * synth.GAMMA & synth.MASK64], dtype=np.uint64)
    assert synth._mix64(zs).tolist() == out[:2]


def test_normal_moments_and_bounds():
    v = synth.normal(0, synth.TID_TEST, (1 << 20,), 1.0, "f32").astype(np.float64)
    assert abs(v.mean()) < 4 * (1 / 1024)
    assert abs(v.var() - 1.0) < 0.01
    assert np.abs(v).max() <= 6.0
    # scaled + bf16 draws are the rounded float32 draws
    b = synth.normal(0, synth.TID_TEST, (4096,), 0.5, "bf16")
    f = synth.normal(0, synth.TID_TEST, (4096,), 0.5, "f32")
    assert np.array_equal(b, synth.f32_to_bf16_bits(f))
    # slices address the same elements
    s = synth.normal(0, synth.TID_TEST, (100,), 1.0, "f32", start=1000)
    assert np.array_equal(s, synth.normal(0, synth.TID_TEST, (1100,), 1.0, "f32")[1000:])


def test_uniform_range():
    u = synth.uniform(0, synth.TID_SEL_BIAS, 1 << 16, -0.1, 0.1)
    assert u.min() >= -0.1 and u.max() < 0.1
    assert abs(u.mean()) < 0.002


def test_uniform_topk_ids_are_subsets():
    ids = synth.uniform_topk_ids(1, synth.TID_TEST, 64, 32, 5)
    assert ids.shape == (64, 5)
    for row in ids:
        assert len(set(row.tolist())) == 5
    freq = np.bincount(synth.uniform_topk_ids(2, synth.TID_TEST, 4000, 8, 2).reshape(-1), minlength=8)
    assert np.abs(freq / freq.sum() - 1 / 8).max() < 0.02


def test_zipf_offsets_skew():
    """Offsets that make argmax(z + o), z ~ N(0, I), follow Zipf(1.1) over 128 experts:
    the hottest expert takes > 20x the mean load."""
    E = 128
    o = workloads.host_logit_offset(workloads.SWITCH)
    z = synth.normal(1, synth.TID_TEST, (1 << 15, E), 1.0, "f32").astype(np.float64)
    freq = np.bincount(np.argmax(z + o, axis=1), minlength=E) / z.shape[0]
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    assert abs(freq[0] - p[0]) < 0.01
    assert freq[0] * E > 20


def test_c_host_generator_matches_numpy_definition():
    for dtype, sigma in (("f32", 1.0), ("bf16", 1.0 / 84.66), ("f32", 0.037)):
        start = (1 << 33) + 12345            # beyond 32-bit element indices
        a = synth.normal(0, synth.TID_W13, (5000,), sigma, dtype, start=start, use_c=True)
        b = synth.normal(0, synth.TID_W13, (5000,), sigma, dtype, start=start, use_c=False)
        assert a.dtype == b.dtype and np.array_equal(a, b)
