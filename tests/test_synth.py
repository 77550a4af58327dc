"""The seeded generators: reproducible, and the vectorised SplitMix64 equals
the plain-integer definition."""
import numpy as np

import synth


def test_splitmix_vectorised_equals_scalar():
    for seed in (0, 1, 0x57A70000, (1 << 64) - 1):
        assert synth.splitmix64(seed, 50).tolist() == synth.splitmix64_scalar(seed, 50)


def test_generators_are_deterministic():
    a = synth.frames_uniform(9, 2, 5, 7)
    b = synth.frames_uniform(9, 2, 5, 7)
    assert np.array_equal(a, b) and a.shape == (2, 5, 21)
    assert not np.array_equal(a[0], a[1])
    assert np.array_equal(synth.normal(3, 101), synth.normal(3, 101))


def test_distributions_are_plausible():
    z = synth.normal_f64(5, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    u = synth.uniform_bytes(6, 1 << 18)
    counts = np.bincount(u, minlength=256)
    assert counts.min() > 800 and counts.max() < 1250
    s = synth.scores_logistic(7, 10000)
    assert s.min() > 0 and s.max() < 1 and 0.015 < np.median(s) < 0.021   # sigma(-4) = 0.018


def test_ties_are_planted():
    x = synth.logits_with_ties(8, 2, 20000)
    for r in range(2):
        dup = 20000 - np.unique(x[r]).size
        assert 500 < dup < 1500          # about 5 % of the entries repeat another


def test_gradient_frame_shape_and_range():
    f = synth.frames_gradient_noise(1, 1, 9, 16)
    assert f.shape == (1, 9, 48) and f.dtype == np.uint8


def test_clustered_candidates():
    a = synth.clustered_candidates(4, 10, 6, num_classes=5)
    b = synth.clustered_candidates(4, 10, 6, num_classes=5)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    assert a["boxes"].shape == (60, 4) and a["boxes"].dtype == np.float32
    assert np.unique(a["anchors"]).size == 60 and a["anchors"].max() < 8400
    assert all(np.unique(a["classes"][i * 6:(i + 1) * 6]).size == 1 for i in range(10))
    assert np.all(a["boxes"][:, 2] > a["boxes"][:, 0])    # jitter small against the side
