"""The seeded input generators: deterministic, with the stated shapes and ranges."""
import numpy as np

from fgp_dual_stencil_gb300 import synth


def test_workload_table():
    w = synth.WORKLOADS
    assert [w[k].shape for k in ("c1", "c2", "c3", "c4", "c5")] == [
        (32, 32, 32), (128, 128, 128), (256, 256, 256), (512, 512, 512), (1000, 600, 300)]
    assert [w[k].total_steps for k in ("c1", "c2", "c3", "c4", "c5")] == [10, 50, 200, 200, 100]
    assert [w[k].lam for k in ("c1", "c2", "c3", "c4", "c5")] == [0.05, 0.03, 0.02, 0.02, 0.1]
    assert w["c4"].phantom_seed == w["c3"].phantom_seed


def test_deterministic_and_shaped():
    w = synth.WORKLOADS["c1"]
    a = synth.make_b(w, 0)
    b = synth.make_b(w, 0)
    assert a.dtype == np.float32 and a.shape == (32, 32, 32) and a.flags.c_contiguous
    assert np.array_equal(a, b)
    assert not np.array_equal(a, synth.make_b(w, 1))      # fresh noise per outer


def test_ellipsoid_ranges():
    ph = synth.phantom(synth.WORKLOADS["c1"])
    vals = np.unique(ph)
    assert vals[0] == 0.0 and np.all((vals[1:] >= 0.2) & (vals[1:] <= 1.0))
    ph2 = synth.phantom(synth.WORKLOADS["c2"])
    assert ph2.max() > 1.0                                  # additive overlap reaches above 1
    ph3 = synth.ellipsoids((64, 64, 64), 10, np.random.default_rng(0), value_range=(0, 1),
                           semi_range=(0.05, 0.4))
    assert 0.0 <= ph3.min() and ph3.max() <= 1.0


def test_blobs_small():
    rng = np.random.default_rng(1)
    vol = synth.gaussian_blobs((100, 60, 30), 5, rng, sigma_range=(3, 6), peak_range=(0.5, 2.0))
    assert vol.min() >= 0.0 and 0.4 < vol.max() <= 2.0 * 5
    assert (vol == 0).mean() > 0.3


def test_scaled_phantom_is_the_same_shape_of_objects():
    """The 512^3 phantom is the 256^3 one drawn from the same seed in relative
    coordinates; downsampling it by 2 reproduces most voxels."""
    small = synth.ellipsoids((32, 32, 32), 10, np.random.default_rng([5, 0]), value_range=(0, 1),
                             semi_range=(0.05, 0.4))
    big = synth.ellipsoids((64, 64, 64), 10, np.random.default_rng([5, 0]), value_range=(0, 1),
                           semi_range=(0.05, 0.4))
    assert (big[::2, ::2, ::2] == small).mean() > 0.9
