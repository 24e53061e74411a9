"""The seeded input generator: published SplitMix64 vectors, determinism,
distribution and the platform-independent series functions.  CPU only."""
import math

import numpy as np

import synth


def test_splitmix64_published_vector():
    # SplitMix64 seeded with 1234567: the first five outputs of the reference
    # generator (Vigna's splitmix64.c) are these.
    G, M = 0x9E3779B97F4A7C15, (1 << 64) - 1
    x, got = 1234567, []
    for _ in range(5):
        x = (x + G) & M
        got.append(synth.mix64(x))
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_series_functions_match_libm():
    for x in (1e-300, 1e-9, 0.1, 0.3, 0.5, 0.7071, 0.99999, 1.0):
        assert math.isclose(synth.series_log(x), math.log(x), rel_tol=2e-15, abs_tol=1e-16)
    for x in np.linspace(-math.pi, math.pi, 101):
        s, c = synth.series_sincos(float(x))
        assert abs(s - math.sin(x)) < 1e-14 and abs(c - math.cos(x)) < 1e-14


def test_counter_based_and_offsets():
    a = synth.normal_bf16(5, 9, (4096,), 0.02)
    b = synth.normal_bf16(5, 9, (100,), 0.02, offset=1001)
    assert np.array_equal(a[1001:1101], b)
    assert not np.array_equal(a, synth.normal_bf16(5, 10, (4096,), 0.02))
    assert not np.array_equal(a, synth.normal_bf16(6, 9, (4096,), 0.02))


def test_normal_moments():
    x = synth.normal_bf16(1, 2, (1 << 20,), 0.02)
    f = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(f.mean()) < 1e-4
    assert abs(f.std() - 0.02) < 2e-4
    assert 0.0020 < np.mean(np.abs(f) > 3 * 0.02) < 0.0034   # 2-sided 3-sigma tail 0.0027


def test_transform_diagonal():
    T = synth.normal_bf16(1, 3, (64, 64), 0.01, diag_add=1.0)
    f = (T.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(np.diag(f) - 1) < 0.06)
    off = f[~np.eye(64, dtype=bool)]
    assert abs(off.std() - 0.01) < 1e-3


def test_uniform_ints_range_and_spread():
    x = synth.uniform_int(3, 4, 100000, 256, 2048)
    assert x.min() >= 256 and x.max() <= 2048
    assert abs(x.mean() - 1152) < 10


def test_workloads():
    w = synth.WORKLOADS["llama3.1-8b-b1"]
    assert w.checkpoints == (4, 8, 12, 16, 20, 24, 28)
    assert synth.WORKLOADS["llama3.2-1b-b1"].checkpoints == (4, 8, 12)
    assert synth.WORKLOADS["codellama-34b-b8"].checkpoints == (8, 16, 24, 32, 40)
    assert synth.WORKLOADS["tiny-b1"].checkpoints == (1, 2)
    lens, pr = synth.workload_inputs(synth.WORKLOADS["llama3.1-8b-b32"])
    assert len(pr) == 32 and all(256 <= n <= 2048 for n in lens)
