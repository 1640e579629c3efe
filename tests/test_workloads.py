"""The seeded input generators: shapes and sizes of the DGC review's workloads (CPU only)."""
import math

import numpy as np

import workloads


def test_resnet50_layout_matches_97mb():
    # DGC review, Abstract: ResNet-50's gradient is 97 MB. 161 tensors, 25,557,032 binary32
    # entries = 102,228,128 bytes = 97.5 MiB.
    shapes = workloads.resnet50_shapes()
    assert len(shapes) == 161
    n = sum(math.prod(s) for _, s in shapes)
    assert n == 25_557_032
    assert round(n * 4 / 2**20) == 97
    off = workloads.resnet50_segments()
    sizes = np.diff(off)
    assert sizes.max() == 512 * 512 * 9
    assert int((np.ceil(sizes / 1000) == 1).sum()) == 85  # tensors where 0.1% rounds up to 1


def test_deepspeech_layout_is_488mb():
    off = workloads.deepspeech_segments()
    assert off[-1] == 122_000_000 and len(off) == 7


def test_generators_are_deterministic_and_chunked():
    a = workloads.gradient("single", 3)
    b = workloads.gradient("single", 3)
    c = workloads.gradient("single", 4)
    assert a.dtype == np.float32 and a.size == 1_048_576
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert abs(float(a.std()) - 0.01) < 2e-4
    # a larger draw with the same words extends the smaller one chunk by chunk
    x = workloads.normal([9, 1], workloads.CHUNK + 10, 1.0)
    y = workloads.normal([9, 1], workloads.CHUNK, 1.0)
    assert np.array_equal(x[:workloads.CHUNK], y)


def test_bucket_outliers_fixed_per_seed():
    n = 1 << 20
    p1 = workloads.outlier_positions(n, 0)
    p2 = workloads.outlier_positions(n, 0)
    assert np.array_equal(p1, p2) and p1.size == round(1e-4 * n)
    assert np.unique(p1).size == p1.size
    g0 = workloads.gradient("bucket1g", 0, n=n)
    g1 = workloads.gradient("bucket1g", 1, n=n)
    assert np.abs(g0[p1]).mean() > 50 * np.abs(g0).mean()
    assert not np.array_equal(g0, g1)
