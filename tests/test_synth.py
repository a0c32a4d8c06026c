"""The seeded input generator: host and torch paths agree bit for bit."""
import numpy as np
import pytest
import torch

import synth
from synth import workloads


def test_splitmix64_known_values():
    # SplitMix64 reference sequence for state 0 (first outputs of the published
    # generator): 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F.
    z = [synth._mix_py((i + 1) * synth.GOLDEN) for i in range(3)]
    assert z == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


@pytest.mark.parametrize("kind", synth.KINDS)
def test_numpy_and_torch_paths_agree(kind):
    n = 100003
    a = synth.buffer_np(kind, 17, n)
    b = synth.buffer_torch(kind, 17, n, "cpu", chunk=4099).numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    idx = np.array([0, 5, 99999, 100002], dtype=np.uint64)
    assert np.array_equal(synth.values_np(kind, 17, idx).view(np.uint16),
                          a[idx.astype(np.int64)].view(np.uint16))


def test_distributions():
    u = synth.buffer_np("uniform", 3, 200000).astype(np.float64)
    assert u.min() >= -1.0 and u.max() <= 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    i = synth.buffer_np("int3", 3, 70000).astype(np.float64)
    vals, counts = np.unique(i, return_counts=True)
    assert list(vals) == [-3, -2, -1, 0, 1, 2, 3]
    assert counts.min() > 9000
    assert not np.array_equal(synth.buffer_np("uniform", 4, 100), synth.buffer_np("uniform", 5, 100))


def test_workload_views_and_strides():
    w = workloads.TAIL_TRANSPOSED_B
    assert w.B.strides == (1, 65) and w.B.buf_shape == (70, 65)
    hv = w.B.host_view()
    assert hv.shape == (65, 70) and hv.strides == (2, 130)
    dv = w.B.device_view("cpu")
    assert tuple(dv.shape) == (65, 70) and tuple(dv.stride()) == (1, 65)
    assert np.array_equal(dv.numpy().view(np.uint16), hv.view(np.uint16))
    r = np.array([0, 64, 3]); c = np.array([69, 0, 5])
    assert np.array_equal(w.B.values_at(r, c).view(np.uint16), hv[r, c].view(np.uint16))
    w4 = workloads.IRREGULAR_3001x1999x4097
    assert w4.A.strides == (1, 3001)
