"""The seeded synthetic inputs against their recipe (CPU): the counter-form
SplitMix64 stream (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) reproduces the generator's published first
outputs, and the uniforms, normals, classes, initialisers and workload
shapes have the stated distributions and sizes."""
import math

import numpy as np
import pytest

from static_graph_nn_gb300 import workloads as W

# first five outputs of SplitMix64 seeded with 1234567, as printed with the
# generator's reference implementation and its ports
SPLITMIX64_1234567 = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                      4593380528125082431, 16408922859458223821]


def test_stream_is_splitmix64_in_counter_form():
    assert [int(v) for v in W.raw_u64(1234567, 0, 5)] == SPLITMIX64_1234567
    # output i of a stream does not depend on where a read starts
    assert [int(v) for v in W.raw_u64(1234567, 2, 3)] == SPLITMIX64_1234567[2:]


def test_streams_are_deterministic_and_distinct():
    s0, s1 = W.stream_seed(7, 0), W.stream_seed(7, 1)
    assert s0 != s1
    assert np.array_equal(W.normal(s0, 1000), W.normal(s0, 1000))
    assert not np.array_equal(W.normal(s0, 1000), W.normal(s1, 1000))


N = 1 << 20


def test_uniform01_top_24_bits():
    u = W.uniform01(W.stream_seed(11, 3), N).astype(np.float64)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2.0 ** 24 == np.floor(u * 2.0 ** 24))     # multiples of 2^-24
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / N)
    assert abs(u.var() - 1 / 12) < 5 * math.sqrt(1 / 180 / N)


def test_normal_moments():
    z = W.normal(W.stream_seed(12, 4), N, 0.0, 1.0).astype(np.float64)
    assert abs(z.mean()) < 5 / math.sqrt(N)
    assert abs(z.var() - 1.0) < 5 * math.sqrt(2.0 / N)
    assert abs(np.mean(z ** 3)) < 5 * math.sqrt(15.0 / N)          # symmetric
    assert abs(np.mean(z ** 4) - 3.0) < 5 * math.sqrt(96.0 / N)    # normal kurtosis
    z2 = W.normal(W.stream_seed(12, 4), N, 1.5, 0.25).astype(np.float64)
    assert abs(z2.mean() - 1.5) < 5 * 0.25 / math.sqrt(N)
    assert abs(z2.std() - 0.25) < 0.01 * 0.25


def test_class_ids_uniform():
    c = 1000
    ids = W.class_ids(W.stream_seed(13, 5), N, c)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < c
    counts = np.bincount(ids, minlength=c).astype(np.float64)
    e = N / c
    chi2 = float(((counts - e) ** 2 / e).sum())
    # chi-square with 999 degrees of freedom: mean 999, sd ~44.7
    assert abs(chi2 - (c - 1)) < 6 * math.sqrt(2 * (c - 1))


@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c5"])
def test_initialisers(key):
    w = W.workload(key)
    if key == "c3":   # the full C3 weights are large: the same recipe at a quarter width
        w = W.scaled(w, 4, 64)
    for (name, shape), a in zip(W.param_shapes(w.layers), W.init_params(w)):
        assert a.shape == tuple(shape) and a.dtype == np.float32
        if name.endswith(".b"):
            assert not a.any()
            continue
        if name.endswith(".gamma"):
            assert np.all(a == 1.0)
            continue
        fan_in, fan_out = shape
        x = a.astype(np.float64).ravel()
        n = x.size
        if w.init == "he_normal":
            sd = math.sqrt(2.0 / fan_in)
        elif w.init == "xavier_uniform":
            lim = math.sqrt(6.0 / (fan_in + fan_out))
            assert np.abs(x).max() <= lim
            sd = lim / math.sqrt(3.0)
        else:
            sd = 0.02
        assert abs(x.mean()) < 6 * sd / math.sqrt(n)
        assert abs(x.std() / sd - 1.0) < 6 * math.sqrt(1.0 / n) + 1e-3


def test_workload_shapes():
    c1, c2, c3, c4, c5 = (W.workload(k) for k in ("c1", "c2", "c3", "c4", "c5"))
    assert (c1.batch, c1.d_in, c1.d_out, c1.loss, c1.optimizer) == (32, 784, 10, "ce_dense", "sgd")
    assert (c2.batch, c2.d_in, c2.d_out, c2.loss, c2.optimizer) == (4096, 784, 10, "ce_dense", "adam")
    assert (c3.batch, c3.d_in, c3.d_out, c3.loss) == (8192, 4096, 1000, "ce_dense")
    assert (c4.batch, c4.d_in, c4.d_out, c4.loss) == (16384, 2048, 32000, "ce_index")
    assert (c5.batch, c5.d_in, c5.d_out, c5.loss) == (8 * 1024, 1024, 1024, "mse")
    assert c1.param_count() == 784 * 128 + 128 * 10
    assert c2.param_count() == 1863690
    assert c3.param_count() == 54440936
    assert c4.param_count() == 333987840
    assert c5.param_count() == 4194304


@pytest.mark.parametrize("loss", ["ce_dense", "ce_index", "mse"])
def test_labels(loss):
    w = W.Workload(name="lbl", index=21, batch=512, layers=[W.linear(16, 12, False)], loss=loss,
                   precisions=("strict",), optimizer="sgd", lr=0.1, steps=1, init="he_normal",
                   x_dist="normal")
    y = W.make_labels(w)
    if loss == "ce_dense":
        assert y.shape == (512, 12) and y.dtype == np.float32
        assert np.all(y.sum(axis=1) == 1.0) and set(np.unique(y)) <= {0.0, 1.0}
    elif loss == "ce_index":
        assert y.shape == (512,) and y.dtype == np.int32 and y.min() >= 0 and y.max() < 12
    else:
        assert y.shape == (512, 12) and y.dtype == np.float32
        assert abs(float(y.mean())) < 0.1 and abs(float(y.std()) - 1.0) < 0.1
    x = W.make_x(w)
    assert x.shape == (512, 16) and x.dtype == np.float32
