"""Checkpoints through the C ABI (GPU): exact round trip of the logical
tensors, a restore that changes nothing when its checks fail, and a trained
model taken over by a plan with another optimizer for inference."""
import struct

import numpy as np
import pytest

from static_graph_nn_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _mlp(optimizer="adam"):
    return W.Workload(name="ckpt_mlp", index=12, batch=96,
                      layers=[W.linear(40, 72, True), W.gelu_tanh(), W.linear(72, 24, True),
                              W.relu(), W.linear(24, 10, False)],
                      loss="ce_dense", precisions=("strict", "bf16"), optimizer=optimizer,
                      lr=1e-3, steps=3, init="he_normal", x_dist="normal")


def _plan(w, precision):
    from static_graph_nn_gb300.binding import Plan
    return Plan.for_workload(w, precision)


def _filled(plan, seed, sentinel=float("nan")):
    """A flat buffer whose logical tensors hold seeded values and whose gaps
    between tensors hold a sentinel (never read or written by the library)."""
    g = np.random.default_rng(seed)
    a = np.full(plan.param_count, sentinel, np.float32)
    for off, r, c in plan.param_info():
        a[off:off + r * c] = g.standard_normal(r * c).astype(np.float32)
    return torch.from_numpy(a).cuda()


def _same(a, b):
    return bool(np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32)))


@pytest.mark.parametrize("precision", ["strict", "bf16"])
def test_round_trip_is_exact_and_keeps_gaps(precision):
    plan = _plan(_mlp(), precision)
    p, m, v = _filled(plan, 1), _filled(plan, 2), _filled(plan, 3).abs()
    img = plan.checkpoint_save(p, m, v)
    logical = sum(r * c for _, r, c in plan.param_info())
    assert len(img) == 64 + 8 * len(plan.param_info()) + 3 * 4 * logical
    assert img[:8] == b"MGCKPT\x00\x01"
    version, nt, flags = struct.unpack_from("<III", img, 8)
    assert (version, nt, flags) == (1, len(plan.param_info()), 3)
    q, mq, vq = (_filled(plan, 9, sentinel=-7.0) for _ in range(3))
    plan.checkpoint_load(img, q, mq, vq)
    for got, want in ((q, p), (mq, m), (vq, v)):
        for off, r, c in plan.param_info():
            assert _same(got[off:off + r * c], want[off:off + r * c])
        # the gaps are untouched
        mask = np.ones(plan.param_count, bool)
        for off, r, c in plan.param_info():
            mask[off:off + r * c] = False
        assert np.all(got.cpu().numpy()[mask] == -7.0)


def test_failed_preflight_changes_nothing():
    plan = _plan(_mlp(), "strict")
    p = _filled(plan, 1)
    img = plan.checkpoint_save(p)              # params only
    dst = _filled(plan, 5)
    before = dst.clone()
    from static_graph_nn_gb300.binding import MGError
    bad = []
    b = bytearray(img); b[0] ^= 1; bad.append(bytes(b))                      # magic
    bad.append(img[:-4])                                                     # truncated
    b = bytearray(img); b[-3] ^= 0x40; bad.append(bytes(b))                  # data (checksum)
    b = bytearray(img); struct.pack_into("<I", b, 64, 41); bad.append(bytes(b))   # a shape
    b = bytearray(img); struct.pack_into("<I", b, 8, 2); bad.append(bytes(b))     # version
    for image in bad:
        with pytest.raises(MGError):
            plan.checkpoint_load(image, dst)
        assert _same(dst, before)
    # moments asked for but not stored
    m = _filled(plan, 6)
    m_before = m.clone()
    with pytest.raises(MGError):
        plan.checkpoint_load(img, dst, m)
    assert _same(dst, before) and _same(m, m_before)
    # another graph's checkpoint
    other = _plan(W.Workload(name="other", index=13, batch=96,
                             layers=[W.linear(40, 64, True), W.relu(), W.linear(64, 10, False)],
                             loss="ce_dense", precisions=("strict",), optimizer="sgd", lr=0.1,
                             steps=1, init="he_normal", x_dist="normal"), "strict")
    with pytest.raises(MGError):
        plan.checkpoint_load(other.checkpoint_save(_filled(other, 7)), dst)
    assert _same(dst, before)


@pytest.mark.parametrize("precision", ["strict", "bf16"])
def test_train_then_deploy_in_another_plan(precision):
    """Three Adam steps in one plan, then the checkpoint's parameters (its
    moments skipped) in a fresh SGD plan: the two plans' forward outputs agree
    bit for bit, and a moment-carrying restore resumes training exactly."""
    import gpu_harness as H
    w = _mlp("adam")
    train = _plan(w, precision)
    x, y, xt, yt = H.to_device_inputs(w, precision)
    dev = H.Device(train, w, precision)
    dev.load(W.init_params(w))
    for t in range(1, 4):
        train.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, t)
    img = train.checkpoint_save(dev.params, dev.m, dev.v)

    w2 = _mlp("sgd")
    deploy = _plan(w2, precision)
    p2 = torch.zeros_like(dev.params)
    deploy.checkpoint_load(img, p2)
    out1 = torch.zeros(w.batch, 10, dtype=torch.float32, device="cuda")
    out2 = torch.zeros_like(out1)
    train.forward(dev.params, xt, out1)
    deploy.forward(p2, xt, out2)
    torch.cuda.synchronize()
    assert _same(out1, out2)

    # resume: a restored copy of the optimizer state continues identically
    resumed = _plan(w, precision)
    p3, m3, v3 = (torch.zeros_like(dev.params) for _ in range(3))
    resumed.checkpoint_load(img, p3, m3, v3)
    g3 = torch.zeros_like(dev.params)
    train.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, 4)
    resumed.train_step(p3, g3, m3, v3, xt, yt, w.lr, 4)
    torch.cuda.synchronize()
    for off, r, c in train.param_info():
        assert _same(p3[off:off + r * c], dev.params[off:off + r * c])
