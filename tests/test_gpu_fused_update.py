"""Adam's weight update fused into the weight-gradient GEMM's epilogue (GPU).

With Adam in bf16, a linear node whose weight gradient runs on the tensor
cores without a split over K updates that weight (parameters, both moments
and the bf16 copy) in the GEMM's epilogue instead of in the optimizer kernel;
it is off unless MG_FUSED_UPDATE=1 at plan creation.  Both paths run the same Adam arithmetic on
the same fp32 gradient, so every step gives the same bits either way (steps
two and three are graph replays, whose step scalars the replay patches).  The
fused path is also checked against the oracle like every other case."""
import os

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


def fused_mlp():
    """Weight gradients of 2048x4096, 4096x4096 and 4096x2048 (128, 256 and
    128 tiles of 256x256, no split over K: all fused; nothing in the step is
    summed by atomics), biases on the hidden layers, a ragged batch."""
    return W.Workload(name="fused_mlp", index=18, batch=1000,
                      layers=[W.linear(2048, 4096, True), W.gelu_tanh(),
                              W.linear(4096, 4096, True), W.gelu_tanh(),
                              W.linear(4096, 2048, False)],
                      loss="ce_index", precisions=("bf16",), optimizer="adam", lr=1e-3,
                      steps=3, init="he_normal", x_dist="normal")


def _run(w, fused, steps):
    import gpu_harness as H
    from static_graph_nn_gb300.binding import Plan
    old = os.environ.get("MG_FUSED_UPDATE")
    os.environ["MG_FUSED_UPDATE"] = "1" if fused else "0"
    try:
        plan = Plan.for_workload(w, "bf16")
    finally:
        if old is None:
            del os.environ["MG_FUSED_UPDATE"]
        else:
            os.environ["MG_FUSED_UPDATE"] = old
    x, y, xt, yt = H.to_device_inputs(w, "bf16")
    dev = H.Device(plan, w, "bf16")
    dev.load(W.init_params(w))
    losses = []
    for t in range(1, steps + 1):
        plan.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, t)
        losses.append(plan.loss())
    out = dev.read()
    dump = plan.dump()
    plan.close()
    return losses, out, dump


def test_fused_update_same_bits():
    w = fused_mlp()
    la, a, dump_a = _run(w, True, 3)
    lb, b, dump_b = _run(w, False, 3)
    for layer in (0, 2, 4):
        assert f"layer {layer}: Adam update of the weight fused" in dump_a
    assert "fused into its gradient GEMM" not in dump_b
    assert la == lb
    names = [n for n, _ in W.param_shapes(w.layers)]
    for key in ("params", "adam_m", "adam_v", "grads"):
        for i, name in enumerate(names):
            assert np.array_equal(a[key][i], b[key][i]), (key, name)


def test_fused_update_parity():
    import gpu_harness as H
    worst = H.compare(fused_mlp(), "bf16", 3)
    print(worst)
