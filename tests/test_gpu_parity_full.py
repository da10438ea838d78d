"""Full-size parity: the workloads at their full shapes, in the launch
configuration the benchmark times, against the oracle (GPU).

C3 and C5: one teacher-forced step at full size against oracle.train_step.
C4 (16384 tokens, 334M parameters): the oracle runs over row chunks; because
the loss is a mean over rows, each chunk's backward with its gradient scaled by
chunk/B contributes exactly its share of every parameter gradient, so the sum
over chunks is the full-batch gradient."""
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


@pytest.mark.parametrize("key", ["c3", "c5"])
def test_full_size_step(key):
    import gpu_harness
    w = W.workload(key)
    worst = gpu_harness.compare(w, "bf16", 1)
    print(key, worst)


def _oracle_chunked_step(w, params, x, y, chunk):
    """Loss and parameter gradients of the full batch, by row chunks."""
    import oracle
    from oracle import step as S
    B = w.batch
    loss = 0.0
    grads = None
    for r0 in range(0, B, chunk):
        xs, ys = x[r0:r0 + chunk], y[r0:r0 + chunk]
        n = xs.shape[0]
        out, tape = oracle.forward(w.layers, params, xs, "bf16")
        l, dout = oracle.loss_and_grad(w.loss, out, ys, "bf16")
        loss += l * n / B
        g, _ = oracle.backward(w.layers, params, tape, dout * (n / B), "bf16")
        grads = g if grads is None else [a + b for a, b in zip(grads, g)]
    return loss, grads


def test_full_size_c4_step():
    import gpu_harness as H
    from static_graph_nn_gb300 import Plan
    w = W.workload("c4")
    p0 = W.init_params(w)
    x, y, xt, yt = H.to_device_inputs(w, "bf16")
    plan = Plan.for_workload(w, "bf16")
    dev = H.Device(plan, w, "bf16")
    dev.load(p0)
    plan.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, 1)
    loss = plan.loss()
    g = dev.read()
    plan.close()
    o_loss, o_grads = _oracle_chunked_step(w, p0, x, y, 1024)
    e = abs(loss - o_loss) / abs(o_loss)
    assert e <= H.BF16_LOSS_TOL, (loss, o_loss)
    names = [n for n, _ in W.param_shapes(w.layers)]
    worst = 1.0
    for n, a, b in zip(names, g["grads"], o_grads):
        c = H.cosine(a, b)
        worst = min(worst, c)
        assert c >= H.BF16_COSINE, (n, c)
    # Adam at t = 1 moves each parameter by at most lr (|g| / (|g| + eps) <= 1)
    for a, b in zip(g["params"], p0):
        assert np.abs(a - b).max() <= w.lr * (1 + 1e-3)
    print("c4 full", {"loss": e, "grad_cosine": worst})
