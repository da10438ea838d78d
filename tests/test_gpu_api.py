"""Smaller entry points of the C ABI (GPU): the asynchronous loss read."""
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


@pytest.mark.parametrize("precision", ["strict", "bf16"])
def test_loss_async_matches_loss(precision):
    """mg_loss_async's (loss, timed_out) pair, read after the stream passes
    it, equals what mg_loss returns, for each of three steps."""
    import gpu_harness as H
    from static_graph_nn_gb300.binding import Plan
    w = W.Workload(name="api_mlp", index=14, batch=64,
                   layers=[W.linear(32, 48, True), W.relu(), W.linear(48, 8, False)],
                   loss="ce_dense", precisions=("strict", "bf16"), optimizer="adam", lr=1e-3,
                   steps=3, init="he_normal", x_dist="normal")
    plan = Plan.for_workload(w, precision)
    x, y, xt, yt = H.to_device_inputs(w, precision)
    dev = H.Device(plan, w, precision)
    dev.load(W.init_params(w))
    host = torch.zeros(3, 2, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    for t in range(1, 4):
        plan.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, t, stream)
        plan.loss_async(host[t - 1].data_ptr(), stream)
        stream.synchronize()
        assert float(host[t - 1, 0]) == plan.loss(stream)
    assert host.view(torch.int32)[:, 1].tolist() == [0, 0, 0]
    assert np.all(np.isfinite(host[:, 0].numpy()))


def test_ffma_peak_is_the_fp32_pipe():
    """mg_ffma_peak measures what the SMs' FP32 units can do: per SM and clock
    (at the maximum clock) at most 128 lanes x 2 flop, and at least half of
    it (eight independent chains per thread, two 1024-thread blocks per SM,
    leave no latency exposed); repeated calls agree within 5%."""
    from static_graph_nn_gb300 import binding
    t1, per_clk = binding.ffma_peak()
    t2, _ = binding.ffma_peak()
    assert 128.0 <= per_clk <= 256.0 * 1.02, per_clk
    assert abs(t1 - t2) <= 0.05 * max(t1, t2), (t1, t2)
