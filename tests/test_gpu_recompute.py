"""GELU pre-activations recomputed in the backward instead of saved
(MG_RECOMPUTE_GELU=1, the memory planner's optional recomputation; GPU): the
same steps give the same loss and gradients -- the recomputation runs the
forward's GEMM on the same inputs and weights -- and the workspace shrinks by
all but one of the saved pre-activations."""
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


def _run(w, precision, recompute, steps):
    import gpu_harness as H
    from static_graph_nn_gb300.binding import Plan
    old = os.environ.get("MG_RECOMPUTE_GELU")
    os.environ["MG_RECOMPUTE_GELU"] = "1" if recompute else "0"
    try:
        plan = Plan.for_workload(w, precision)
    finally:
        if old is None:
            del os.environ["MG_RECOMPUTE_GELU"]
        else:
            os.environ["MG_RECOMPUTE_GELU"] = old
    x, y, xt, yt = H.to_device_inputs(w, precision)
    dev = H.Device(plan, w, precision)
    dev.load(W.init_params(w))
    losses = []
    for t in range(1, steps + 1):
        plan.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, t)
        losses.append(plan.loss())
    out = dev.read()
    ws = plan.workspace_bytes
    dump = plan.dump()
    plan.close()
    return losses, out, ws, dump


CASES = {
    "c4_w8_strict": (lambda: W.scaled(W.workload("c4"), 8, 8), "strict"),
    "c4_w8_bf16": (lambda: W.scaled(W.workload("c4"), 8, 8), "bf16"),
    "c3_w4_bf16": (lambda: W.scaled(W.workload("c3"), 4, 4), "bf16"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_recompute_changes_no_result(case):
    mk, precision = CASES[case]
    w = mk()
    steps = 2 if precision == "strict" else 1
    la, ga, ws_a, dump_a = _run(w, precision, False, steps)
    lb, gb, ws_b, dump_b = _run(w, precision, True, steps)
    assert "recomputed in the backward" in dump_b and "recomputed" not in dump_a
    # one buffer instead of one per GELU layer
    es = 4 if precision == "strict" else 2
    z = [l["d_out"] for i, l in enumerate(w.layers[:-1])
         if l["op"] == "linear" and w.layers[i + 1]["op"] == "gelu_tanh"]
    saved = w.batch * es * (sum(z) - max(z))
    assert ws_a - ws_b >= saved - 4096 * len(z), (ws_a, ws_b, saved)
    # bf16 weight gradients may be summed in a different order by split-K
    # atomics from run to run; everything else is deterministic
    tol = 0.0 if precision == "strict" else 1e-5
    for a, b in zip(la, lb):
        assert abs(a - b) <= tol * abs(b)
    for a, b in zip(ga["grads"], gb["grads"]):
        assert np.abs(a - b).max() <= tol * max(np.abs(b).max(), 1e-30)


def test_recompute_full_size_residual_network_workspace():
    """The 8-block residual network at full size: the workspace drops by the
    seven GELU pre-activations it no longer keeps (16384 x 8192 bf16 each)."""
    w = W.workload("c4")
    _, _, ws_a, _ = _run(w, "bf16", False, 1)
    _, _, ws_b, _ = _run(w, "bf16", True, 1)
    print("c4 workspace GiB: saved", ws_a / 2 ** 30, "recomputed", ws_b / 2 ** 30)
    assert ws_a - ws_b >= 7 * 16384 * 8192 * 2 - 8 * 4096
