"""Lifetime sharing of gradient buffers (GPU): the same steps with and
without sharing (MG_NO_ALIAS=1) give the same loss and gradients, and sharing
shrinks the gradient storage of a residual network."""
import os
import re

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


def _run(w, precision, alias, steps=2):
    import gpu_harness as H
    from static_graph_nn_gb300.binding import Plan
    old = os.environ.get("MG_NO_ALIAS")
    os.environ["MG_NO_ALIAS"] = "0" if alias else "1"
    try:
        plan = Plan.for_workload(w, precision)
    finally:
        if old is None:
            del os.environ["MG_NO_ALIAS"]
        else:
            os.environ["MG_NO_ALIAS"] = old
    x, y, xt, yt = H.to_device_inputs(w, precision)
    dev = H.Device(plan, w, precision)
    dev.load(W.init_params(w))
    losses = []
    for t in range(1, steps + 1):
        plan.train_step(dev.params, dev.grads, dev.m, dev.v, xt, yt, w.lr, t)
        losses.append(plan.loss())
    g = dev.read()
    m = re.search(r"gradient storage: (\d+) bytes \((\d+) without", plan.dump())
    return losses, g, (int(m.group(1)), int(m.group(2))), plan.workspace_bytes


CASES = {
    "c4_w8_strict": (lambda: W.scaled(W.workload("c4"), 8, 8), "strict"),
    "c4_w8_bf16": (lambda: W.scaled(W.workload("c4"), 8, 8), "bf16"),
    "c5_h4_b2": (lambda: W.scaled(W.workload("c5"), 4, 4), "bf16"),
    "c2_strict": (lambda: W.workload("c2"), "strict"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_sharing_changes_no_result(case):
    mk, precision = CASES[case]
    w = mk()
    # one step in bf16: a second would start from Adam updates of gradients
    # that split-K atomics may round differently, which Adam's normalised step
    # amplifies near g = 0
    steps = 2 if precision == "strict" else 1
    la, ga, (shared, unshared), ws_a = _run(w, precision, True, steps)
    lb, gb, (shared_b, unshared_b), ws_b = _run(w, precision, False, steps)
    assert shared_b == unshared_b == unshared and shared <= unshared and ws_a <= ws_b
    # bf16 weight gradients may be summed in a different order by split-K
    # atomics from run to run; everything else is deterministic
    tol = 0.0 if precision == "strict" else 1e-5
    for a, b in zip(la, lb):
        assert abs(a - b) <= tol * abs(b)
    for a, b in zip(ga["grads"], gb["grads"]):
        assert np.abs(a - b).max() <= tol * max(np.abs(b).max(), 1e-30)
    if case.startswith("c4"):
        # eight residual blocks: the backward's gradients fit in a few shared buffers
        assert shared * 3 < unshared
