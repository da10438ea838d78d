"""The CUDA path against the oracle on the same seeded inputs (GPU)."""
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


def _h():
    import gpu_harness
    return gpu_harness


def ragged():
    """Widths that are not tile multiples, a batch with a ragged last tile."""
    return W.Workload(name="ragged", index=9, batch=300,
                      layers=[W.linear(200, 136, True), W.gelu_tanh(), W.linear(136, 72, True),
                              W.relu(), W.linear(72, 24, False)],
                      loss="ce_dense", precisions=("strict", "bf16"), optimizer="adam",
                      lr=1e-3, steps=3, init="he_normal", x_dist="normal")


CASES = {
    "c1": (lambda: W.workload("c1"), "strict", 1),
    "c2_strict": (lambda: W.workload("c2"), "strict", 10),
    "c2_bf16": (lambda: W.workload("c2"), "bf16", 10),
    "c3_w4": (lambda: W.scaled(W.workload("c3"), 4, 4), "bf16", 20),
    "c4_w8": (lambda: W.scaled(W.workload("c4"), 8, 8), "bf16", 10),
    "c5_h4_b2": (lambda: W.scaled(W.workload("c5"), 4, 4), "bf16", 3),
    "ragged_strict": (ragged, "strict", 3),
    "ragged_bf16": (ragged, "bf16", 3),
    "ragged_sgd_strict": (lambda: _sgd(ragged()), "strict", 2),
}


def _sgd(w):
    w.optimizer = "sgd"
    w.lr = 0.05
    return w


@pytest.mark.parametrize("case", sorted(CASES))
def test_parity(case):
    mk, prec, steps = CASES[case]
    w = mk()
    worst = _h().compare(w, prec, steps)
    print(case, worst)
