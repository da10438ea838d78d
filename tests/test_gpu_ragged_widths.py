"""bf16 layers whose rows break the 16-byte rule of the tensor-memory copies
(GPU): a hidden width of 36 and heads of 10 and 17 classes run on the
CUDA-core kernels, the narrow-side ones included (forward with N <= 32, input
gradient with K <= 32, weight gradient with N <= 32), on their unaligned and
scalar paths, and must match the oracle like every other bf16 case."""
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


def _mlp(d_in, hidden, classes, act, bias, loss, index):
    return W.Workload(name=f"w{hidden}_c{classes}", index=index, batch=200,
                      layers=[W.linear(d_in, hidden, True), act(), W.linear(hidden, classes, bias)],
                      loss=loss, precisions=("bf16",), optimizer="adam", lr=1e-3, steps=3,
                      init="he_normal", x_dist="normal")


CASES = {
    "w36_c10_gelu_dense": (lambda: _mlp(40, 36, 10, W.gelu_tanh, True, "ce_dense", 16), 3),
    "w36_c17_relu_index": (lambda: _mlp(48, 36, 17, W.relu, False, "ce_index", 17), 3),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_parity_unaligned_widths(case):
    import gpu_harness as H
    mk, steps = CASES[case]
    worst = H.compare(mk(), "bf16", steps)
    print(case, worst)
