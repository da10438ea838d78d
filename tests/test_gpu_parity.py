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


def attn(seq: int, heads: int, nseq: int, name: str):
    """One causal attention layer (head_dim 64) between two projections, MSE,
    Adam: sequence lengths with an odd number of 128-row blocks, a single
    block, more (pair, head, sequence) units than SMs, and a length that is
    not a multiple of 128."""
    d = heads * 64
    return W.Workload(name=name, index=11, batch=seq * nseq,
                      layers=[W.linear(d, 3 * d, False), W.causal_attention(heads, 64, seq),
                              W.linear(d, d, False)],
                      loss="mse", precisions=("bf16",), optimizer="adam", lr=1e-3,
                      steps=2, init="normal002", x_dist="normal")


CASES = {
    "attn_s128_h3_b2": (lambda: attn(128, 3, 2, "attn_s128"), "bf16", 2),
    "attn_s384_h5_b3": (lambda: attn(384, 5, 3, "attn_s384"), "bf16", 2),
    "attn_s640_h2_b2": (lambda: attn(640, 2, 2, "attn_s640"), "bf16", 2),
    "attn_s256_h8_b24": (lambda: attn(256, 8, 24, "attn_s256"), "bf16", 2),
    "attn_s192_h2_b2": (lambda: attn(192, 2, 2, "attn_s192"), "bf16", 2),
    "c1": (lambda: W.workload("c1"), "strict", 1),
    "c2_strict": (lambda: W.workload("c2"), "strict", 10),
    "c2_bf16": (lambda: W.workload("c2"), "bf16", 10),
    "c3_w4": (lambda: W.scaled(W.workload("c3"), 4, 4), "bf16", 20),
    "c4_w8": (lambda: W.scaled(W.workload("c4"), 8, 8), "bf16", 10),
    "c5_h4_b2": (lambda: W.scaled(W.workload("c5"), 4, 4), "bf16", 3),
    "ragged_strict": (ragged, "strict", 3),
    "ragged_bf16": (ragged, "bf16", 3),
    "ragged_sgd_strict": (lambda: _sgd(ragged()), "strict", 2),
    "ragged_laprop_strict": (lambda: _opt(ragged(), "laprop", 1e-3), "strict", 3),
    "ragged_laprop_bf16": (lambda: _opt(ragged(), "laprop", 1e-3), "bf16", 3),
    "ragged_momentum_strict": (lambda: _opt(ragged(), "sgd_momentum", 0.05), "strict", 3),
    "ragged_momentum_bf16": (lambda: _opt(ragged(), "sgd_momentum", 0.05), "bf16", 3),
}


def _opt(w, name, lr):
    w.optimizer = name
    w.lr = lr
    return w


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
