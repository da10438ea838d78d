"""mg_forward (the forward-only entry point, a deploy-time session over the
same graph as in the "Meganeura" README's Example section) against the
oracle's forward pass, element by element on the same seeded inputs (GPU).

Strict f32: max|a-b| / max|b| <= 1e-4 over the whole output.  bf16: cosine
>= 0.999 over the output (the gradient gate of the bf16 path applied to the
model output), with the max relative error printed.  Full sizes, in the
launch configuration the benchmark times: the GPU runs the whole batch and
the oracle a row sample -- rows are independent in the MLP and residual
stacks, and sequences are in the attention layer, so the sample's outputs
are the full batch's."""
import numpy as np
import pytest

import oracle
from static_graph_nn_gb300 import Plan
from static_graph_nn_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STRICT_TOL = 1e-4
BF16_COSINE = 0.999


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _gpu_forward(w, precision, p0, x):
    import gpu_harness as H
    plan = Plan.for_workload(w, precision)
    params = H.pack(plan, p0)
    xt = torch.from_numpy(x).cuda()
    if precision == "bf16":
        xt = xt.to(torch.bfloat16)
    out = torch.full((w.batch, w.d_out), float("nan"), dtype=torch.float32, device="cuda")
    plan.forward(params, xt.contiguous(), out)
    torch.cuda.synchronize()
    plan.close()
    return out.double().cpu().numpy()


def _compare(got, want, precision, label):
    import gpu_harness as H
    assert np.isfinite(got).all(), label
    e = H.max_rel(got, want)
    if precision == "strict":
        assert e <= STRICT_TOL, f"{label}: max rel err {e:.3g}"
        return {"max_rel": e}
    c = H.cosine(got, want)
    assert c >= BF16_COSINE, f"{label}: cosine {c:.6f} (max rel {e:.3g})"
    return {"cosine": c, "max_rel": e}


def _ragged():
    return W.Workload(name="ragged", index=9, batch=300,
                      layers=[W.linear(200, 136, True), W.gelu_tanh(), W.linear(136, 72, True),
                              W.relu(), W.linear(72, 24, False)],
                      loss="ce_dense", precisions=("strict", "bf16"), optimizer="adam",
                      lr=1e-3, steps=3, init="he_normal", x_dist="normal")


CASES = {
    "c1_strict": (lambda: W.workload("c1"), "strict"),
    "c2_strict": (lambda: W.workload("c2"), "strict"),
    "c2_bf16": (lambda: W.workload("c2"), "bf16"),
    "c3_w4_bf16": (lambda: W.scaled(W.workload("c3"), 4, 4), "bf16"),
    "c4_w8_bf16": (lambda: W.scaled(W.workload("c4"), 8, 8), "bf16"),
    "c5_h4_b2_bf16": (lambda: W.scaled(W.workload("c5"), 4, 4), "bf16"),
    "ragged_strict": (_ragged, "strict"),
    "ragged_bf16": (_ragged, "bf16"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_matches_the_oracle(case):
    mk, prec = CASES[case]
    w = mk()
    p0 = W.init_params(w)
    x = W.make_x(w)
    got = _gpu_forward(w, prec, p0, x)
    want, _ = oracle.forward(w.layers, p0, x, prec)
    print(case, _compare(got, want, prec, case))


@pytest.mark.parametrize("key", ["c3", "c4", "c5"])
def test_forward_full_size_sampled(key):
    """The whole batch on the GPU; the oracle on a sample: 256 rows spread
    over the batch (first, last and strided) for the MLP and residual stacks,
    two whole sequences (the first and the last) for the attention layer."""
    w = W.workload(key)
    p0 = W.init_params(w)
    x = W.make_x(w)
    got = _gpu_forward(w, "bf16", p0, x)
    seq = next((l["seq_len"] for l in w.layers if l["op"] == "causal_attention"), None)
    if seq:
        rows = np.concatenate([np.arange(seq), np.arange(w.batch - seq, w.batch)])
    else:
        rows = np.unique(np.concatenate([np.arange(64), np.arange(w.batch - 64, w.batch),
                                         np.linspace(0, w.batch - 1, 128).astype(int)]))
    want, _ = oracle.forward(w.layers, p0, x[rows], "bf16")
    print(key, len(rows), "rows", _compare(got[rows], want, "bf16", key))
