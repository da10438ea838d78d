"""The oracle against PyTorch CPU float64 autograd and torch.optim on every
workload's structure (scaled down): a library special case, independent of the
oracle's code."""
import numpy as np
import pytest

import oracle
import torch_ref
from static_graph_nn_gb300 import workloads as W

SMALL = {
    "c1": dict(width_div=8, batch_div=4),
    "c2": dict(width_div=32, batch_div=256),
    "c3": dict(width_div=128, batch_div=512),
    "c4": dict(width_div=128, batch_div=1024, blocks=2),
    "c5": dict(width_div=8, batch_div=1, name_suffix="_tiny"),
}


def small(key):
    w = W.scaled(W.workload(key), **SMALL[key])
    if key == "c5":
        for l in w.layers:
            if l["op"] == "causal_attention":
                l["seq_len"] = 16
        w.batch = 32
    return w


CASES = [(k, p) for k in SMALL for p in ("exact",) + W.workload(k).precisions]


@pytest.mark.parametrize("key,precision", CASES)
def test_oracle_matches_torch(key, precision):
    w = small(key)
    params = W.init_params(w)
    x, y = W.make_x(w), W.make_labels(w)
    steps = 3
    ho = oracle.run_steps(w.layers, params, x, y, w.loss, precision, w.optimizer, w.lr, steps)
    ht = torch_ref.run(w.layers, params, x, y, w.loss, precision, w.optimizer, w.lr, steps)
    for t, (a, b) in enumerate(zip(ho, ht)):
        # step 1 starts from identical params; later steps carry the float32
        # storage of the oracle's params (torch keeps float64)
        tol = 1e-12 if t == 0 else 1e-7
        assert abs(a["loss"] - b["loss"]) <= tol * max(1.0, abs(b["loss"]))
        for ga, gb in zip(a["grads"], b["grads"]):
            scale = max(np.abs(gb).max(), 1e-30)
            # oracle params are stored float32 after each update: ~1e-7 relative drift
            assert np.abs(ga - gb).max() / scale < 1e-5
        for pa, pb in zip(a["params"], b["params"]):
            assert np.abs(pa - pb).max() <= 1e-6 * max(1.0, np.abs(pb).max())
