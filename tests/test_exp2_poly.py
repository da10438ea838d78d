"""The FMA-pipe 2^x used for part of the attention probabilities, replayed in
float32 on the CPU from the constants in the CUDA source: relative error
against exact 2^x over the range the softmax feeds it, far below the bf16
rounding the probabilities then get, and the clamp for masked (-inf) keys."""
import pathlib
import re

import numpy as np

SRC = pathlib.Path(__file__).resolve().parents[1] / "static_graph_nn_gb300" / "csrc" / "attention_tc.cu"


def _consts():
    text = SRC.read_text()
    body = text[text.index("float2 ex2_poly2("):]
    body = body[:body.index("\n}\n")]
    vals = dict(re.findall(r"\b(C[0-3]|RND) = ([0-9.e+-]+)f", body))
    return [np.float32(float(vals[k])) for k in ("C0", "C1", "C2", "C3")], np.float32(float(vals["RND"]))


def ex2_poly(x):
    """The device steps in float32: clamp, round via the 1.5 * 2^23 add, the
    cubic in f, and the integer add of j into the exponent field."""
    (c0, c1, c2, c3), rnd = _consts()
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-125.0))
    t = (x + rnd).astype(np.float32)
    j = (t - rnd).astype(np.float32)
    f = (x - j).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def test_relative_error_over_softmax_range():
    # the softmax feeds x = s * log2(e) / 8 - m <= 8 (the rescale threshold)
    x = np.linspace(-60.0, 8.0, 400001, dtype=np.float32)
    got = ex2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1.0e-4, rel.max()
    # bf16 keeps 8 significant bits: half an ulp is 2^-9
    assert rel.max() < 2.0 ** -9 / 10


def test_integers_and_halves():
    x = np.array([-3.0, -2.5, -1.0, -0.5, 0.0, 0.5, 1.0, 7.5, 8.0], dtype=np.float32)
    got = ex2_poly(x).astype(np.float64)
    np.testing.assert_allclose(got, np.exp2(x.astype(np.float64)), rtol=1.0e-4)


def test_masked_keys_give_a_negligible_positive():
    got = ex2_poly(np.array([-np.inf, -1.0e30, -200.0], dtype=np.float32))
    assert np.all(got > 0.0) and np.all(got < 2.0 ** -124)
