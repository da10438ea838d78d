"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (finite differences, closed forms, exact brute force, invariants).

Each check returns a number (an error, a residual) so that the mutation test
can plant a mistake in the oracle and see at least one check fail.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np

import oracle
from oracle import step as ostep
from static_graph_nn_gb300 import workloads as W


def _rng(seed):
    return np.random.default_rng(seed)


def tiny_graphs():
    """Tiny graphs covering every op and loss, for finite differences."""
    L = W
    return {
        "linear_bias_relu_ce_dense": ([L.linear(3, 4, True), L.relu(), L.linear(4, 3, True)],
                                      5, 3, "ce_dense"),
        "gelu_ce_index": ([L.linear(3, 4, True), L.gelu_tanh(), L.linear(4, 5, False)],
                          4, 3, "ce_index"),
        "rmsnorm_residual": ([L.residual_begin(), L.rmsnorm(5, 1e-6), L.linear(5, 6, False),
                              L.gelu_tanh(), L.linear(6, 5, False), L.residual_end(),
                              L.residual_begin(), L.rmsnorm(5, 1e-3), L.linear(5, 5, False),
                              L.residual_end(), L.linear(5, 4, False)], 3, 5, "ce_index"),
        "attention_mse": ([L.linear(4, 12, False), L.causal_attention(2, 2, 3),
                           L.linear(4, 4, False)], 6, 4, "mse"),
        "attention_one_head_mse": ([L.linear(2, 6, False), L.causal_attention(1, 2, 3),
                                    L.linear(2, 2, False)], 3, 2, "mse"),
    }


def make_case(layers, rows, d_in, loss, seed=0):
    r = _rng(seed)
    params = []
    for name, shape in W.param_shapes(layers):
        if name.endswith(".gamma"):
            params.append(1.0 + 0.3 * r.standard_normal(shape))
        else:
            params.append(0.7 * r.standard_normal(shape))
    x = r.standard_normal((rows, d_in))
    d_out = W.output_width(layers)
    if loss == "ce_dense":
        y = np.zeros((rows, d_out))
        y[np.arange(rows), r.integers(0, d_out, rows)] = 1.0
    elif loss == "ce_index":
        y = r.integers(0, d_out, rows)
    else:
        y = r.standard_normal((rows, d_out))
    return params, x, y


def loss_of(layers, params, x, y, loss):
    out, _ = oracle.forward(layers, params, x, "exact")
    return oracle.loss_and_grad(loss, out, y)[0]


def fd_error(layers, rows, d_in, loss, h=1e-6, seed=0):
    """max |analytic - central difference| / max |analytic| over all parameters."""
    params, x, y = make_case(layers, rows, d_in, loss, seed)
    out, tape = oracle.forward(layers, params, x, "exact")
    _, dout = oracle.loss_and_grad(loss, out, y)
    grads, _ = oracle.backward(layers, params, tape, dout)
    worst = 0.0
    for i, p in enumerate(params):
        fd = np.zeros_like(p)
        for j in np.ndindex(p.shape):
            keep = p[j]
            p[j] = keep + h
            lp = loss_of(layers, params, x, y, loss)
            p[j] = keep - h
            lm = loss_of(layers, params, x, y, loss)
            p[j] = keep
            fd[j] = (lp - lm) / (2 * h)
        scale = max(np.abs(grads[i]).max(), 1e-12)
        worst = max(worst, float(np.abs(fd - grads[i]).max() / scale))
    return worst


# ---------------------------------------------------------------- closed forms

def ce_closed_form_error(seed=1):
    """Dense CE with one-hot labels: dz = (softmax(z) - y)/B, rows sum to 0."""
    r = _rng(seed)
    z = r.standard_normal((7, 5)) * 3
    y = np.zeros((7, 5))
    y[np.arange(7), r.integers(0, 5, 7)] = 1.0
    loss, g = oracle.loss_and_grad("ce_dense", z, y)
    e = np.exp(z - z.max(1, keepdims=True))
    sm = e / e.sum(1, keepdims=True)
    want_loss = -np.log(sm[y.astype(bool)]).mean()
    err = np.abs(g - (sm - y) / 7).max()
    err = max(err, abs(loss - want_loss), np.abs(g.sum(1)).max())
    # index form must agree with the dense form on the same labels
    li, gi = oracle.loss_and_grad("ce_index", z, y.argmax(1))
    return float(max(err, abs(li - loss), np.abs(gi - g).max()))


def mse_closed_form_error():
    o = np.array([[1.0, 2.0], [3.0, 5.0]])
    t = np.array([[0.0, 2.0], [4.0, 3.0]])
    loss, g = oracle.loss_and_grad("mse", o, t)
    # (1 + 0 + 1 + 4) / 4 = 1.5 ; grad 2 (o - t) / 4
    return float(max(abs(loss - 1.5), np.abs(g - np.array([[0.5, 0.0], [-0.5, 1.0]])).max()))


def adam_t1_error(seed=2):
    """At t = 1 Adam moves p by lr * g / (|g| + eps) exactly."""
    r = _rng(seed)
    p = r.standard_normal(50).astype(np.float32)
    g = r.standard_normal(50) * 10 ** r.uniform(-4, 1, 50)
    lr, eps = 1e-3, 1e-8
    p2, m2, v2 = oracle.adam_update(p, g, np.zeros(50, np.float32), np.zeros(50, np.float32),
                                    lr, 1, 0.9, 0.999, eps)
    want = (p.astype(np.float64) - lr * g / (np.abs(g) + eps)).astype(np.float32)
    e1 = np.abs(p2.astype(np.float64) - want).max()
    e2 = np.abs(m2 - (0.1 * g).astype(np.float32)).max()
    e3 = np.abs(v2 - (0.001 * g * g).astype(np.float32)).max() / max(np.abs(v2).max(), 1e-30)
    return float(max(e1, e2, e3))


def adam_t2_error():
    """Two steps with g1 = 1, g2 = -1 (beta1 .9, beta2 .999): by hand,
    m2 = .09 - .1 = -.01, v2 = .000999 + .001 = .001999,
    mhat = -.01/.19, vhat = .001999/.001999 = 1, so p2 = p1 + lr*(.01/.19)/(1+eps)."""
    lr, eps = 0.5, 1e-8
    p0 = np.array([2.0], np.float32)
    p1, m1, v1 = oracle.adam_update(p0, np.array([1.0]), np.zeros(1, np.float32),
                                    np.zeros(1, np.float32), lr, 1, 0.9, 0.999, eps)
    p2, _, _ = oracle.adam_update(p1, np.array([-1.0]), m1, v1, lr, 2, 0.9, 0.999, eps)
    want1 = 2.0 - lr * 1.0 / (1.0 + eps)
    want2 = want1 + lr * (0.01 / 0.19) / (1.0 + eps)
    return float(max(abs(p1[0] - want1), abs(p2[0] - want2)))


def sgd_error():
    p = np.array([1.0, -2.0, 0.5], np.float32)
    g = np.array([0.5, 0.25, -1.0])
    return float(np.abs(oracle.sgd_update(p, g, 0.1) - np.array([0.95, -2.025, 0.6])).max())


def laprop_t1_error(seed=4):
    """At t = 1 LaProp's second moment is (1-b2) g^2, whose bias-corrected root
    is |g|; the momentum holds (1-b1) g/(|g|+eps), and dividing by (1-b1)
    moves p by lr * g / (|g| + eps): a sign step of size lr."""
    r = _rng(seed)
    p = r.standard_normal(40).astype(np.float32)
    g = r.standard_normal(40) * 10 ** r.uniform(-4, 1, 40)
    lr, eps = 1e-3, 1e-8
    p2, m2, v2 = oracle.laprop_update(p, g, np.zeros(40, np.float32), np.zeros(40, np.float32),
                                      lr, 1, 0.9, 0.999, eps)
    want = (p.astype(np.float64) - lr * g / (np.abs(g) + eps)).astype(np.float32)
    e1 = np.abs(p2.astype(np.float64) - want).max()
    e2 = np.abs(m2 - (0.1 * g / (np.abs(g) + eps)).astype(np.float32)).max()
    e3 = np.abs(v2 - (0.001 * g * g).astype(np.float32)).max() / max(np.abs(v2).max(), 1e-30)
    return float(max(e1, e2, e3))


def laprop_constant_gradient_error():
    """With the same gradient every step both bias corrections are exact, so
    every step of LaProp moves p by lr * g / (|g| + eps): after five steps
    p5 = p0 - 5 lr g / (|g| + eps)."""
    lr, eps = 1e-2, 1e-8
    g = np.array([0.3, -2.0, 1e-3])
    p = np.array([1.0, 0.0, -1.0], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    for t in range(1, 6):
        p, m, v = oracle.laprop_update(p, g, m, v, lr, t, 0.9, 0.999, eps)
    want = np.array([1.0, 0.0, -1.0]) - 5 * lr * g / (np.abs(g) + eps)
    return float(np.abs(p - want).max())


def laprop_t2_error():
    """g1 = 1 then g2 = -2 (b1 .9, b2 .999, eps 0), worked by hand: v2 = .999 *
    .001 + .001 * 4 = .004999, corrected by 1 - .999^2 = .001999 to 2.50075037...,
    root 1.58137610...; the normalised gradient -2 / 1.58137610 = -1.26472128
    joins m1 = .1: m2 = .09 - .126472128 = -.0364721275, over 1 - .81 = .19:
    p2 = p1 + lr * .191958566.  (Adam, feeding the raw gradient to m, would step
    by .578947 / 1.581376 = .366104 instead.)"""
    lr = 0.5
    p0 = np.array([2.0], np.float32)
    p1, m1, v1 = oracle.laprop_update(p0, np.array([1.0]), np.zeros(1, np.float32),
                                      np.zeros(1, np.float32), lr, 1, 0.9, 0.999, 0.0)
    p2, m2, _ = oracle.laprop_update(p1, np.array([-2.0]), m1, v1, lr, 2, 0.9, 0.999, 0.0)
    want1 = 2.0 - lr
    want2 = want1 + lr * 0.1919585659024943
    return float(max(abs(p1[0] - want1), abs(p2[0] - want2), abs(m2[0] + 0.03647212752147392)))


def laprop_scale_invariance_error(seed=5):
    """With eps = 0 LaProp's steps do not change when every gradient is scaled
    by the same c > 0 (the gradient enters only through g / sqrt(v))."""
    r = _rng(seed)
    gs = [r.standard_normal(16) for _ in range(4)]

    def run(c):
        p = np.zeros(16, np.float32)
        m = np.zeros(16, np.float32)
        v = np.zeros(16, np.float32)
        for t, g in enumerate(gs, 1):
            p, m, v = oracle.laprop_update(p, c * g, m, v, 1e-2, t, 0.9, 0.99, 0.0)
        return p.astype(np.float64)

    a, b = run(1.0), run(37.0)
    return float(np.abs(a - b).max() / np.abs(a).max())


def momentum_error():
    """Heavy-ball SGD from b = 0: the first step is plain SGD; with a constant
    gradient b_t = g (1 - mu^t) / (1 - mu), so after four steps p has moved by
    lr g (1 + 1.9 + 2.71 + 3.439) = 9.049 lr g for mu = .9."""
    p0 = np.array([1.0, -2.0], np.float32)
    g = np.array([0.5, -0.25])
    lr = 0.01
    p1, b1 = oracle.sgd_momentum_update(p0, g, np.zeros(2, np.float32), lr, 0.9)
    e1 = np.abs(p1 - oracle.sgd_update(p0, g, lr)).max()
    p, b = p1, b1
    for _ in range(3):
        p, b = oracle.sgd_momentum_update(p, g, b, lr, 0.9)
    e2 = np.abs(p.astype(np.float64) - (np.array([1.0, -2.0]) - 9.049 * lr * g)).max()
    e3 = np.abs(b.astype(np.float64) - 3.439 * g).max()
    return float(max(e1, e2, e3))


def gelu_special_error():
    z = np.array([0.0, 20.0, -20.0, 1.0])
    v = oracle.gelu_tanh(z)
    d = oracle.gelu_tanh_grad(z)
    # gelu(1) = 0.5*(1+tanh(sqrt(2/pi)*1.044715))
    g1 = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))
    errs = [abs(v[0]), abs(v[1] - 20.0), abs(v[2]), abs(d[0] - 0.5), abs(d[1] - 1.0),
            abs(d[2]), abs(v[3] - g1)]
    return float(max(errs))


def attention_special_error(seed=3):
    """Row 0 of causal attention is V_0; with Q = 0 row i is the mean of V_0..V_i;
    seq_len 1 is the identity on V."""
    r = _rng(seed)
    layer = W.causal_attention(2, 3, 4)
    qkv = r.standard_normal((8, 18))
    out, _ = oracle.attention_fwd(layer, qkv)
    errs = []
    for b in range(2):
        for h in range(2):
            v = qkv[b * 4:(b + 1) * 4, 12 + 3 * h: 12 + 3 * h + 3]
            errs.append(np.abs(out[b * 4, 3 * h:3 * h + 3] - v[0]).max())
    q0 = qkv.copy()
    q0[:, :6] = 0.0
    out0, _ = oracle.attention_fwd(layer, q0)
    for b in range(2):
        for h in range(2):
            v = q0[b * 4:(b + 1) * 4, 12 + 3 * h: 12 + 3 * h + 3]
            pref = np.cumsum(v, 0) / np.arange(1, 5)[:, None]
            errs.append(np.abs(out0[b * 4:(b + 1) * 4, 3 * h:3 * h + 3] - pref).max())
    l1 = W.causal_attention(2, 3, 1)
    out1, _ = oracle.attention_fwd(l1, qkv)
    errs.append(np.abs(out1 - qkv[:, 12:18]).max())
    return float(max(errs))


def attention_brute_force_error(seed=4):
    """Per-element causal attention with scalar loops and the 1/sqrt(d_h) scale."""
    r = _rng(seed)
    layer = W.causal_attention(2, 2, 3)
    qkv = r.standard_normal((3, 12))
    out, _ = oracle.attention_fwd(layer, qkv)
    worst = 0.0
    for h in range(2):
        for i in range(3):
            sc = []
            for j in range(i + 1):
                s = 0.0
                for c in range(2):
                    s += qkv[i, 2 * h + c] * qkv[j, 4 + 2 * h + c]
                sc.append(s / math.sqrt(2))
            mx = max(sc)
            ex = [math.exp(s - mx) for s in sc]
            tot = sum(ex)
            for c in range(2):
                o = sum(ex[j] / tot * qkv[j, 8 + 2 * h + c] for j in range(i + 1))
                worst = max(worst, abs(o - out[i, 2 * h + c]))
    return worst


def rmsnorm_invariant_error(seed=5):
    """gamma = 1: rms(y) = sqrt(ms/(ms+eps)); and sum(x * dx) = eps-size for eps -> 0."""
    r = _rng(seed)
    layers = [W.rmsnorm(6, 1e-6)]
    x = r.standard_normal((4, 6)) * 3
    params = [np.ones(6)]
    y, tape = oracle.forward(layers, params, x)
    ms = (x * x).mean(1)
    e1 = np.abs(np.sqrt((y * y).mean(1)) - np.sqrt(ms / (ms + 1e-6))).max()
    layers0 = [W.rmsnorm(6, 0.0)]
    y0, tape0 = oracle.forward(layers0, [r.standard_normal(6)], x)
    _, dx = oracle.backward(layers0, [r.standard_normal(6)], tape0, r.standard_normal((4, 6)))
    e2 = np.abs((x * dx).sum(1)).max()
    return float(max(e1, e2))


def bf16_round_error():
    # 8 significant bits: ties go to the even neighbour (1+2^-8 -> 1, 257 -> 256,
    # 259 -> 260, 1+3*2^-8 -> 1+2^-6); below half rounds down; subnormals kept.
    vals = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -7 + 2 ** -9),
                     256.5, 257.0, 259.0, 2 ** -130, 0.0], np.float32)
    want = np.array([1.0, 1.0, 1 + 2 ** -6, -(1 + 2 ** -7), 256.0, 256.0, 260.0,
                     2 ** -130, 0.0])
    got = oracle.bf16_round(vals)
    return float(np.abs(got - want).max())


# ---------------------------------------------------------------- brute force

def brute_force_mlp_232(seed=6, prec=40):
    """2x3x2 graph: x[2,3] -> Linear(3,2)+b -> ReLU -> Linear(2,2) -> CE (dense),
    then one SGD step, written as explicit scalar sums in 40-digit decimals.
    Returns (loss, [dW1, db1, dW2]) from the explicit expansion."""
    getcontext().prec = prec
    r = _rng(seed)
    x = r.standard_normal((2, 3))
    w1 = r.standard_normal((3, 2))
    b1 = r.standard_normal(2)
    w2 = r.standard_normal((2, 2))
    y = np.array([[1.0, 0.0], [0.0, 1.0]])
    D = lambda v: Decimal(float(v))  # noqa: E731
    X = [[D(x[i, k]) for k in range(3)] for i in range(2)]
    W1 = [[D(w1[k, j]) for j in range(2)] for k in range(3)]
    B1 = [D(b1[j]) for j in range(2)]
    W2 = [[D(w2[k, j]) for j in range(2)] for k in range(2)]
    Y = [[D(y[i, j]) for j in range(2)] for i in range(2)]
    loss = Decimal(0)
    dW1 = [[Decimal(0)] * 2 for _ in range(3)]
    dB1 = [Decimal(0)] * 2
    dW2 = [[Decimal(0)] * 2 for _ in range(2)]
    for i in range(2):
        z = [sum(X[i][k] * W1[k][j] for k in range(3)) + B1[j] for j in range(2)]
        hh = [zz if zz > 0 else Decimal(0) for zz in z]
        lo = [sum(hh[k] * W2[k][c] for k in range(2)) for c in range(2)]
        ex = [v.exp() for v in lo]
        tot = ex[0] + ex[1]
        p = [e / tot for e in ex]
        loss -= sum(Y[i][c] * (p[c].ln()) for c in range(2)) / 2
        dlo = [(p[c] * (Y[i][0] + Y[i][1]) - Y[i][c]) / 2 for c in range(2)]
        for k in range(2):
            for c in range(2):
                dW2[k][c] += hh[k] * dlo[c]
        dh = [sum(dlo[c] * W2[k][c] for c in range(2)) for k in range(2)]
        dz = [dh[j] if z[j] > 0 else Decimal(0) for j in range(2)]
        for j in range(2):
            dB1[j] += dz[j]
            for k in range(3):
                dW1[k][j] += X[i][k] * dz[j]
    tofl = lambda M: np.array([[float(v) for v in row] for row in M])  # noqa: E731
    layers = [W.linear(3, 2, True), W.relu(), W.linear(2, 2, False)]
    return (layers, [w1, b1, w2], x, y, float(loss),
            [tofl(dW1), np.array([float(v) for v in dB1]), tofl(dW2)])


def brute_force_error(seed=6):
    layers, params, x, y, loss, grads = brute_force_mlp_232(seed)
    res = oracle.train_step(layers, params, x, y, "ce_dense", "exact", "sgd", 0.1, 1)
    err = abs(res["loss"] - loss) / abs(loss)
    for g, want in zip(res["grads"], grads):
        err = max(err, float(np.abs(g - want).max() / max(np.abs(want).max(), 1e-30)))
    return err


def loss_decrease_ok(seed=7):
    layers = [W.linear(6, 8, True), W.gelu_tanh(), W.linear(8, 4, True)]
    params, x, y = make_case(layers, 16, 6, "ce_dense", seed)
    hist = oracle.run_steps(layers, [p.astype(np.float32) for p in params], x, y,
                            "ce_dense", "exact", "adam", 1e-2, 8)
    ls = [h["loss"] for h in hist]
    return all(b < a for a, b in zip(ls, ls[1:]))


def all_checks():
    """(name, passed?) for every pin; the mutation test uses it."""
    res = []
    for name, (layers, rows, d_in, loss) in tiny_graphs().items():
        res.append(("fd:" + name, lambda l=layers, r=rows, d=d_in, lo=loss: fd_error(l, r, d, lo) < 1e-6))
    res += [
        ("ce", lambda: ce_closed_form_error() < 1e-13),
        ("mse", lambda: mse_closed_form_error() < 1e-15),
        ("adam1", lambda: adam_t1_error() < 1e-6),
        ("adam2", lambda: adam_t2_error() < 1e-6),
        ("sgd", lambda: sgd_error() < 1e-7),
        ("laprop1", lambda: laprop_t1_error() < 1e-6),
        ("laprop_const", lambda: laprop_constant_gradient_error() < 1e-6),
        ("laprop2", lambda: laprop_t2_error() < 1e-6),
        ("laprop_scale", lambda: laprop_scale_invariance_error() < 1e-5),
        ("momentum", lambda: momentum_error() < 1e-6),
        ("gelu", lambda: gelu_special_error() < 1e-12),
        ("attn_special", lambda: attention_special_error() < 1e-12),
        ("attn_brute", lambda: attention_brute_force_error() < 1e-12),
        ("rmsnorm", lambda: rmsnorm_invariant_error() < 1e-10),
        ("bf16", lambda: bf16_round_error() == 0.0),
        ("brute232", lambda: brute_force_error() < 1e-12),
        ("decrease", loss_decrease_ok),
    ]
    out = []
    for name, fn in res:
        try:
            ok = bool(fn())
        except Exception:   # a planted mistake may break shapes outright
            ok = False
        out.append((name, ok))
    return out
