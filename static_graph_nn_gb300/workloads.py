"""Seeded synthetic workloads: graph shapes, initial parameters, inputs and labels.

This module is shared by the tests, the benchmark and the smoke check.  It holds
none of the training step's arithmetic (no forward, backward, loss or update):
only the layer lists of the five workloads and a counter-based random-number
generator that fills their tensors.

Workloads (the Meganeura pages' README example and the five training workloads
the library targets; see "Meganeura", Example section, and the abstract of
"Meganeura: Portable GPU Training and Inference through Vulkan and Metal"):

* ``c1`` README MLP: x[32,784] ~ U[0,1), one-hot labels over 10 classes,
  w1[784,128], w2[128,10] He-normal, no bias, matmul-ReLU-matmul, softmax
  cross-entropy (mean), plain SGD lr=0.01, 1 step.
* ``c2`` MLP 784-1024-1024-10 with biases and ReLU, batch 4096, strict f32 and
  bf16; x ~ N(0,1), one-hot labels over 10 classes, Adam(0.9, 0.999, 1e-8),
  lr=1e-3, 10 steps.
* ``c3`` MLP 4096-4096-4096-4096-1000, GELU(tanh), batch 8192, bf16, biases,
  Xavier-uniform init, one-hot labels over 1000 classes, Adam, 20 steps.
* ``c4`` 8 pre-norm residual blocks RMSNorm(1e-6) -> Linear 2048->8192 -> GELU
  -> Linear 8192->2048 (+ residual), head Linear 2048->32000, cross-entropy on
  integer token ids, 16384 tokens, bf16, Adam, 10 steps.
* ``c5`` one causal self-attention layer: QKV projection 1024->3072, 16 heads
  of 64, output projection 1024->1024, batch 8 x seq 1024, bf16, N(0, 0.02^2)
  init, mean-squared-error loss against an N(0,1) target, Adam.

Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) in its counter form, where the
i-th output of a stream with seed s is mix(s + (i+1)*gamma); uniforms take the
top 24 bits; normals use the Box-Muller transform on two uniforms.
"""
from __future__ import annotations

import copy
import math
from dataclasses import dataclass, field

import numpy as np

# --------------------------------------------------------------------------
# Layer list: plain dicts so that any consumer can read them.
# --------------------------------------------------------------------------


def linear(d_in: int, d_out: int, bias: bool) -> dict:
    return {"op": "linear", "d_in": d_in, "d_out": d_out, "bias": bool(bias)}


def relu() -> dict:
    return {"op": "relu"}


def gelu_tanh() -> dict:
    return {"op": "gelu_tanh"}


def rmsnorm(d: int, eps: float) -> dict:
    return {"op": "rmsnorm", "d": d, "eps": float(eps)}


def residual_begin() -> dict:
    return {"op": "residual_begin"}


def residual_end() -> dict:
    return {"op": "residual_end"}


def causal_attention(n_heads: int, head_dim: int, seq_len: int) -> dict:
    return {"op": "causal_attention", "n_heads": n_heads, "head_dim": head_dim,
            "seq_len": seq_len}


def param_shapes(layers: list[dict]) -> list[tuple[str, tuple[int, ...]]]:
    """Trainable tensors in declaration order: W[in,out] then b[out]; gamma[d]."""
    out = []
    for i, l in enumerate(layers):
        if l["op"] == "linear":
            out.append((f"l{i}.w", (l["d_in"], l["d_out"])))
            if l["bias"]:
                out.append((f"l{i}.b", (l["d_out"],)))
        elif l["op"] == "rmsnorm":
            out.append((f"l{i}.gamma", (l["d"],)))
    return out


def input_width(layers: list[dict]) -> int:
    for l in layers:
        if l["op"] == "linear":
            return l["d_in"]
        if l["op"] == "rmsnorm":
            return l["d"]
    raise ValueError("graph has no layer that fixes the input width")


def output_width(layers: list[dict]) -> int:
    for l in reversed(layers):
        if l["op"] == "linear":
            return l["d_out"]
        if l["op"] == "rmsnorm":
            return l["d"]
    raise ValueError("graph has no layer that fixes the output width")


@dataclass
class Workload:
    name: str
    index: int                 # seeds derive from it
    batch: int                 # rows of x (tokens for c4/c5)
    layers: list
    loss: str                  # "ce_dense" | "ce_index" | "mse"
    precisions: tuple          # subset of ("strict", "bf16")
    optimizer: str             # "sgd" | "adam" | "laprop" | "sgd_momentum"
    lr: float
    steps: int
    init: str                  # "he_normal" | "xavier_uniform" | "normal002"
    x_dist: str                # "uniform01" | "normal"
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def d_in(self) -> int:
        return input_width(self.layers)

    @property
    def d_out(self) -> int:
        return output_width(self.layers)

    def flops_per_step(self) -> float:
        """Algorithmic fwd+bwd contraction flops (2*M*N*K per GEMM; causal half
        of attention).  An input gradient that no parameter upstream needs (the
        first Linear fed directly by x) is not computed and not counted."""
        f = 0.0
        upstream_param = False
        for l in self.layers:
            if l["op"] == "linear":
                g = 2.0 * self.batch * l["d_in"] * l["d_out"]
                f += g * (3.0 if upstream_param else 2.0)
                upstream_param = True
            elif l["op"] == "rmsnorm":
                upstream_param = True
            elif l["op"] == "causal_attention":
                h, dh, s = l["n_heads"], l["head_dim"], l["seq_len"]
                nb = self.batch // s
                causal_pairs = s * (s + 1) / 2.0
                # fwd: QK^T and PV; bwd: recompute QK^T, dV, dP, dQ, dK
                f += nb * h * causal_pairs * dh * 2.0 * (2 + 5)
        return f

    def param_count(self) -> int:
        return sum(int(np.prod(s)) for _, s in param_shapes(self.layers))


def _c1() -> Workload:
    return Workload(
        name="c1_readme_mlp", index=0, batch=32,
        layers=[linear(784, 128, False), relu(), linear(128, 10, False)],
        loss="ce_dense", precisions=("strict",), optimizer="sgd", lr=0.01,
        steps=1, init="he_normal", x_dist="uniform01",
        description="README MLP 784-128-10, strict f32, SGD")


def _c2() -> Workload:
    return Workload(
        name="c2_mlp1024", index=1, batch=4096,
        layers=[linear(784, 1024, True), relu(), linear(1024, 1024, True), relu(),
                linear(1024, 10, True)],
        loss="ce_dense", precisions=("strict", "bf16"), optimizer="adam", lr=1e-3,
        steps=10, init="he_normal", x_dist="normal",
        description="MLP 784-1024-1024-10, ReLU, biases, batch 4096, Adam")


def _c3() -> Workload:
    ls = []
    for _ in range(3):
        ls += [linear(4096, 4096, True), gelu_tanh()]
    ls.append(linear(4096, 1000, True))
    return Workload(
        name="c3_mlp4096_gelu", index=2, batch=8192, layers=ls,
        loss="ce_dense", precisions=("bf16",), optimizer="adam", lr=1e-3,
        steps=20, init="xavier_uniform", x_dist="normal",
        description="MLP 4096-4096-4096-4096-1000, GELU(tanh), batch 8192, bf16, Adam")


def _c4() -> Workload:
    ls = []
    for _ in range(8):
        ls += [residual_begin(), rmsnorm(2048, 1e-6), linear(2048, 8192, False),
               gelu_tanh(), linear(8192, 2048, False), residual_end()]
    ls.append(linear(2048, 32000, False))
    return Workload(
        name="c4_prenorm_resmlp", index=3, batch=16384, layers=ls,
        loss="ce_index", precisions=("bf16",), optimizer="adam", lr=1e-3,
        steps=10, init="xavier_uniform", x_dist="normal",
        description="8 pre-norm residual MLP blocks 2048-8192 + 32000 head, 16384 tokens, bf16, Adam")


def _c5() -> Workload:
    return Workload(
        name="c5_causal_attention", index=4, batch=8 * 1024,
        layers=[linear(1024, 3072, False), causal_attention(16, 64, 1024),
                linear(1024, 1024, False)],
        loss="mse", precisions=("bf16",), optimizer="adam", lr=1e-3,
        steps=1, init="normal002", x_dist="normal",
        description="causal self-attention layer B8 S1024 H16 D64, bf16, MSE, Adam",
        extra={"timing_steps": 10})


WORKLOADS = {"c1": _c1, "c2": _c2, "c3": _c3, "c4": _c4, "c5": _c5}


def workload(key: str) -> Workload:
    return WORKLOADS[key]()


def scaled(w: Workload, width_div: int = 1, batch_div: int = 1,
           blocks: int | None = None, name_suffix: str = "") -> Workload:
    """Same structure with every width divided by ``width_div`` and the batch
    by ``batch_div`` (kept a multiple of the attention sequence length).
    ``blocks`` keeps only the first n residual blocks (the head is kept).
    Used for parity cases the oracle finishes in seconds."""
    w = copy.deepcopy(w)

    def dv(n: int) -> int:
        return max(1, n // width_div)

    layers, nblk, dropping = [], 0, False
    for l in w.layers:
        l = dict(l)
        if l["op"] == "residual_begin":
            nblk += 1
            dropping = blocks is not None and nblk > blocks
        if dropping:
            if l["op"] == "residual_end":
                dropping = False
            continue
        if l["op"] == "linear":
            l["d_in"], l["d_out"] = dv(l["d_in"]), dv(l["d_out"])
        elif l["op"] == "rmsnorm":
            l["d"] = dv(l["d"])
        elif l["op"] == "causal_attention":
            l["n_heads"] = max(1, l["n_heads"] // width_div)
        layers.append(l)
    w.layers = layers
    w.batch = max(1, w.batch // batch_div)
    for l in layers:
        if l["op"] == "causal_attention":
            s = l["seq_len"]
            w.batch = max(s, (w.batch // s) * s)
    w.name = w.name + (name_suffix or f"_w{width_div}_b{batch_div}")
    return w


# --------------------------------------------------------------------------
# Counter-based SplitMix64 streams
# --------------------------------------------------------------------------
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_seed(base: int, tensor: int) -> int:
    """A separate stream per tensor: the seed is the mixed (base, tensor) pair."""
    with np.errstate(over="ignore"):
        z = np.array([(base * 1_000_003 + tensor) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return int(_mix(z + _GAMMA)[0])


def raw_u64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream with this seed."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(np.uint64(seed) + idx * _GAMMA)


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """U[0,1) with 24-bit resolution, as float32 (exactly representable)."""
    out = np.empty(n, dtype=np.float32)
    for c in range(0, n, _CHUNK):
        m = min(_CHUNK, n - c)
        u = raw_u64(seed, start + c, m) >> np.uint64(40)
        out[c:c + m] = u.astype(np.float32) * np.float32(2.0 ** -24)
    return out


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """N(mean, std^2) by Box-Muller on the pair (u[2i], u[2i+1]), as float32."""
    out = np.empty(n, dtype=np.float32)
    for c in range(0, n, _CHUNK):
        m = min(_CHUNK, n - c)
        u = raw_u64(seed, 2 * c, 2 * m) >> np.uint64(40)
        u = u.astype(np.float64) * 2.0 ** -24
        u1 = 1.0 - u[0::2]          # (0, 1]
        u2 = u[1::2]
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        out[c:c + m] = (mean + std * z).astype(np.float32)
    return out


def class_ids(seed: int, n: int, n_classes: int) -> np.ndarray:
    """Uniform integer classes in [0, n_classes) from the top 53 bits."""
    u = (raw_u64(seed, 0, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return np.minimum((u * n_classes).astype(np.int64), n_classes - 1).astype(np.int32)


# --------------------------------------------------------------------------
# Tensors of a workload
# --------------------------------------------------------------------------

def base_seed(w: Workload) -> int:
    return 0x5EED0000 + w.index


def init_params(w: Workload) -> list[np.ndarray]:
    """Initial parameters in declaration order (float32).

    He-normal: N(0, 2/fan_in).  Xavier: U(+-sqrt(6/(fan_in+fan_out))).
    normal002: N(0, 0.02^2).  Biases 0, RMSNorm gamma 1."""
    seed = base_seed(w)
    out = []
    t = 0
    for name, shape in param_shapes(w.layers):
        n = int(np.prod(shape))
        s = stream_seed(seed, t)
        t += 1
        if name.endswith(".b"):
            out.append(np.zeros(shape, dtype=np.float32))
        elif name.endswith(".gamma"):
            out.append(np.ones(shape, dtype=np.float32))
        else:
            fan_in, fan_out = shape
            if w.init == "he_normal":
                a = normal(s, n, 0.0, math.sqrt(2.0 / fan_in))
            elif w.init == "xavier_uniform":
                lim = math.sqrt(6.0 / (fan_in + fan_out))
                a = ((uniform01(s, n) * 2.0 - 1.0) * lim).astype(np.float32)
            elif w.init == "normal002":
                a = normal(s, n, 0.0, 0.02)
            else:
                raise ValueError(w.init)
            out.append(a.reshape(shape))
    return out


def make_x(w: Workload) -> np.ndarray:
    s = stream_seed(base_seed(w), 1000)
    n = w.batch * w.d_in
    if w.x_dist == "uniform01":
        a = uniform01(s, n)
    else:
        a = normal(s, n)
    return a.reshape(w.batch, w.d_in)


def make_labels(w: Workload) -> np.ndarray:
    """ce_dense: float32 one-hot [B, C]; ce_index: int32 [B]; mse: float32 [B, d_out]."""
    s = stream_seed(base_seed(w), 2000)
    c = w.d_out
    if w.loss == "ce_dense":
        ids = class_ids(s, w.batch, c)
        y = np.zeros((w.batch, c), dtype=np.float32)
        y[np.arange(w.batch), ids] = 1.0
        return y
    if w.loss == "ce_index":
        return class_ids(s, w.batch, c)
    if w.loss == "mse":
        return normal(s, w.batch * c).reshape(w.batch, c)
    raise ValueError(w.loss)


def sample_rows(w: Workload, n: int, salt: int = 0) -> np.ndarray:
    """A seeded, sorted sample of distinct row indices (for full-size checks)."""
    s = stream_seed(base_seed(w), 3000 + salt)
    u = raw_u64(s, 0, 4 * n) % np.uint64(w.batch)
    rows = np.unique(u.astype(np.int64))[:n]
    return np.sort(rows)
