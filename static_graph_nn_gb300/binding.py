"""Thin ctypes binding of libmg.so: the C ABI of include/mg.h under the same
names, plus a small ``Plan`` wrapper that marshals torch tensors into pointers.

Argument marshalling only: every step of the training step runs in the
library's CUDA kernels.  If the library is missing the import of the binding
fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmg.so")

MG_OK, MG_ERR_INVALID_ARG, MG_ERR_UNSUPPORTED, MG_ERR_SHAPE, MG_ERR_ALIGN = 0, -1, -2, -3, -4
MG_ERR_OOM, MG_ERR_CUDA, MG_ERR_NONFINITE, MG_ERR_TIMEOUT, MG_ERR_INTERNAL = -5, -6, -7, -8, -9
STATUS_NAMES = {0: "MG_OK", -1: "MG_ERR_INVALID_ARG", -2: "MG_ERR_UNSUPPORTED", -3: "MG_ERR_SHAPE",
                -4: "MG_ERR_ALIGN", -5: "MG_ERR_OOM", -6: "MG_ERR_CUDA", -7: "MG_ERR_NONFINITE",
                -8: "MG_ERR_TIMEOUT", -9: "MG_ERR_INTERNAL"}

OPS = {"linear": 0, "relu": 1, "gelu_tanh": 2, "rmsnorm": 3, "residual_begin": 4,
       "residual_end": 5, "causal_attention": 6}
LOSSES = {"ce_dense": 0, "ce_index": 1, "mse": 2}
PRECISIONS = {"strict": 0, "bf16": 1}
OPTIMIZERS = {"sgd": 0, "adam": 1, "laprop": 2, "sgd_momentum": 3}


class mg_layer(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int), ("d_in", ctypes.c_int), ("d_out", ctypes.c_int),
                ("has_bias", ctypes.c_int), ("eps", ctypes.c_float), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("seq_len", ctypes.c_int)]


class mg_graph_desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_layers", ctypes.c_int),
                ("layers", ctypes.POINTER(mg_layer)), ("loss", ctypes.c_int),
                ("precision", ctypes.c_int), ("optimizer", ctypes.c_int),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("adam_eps", ctypes.c_float)]


_P = ctypes.c_void_p
_SIGS = {
    "mg_step_plan_create": (ctypes.c_int, [ctypes.POINTER(mg_graph_desc), ctypes.POINTER(_P)]),
    "mg_step_plan_destroy": (None, [_P]),
    "mg_param_count": (ctypes.c_size_t, [_P]),
    "mg_param_tensor_count": (ctypes.c_int, [_P]),
    "mg_param_info": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "mg_workspace_bytes": (ctypes.c_size_t, [_P]),
    "mg_forward": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "mg_train_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_float, ctypes.c_int, _P]),
    "mg_loss": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_float), _P]),
    "mg_loss_device_ptr": (_P, [_P]),
    "mg_loss_async": (ctypes.c_int, [_P, ctypes.c_void_p, _P]),
    "mg_refresh_params": (ctypes.c_int, [_P, _P, _P]),
    "mg_plan_dump": (ctypes.c_size_t, [_P, ctypes.c_char_p, ctypes.c_size_t]),
    "mg_last_error": (ctypes.c_char_p, [_P]),
    "mg_debug_check_finite": (ctypes.c_int, [_P, _P, ctypes.c_size_t,
                                             ctypes.POINTER(ctypes.c_longlong), _P]),
    "mg_last_launch_count": (ctypes.c_int, [_P]),
    "mg_graph_replays": (ctypes.c_longlong, [_P]),
    "mg_profile_begin": (ctypes.c_int, [_P, ctypes.c_int]),
    "mg_profile_end": (ctypes.c_int, [_P]),
    "mg_profile_entries": (ctypes.c_int, [_P]),
    "mg_ffma_peak": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                    _P]),
    "mg_softmax_ce_noalloc": (ctypes.c_int, [ctypes.c_int, _P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, _P, _P, _P, _P]),
    "mg_checkpoint_bytes": (ctypes.c_size_t, [_P, ctypes.c_int, ctypes.c_int]),
    "mg_checkpoint_save": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.POINTER(ctypes.c_size_t), _P]),
    "mg_checkpoint_load": (ctypes.c_int, [_P, ctypes.c_void_p, ctypes.c_size_t, _P, _P, _P, _P]),
    "mg_profile_entry": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_char_p, ctypes.c_size_t,
                                        ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double)]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmg.so (built by build.py / __graft_entry__.build()).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmg.so not built at {path}; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


class MGError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def layer_struct(l: dict) -> mg_layer:
    s = mg_layer()
    s.op = OPS[l["op"]]
    if l["op"] == "linear":
        s.d_in, s.d_out, s.has_bias = l["d_in"], l["d_out"], int(l["bias"])
    elif l["op"] == "rmsnorm":
        s.d_in, s.eps = l["d"], l["eps"]
    elif l["op"] == "causal_attention":
        s.n_heads, s.head_dim, s.seq_len = l["n_heads"], l["head_dim"], l["seq_len"]
    return s


class Plan:
    """A step plan for one graph; owns the library's workspace until close()."""

    def __init__(self, layers: list[dict], batch: int, loss: str, precision: str,
                 optimizer: str, beta1: float = 0.9, beta2: float = 0.999,
                 adam_eps: float = 1e-8):
        self.lib = load()
        arr = (mg_layer * len(layers))(*[layer_struct(l) for l in layers])
        d = mg_graph_desc()
        d.batch, d.n_layers, d.layers = batch, len(layers), arr
        d.loss, d.precision, d.optimizer = LOSSES[loss], PRECISIONS[precision], OPTIMIZERS[optimizer]
        d.beta1, d.beta2, d.adam_eps = beta1, beta2, adam_eps
        h = _P()
        st = self.lib.mg_step_plan_create(ctypes.byref(d), ctypes.byref(h))
        if st != MG_OK:
            raise MGError(st, self.lib.mg_last_error(None).decode())
        self.h = h
        self.batch, self.precision, self.loss_kind = batch, precision, loss

    @classmethod
    def for_workload(cls, w, precision: str):
        return cls(w.layers, w.batch, w.loss, precision, w.optimizer, w.beta1, w.beta2,
                   w.adam_eps)

    def _check(self, st: int):
        if st != MG_OK:
            raise MGError(st, self.lib.mg_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.mg_step_plan_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def param_count(self) -> int:
        return self.lib.mg_param_count(self.h)

    @property
    def workspace_bytes(self) -> int:
        return self.lib.mg_workspace_bytes(self.h)

    def param_info(self) -> list[tuple[int, int, int]]:
        out = []
        for i in range(self.lib.mg_param_tensor_count(self.h)):
            o, r, c = ctypes.c_size_t(), ctypes.c_int(), ctypes.c_int()
            self._check(self.lib.mg_param_info(self.h, i, ctypes.byref(o), ctypes.byref(r),
                                               ctypes.byref(c)))
            out.append((o.value, r.value, c.value))
        return out

    def forward(self, params, x, out, stream=None):
        self._check(self.lib.mg_forward(self.h, _ptr(params), _ptr(x), _ptr(out), _stream(stream)))

    def train_step(self, params, grads, adam_m, adam_v, x, labels, lr: float, step: int,
                   stream=None):
        self._check(self.lib.mg_train_step(self.h, _ptr(params), _ptr(grads), _ptr(adam_m),
                                           _ptr(adam_v), _ptr(x), _ptr(labels), float(lr),
                                           int(step), _stream(stream)))

    def loss(self, stream=None) -> float:
        v = ctypes.c_float()
        self._check(self.lib.mg_loss(self.h, ctypes.byref(v), _stream(stream)))
        return v.value

    def loss_async(self, host_dst, stream=None):
        """Enqueue the copy of this step's (loss, timed_out) pair into 8 bytes of
        host memory (a pinned tensor or an address); no wait."""
        self._check(self.lib.mg_loss_async(self.h, _ptr(host_dst), _stream(stream)))

    def loss_device_ptr(self) -> int:
        return self.lib.mg_loss_device_ptr(self.h)

    def refresh_params(self, params, stream=None):
        self._check(self.lib.mg_refresh_params(self.h, _ptr(params), _stream(stream)))

    def checkpoint_save(self, params, m=None, v=None, stream=None) -> bytes:
        """The checkpoint image of params (and moments when given) as bytes."""
        n = self.lib.mg_checkpoint_bytes(self.h, int(m is not None), int(v is not None))
        buf = ctypes.create_string_buffer(n)
        written = ctypes.c_size_t()
        self._check(self.lib.mg_checkpoint_save(self.h, _ptr(params), _ptr(m), _ptr(v), buf, n,
                                                ctypes.byref(written), _stream(stream)))
        return buf.raw[:written.value]

    def checkpoint_load(self, image: bytes, params, m=None, v=None, stream=None):
        """Restore params (and moments when given) from a checkpoint image; the
        image is checked in full first and nothing changes if it fails."""
        buf = ctypes.create_string_buffer(bytes(image), len(image))
        self._check(self.lib.mg_checkpoint_load(self.h, buf, len(image), _ptr(params), _ptr(m),
                                                _ptr(v), _stream(stream)))

    def dump(self) -> str:
        n = self.lib.mg_plan_dump(self.h, None, 0)
        buf = ctypes.create_string_buffer(n + 1)
        self.lib.mg_plan_dump(self.h, buf, n + 1)
        return buf.value.decode()

    def check_finite(self, data, n: int, stream=None) -> int:
        """-1 if all finite, else the first bad index."""
        idx = ctypes.c_longlong()
        st = self.lib.mg_debug_check_finite(self.h, _ptr(data), n, ctypes.byref(idx),
                                            _stream(stream))
        if st not in (MG_OK, MG_ERR_NONFINITE):
            self._check(st)
        return idx.value

    def last_launch_count(self) -> int:
        return self.lib.mg_last_launch_count(self.h)

    def graph_replays(self) -> int:
        return self.lib.mg_graph_replays(self.h)

    def profile_begin(self, max_calls: int):
        self._check(self.lib.mg_profile_begin(self.h, max_calls))

    def profile_end(self) -> list[dict]:
        self._check(self.lib.mg_profile_end(self.h))
        out = []
        for i in range(self.lib.mg_profile_entries(self.h)):
            name = ctypes.create_string_buffer(256)
            n, ms, fl, by = ctypes.c_int(), ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
            self._check(self.lib.mg_profile_entry(self.h, i, name, 256, ctypes.byref(n),
                                                  ctypes.byref(ms), ctypes.byref(fl),
                                                  ctypes.byref(by)))
            out.append({"name": name.value.decode(), "launches": n.value, "total_ms": ms.value,
                        "flops": fl.value, "bytes": by.value})
        return out


def ffma_peak(stream=None) -> tuple[float, float]:
    """Measured FP32 FFMA rate of the current device: (TFLOP/s, flop per clock
    per SM), the strict path's roofline denominator."""
    lib = load()
    t, c = ctypes.c_double(), ctypes.c_double()
    st = lib.mg_ffma_peak(ctypes.byref(t), ctypes.byref(c), _stream(stream))
    if st != MG_OK:
        raise MGError(st, lib.mg_last_error(None).decode())
    return t.value, c.value
