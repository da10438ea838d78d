"""GB300 training-step library: one full training step (forward, backward,
SGD/Adam update) of a typed static graph in hand-written sm_103a CUDA, behind
the C ABI of include/mg.h.  ``binding`` is the ctypes layer; ``workloads``
holds the seeded synthetic workloads."""
from .binding import Plan, load  # noqa: F401
