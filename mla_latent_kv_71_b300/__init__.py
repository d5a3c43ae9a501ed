"""B300-native weight-absorbed MLA decode.

The compute path is the C-ABI library ``libmla.so`` (hand-written CUDA for
sm_103a, sources in ``csrc/``); ``mla`` is its thin ctypes binding and
``workloads`` draws the seeded synthetic inputs.
"""

__all__ = ["mla", "workloads"]
