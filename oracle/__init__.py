"""fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
anything in this package. The CUDA library and its Python binding never import
it, and it imports nothing from them.

Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
hand-worked golden fixtures, textbook special cases, brute force on tiny
inputs, and planted-mutation sensitivity checks). No function is parity
unpinned.
"""

from .kda_oracle import (  # noqa: F401
    L2NORM_EPS,
    chunk_matrices,
    forward_substitution,
    kda_chunked,
    kda_decode,
    kda_forward,
    kda_gate,
    kda_recurrent,
    l2_normalize,
    neumann_inverse,
    sigmoid,
    softplus,
)
