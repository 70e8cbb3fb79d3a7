"""KDA oracle: plain, slow, obviously-correct CPU references (fp64).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library and its Python binding never import, link or call it,
and it shares no code with them (the only common module is the seeded input
generator, which holds none of the method's arithmetic).

Contents:
  - ``kda_oracle.c`` (compiled to ``libkda_oracle.so``): the token-by-token fp64
    recurrence of Eq. 1 / Eq. 3 / Eq. 6, see ``recurrence.py`` for the wrapper.
  - ``chunkwise_bruteforce.py``: a numpy fp64 evaluation of the chunkwise
    (Eq. 4) form with explicit pairwise decays and an explicit matrix inverse;
    used only to pin the recurrence and the chunk derivation against each other.
  - ``gradients.py``: the same recurrence restated in fp64 PyTorch and differentiated
    by autograd (gradients of the backward pass), pinned to ``kda_oracle.c`` and to
    finite differences.
"""
from .recurrence import (  # noqa: F401
    build_oracle,
    oracle_kda_prefill,
    oracle_kda_decode,
    oracle_threads,
)
from .gradients import oracle_kda_backward, recurrence_torch  # noqa: F401
