"""CPU oracle for the KDA chunked forward pass.

TEST INFRASTRUCTURE.  Everything in this package exists to check the CUDA
path, never to stand in for it: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may
import it.  It shares no code, header, table or constant with
``kimi_delta_attention_05_gb300`` and imports nothing from it.

Two independent fp64 implementations live here:

* :func:`kda_recurrence` -- the plain token-by-token recurrence (C, OpenMP
  over (sequence, head) units; ``kda_oracle.c``).  This is *the* oracle.
* :func:`chunk_form` -- the chunked (WY/UT) algebra written out literally in
  numpy with exact exponentials.  It is pinned to the recurrence and exposes
  per-chunk intermediates (cumulative decay, A, T, W, U, P, per-chunk states)
  for debugging the GPU stages one by one.

and, for the backward pass, :func:`kda_backward`: fp64 gradients by autograd
over a plain torch restatement of the same token recurrence
(``backward.py``), and :func:`chunk_backward`: the same gradients derived by
hand through the chunk algebra (``chunk_backward.py``), pinned to the autograd
oracle and exposing per-chunk gradient intermediates.

Parity status: every function is pinned (see ``tests/test_oracle_pins.py``,
``tests/test_oracle_mutations.py`` and ``tests/test_backward_oracle.py``).
"""
from .recurrence import build, kda_recurrence, gate_activation, max_threads  # noqa: F401
from .chunk_form import chunk_form  # noqa: F401
from .backward import kda_backward, kda_forward_torch  # noqa: F401
from .chunk_backward import chunk_backward  # noqa: F401
