"""fp64 CPU oracle for the per-layer gradient-to-update step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, constant or helper with the CUDA library under
``layer_optimizer_gb300/csrc``; the two meet only through the seeded input
generator, which holds none of the method's arithmetic.

Everything here is plain numpy in float64, written to be checked by eye
against its definition:

* ``adamw``  -- the AdamW element update that the layer-sliding engine runs
  per layer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
  Single GPU", technical summary, section 2.A "asynchronous update" and
  2.B "flattened optimizer states"), in the published form of Adam
  (Kingma & Ba 2015, Algorithm 1) with decoupled weight decay
  (Loshchilov & Hutter 2019, Algorithm 2).
* ``lsp``    -- the learned-sparse-projector compress / compressed update /
  decompress-apply and the projector index bookkeeping ("Practical
  offloading for fine-tuning LLM on commodity GPU via learned sparse
  projectors", method section and abstract).
* ``bf16``   -- round-to-nearest-even to bfloat16 and ulp distance, from the
  IEEE-754 binary format definition.

Parity status: every function is pinned by ``tests/test_oracle_*.py``
(closed forms, brute force, identities, printed tables under
``tests/golden/``).  No function is "parity unpinned".
"""

from . import adamw, bf16, lsp  # noqa: F401
