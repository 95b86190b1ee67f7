"""CPU oracle for MLA ragged paged prefill -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the two stages compute:

* ``oracle.plan``: the prefill plan (buffer_row_offsets, cache_offsets,
  buffer_lengths) in exact integer arithmetic, once from closed-form window
  formulas and once by walking tokens one at a time into fixed-size buffers.
* ``oracle.attention``: ragged causal MLA attention in float64 with the full
  masked score matrix materialised per (sequence, head) and the paged K_rope
  dereferenced one token at a time.
* ``oracle.numerics``: bf16 and fp8-e4m3 decoding from the format definitions.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it; the only shared module is ``workloads`` (seeded input
draws, no method arithmetic).
"""
