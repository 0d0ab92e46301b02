"""fp64 CPU oracle for decode attention over a LeanK-pruned KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py`` may import it.  The library
(``decode_attention_pruned_gb300``) never imports it and has no CPU path.

The oracle works on the *dense history* of every token ever appended and never
looks at the compressed cache, so it is independent of the CUDA layout.  It
shares no code, constant or table with the CUDA path; both receive the same
seeded inputs from ``decode_attention_pruned_gb300.synth``.

Modules
  attention  -- decode attention per (batch, query head), fp64
  layout     -- which token each cache row must hold after N appends
  footprint  -- KV-cache byte counts (dense formula and pruned resident bytes)

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
something other than itself (library SDPA, brute force, closed forms and the
pages' printed worked examples).  No function is "parity unpinned".
"""
