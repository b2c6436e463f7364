"""fp64 CPU oracle for ring attention.  TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the bench's CPU-baseline leg may
import this package.  The GPU library never calls it, and it shares no code
with the GPU library: the only module both sides use is ``workloads`` (the
seeded input draws, which hold no attention arithmetic).

What it computes and where that is stated
-----------------------------------------
* ``attention``: plain monolithic masked softmax attention in float64, forward
  (O and the log-sum-exp) and backward (dQ, dK, dV).  Ring attention keeps the
  mathematical equivalence with standard attention (NVSHMEM/XLA page, section
  "Paralelismo de contexto y atencion en anillo"), so the monolithic definition
  is the reference result.  Document masking on a packed THD batch follows the
  ``cu_seqlens`` convention of the Dynamic-CP page (section "Reprogramacion
  dinamica y empaquetado de datos"); the causal mask follows the Accelerate
  guide ("SDPA sem mascara ou com mascara causal").
* ``ring``: the same result reached the ring way, in float64: the sequence is
  cut into cp shards (Accelerate guide, "Detalhes tecnicos": a shard along
  dimension D over N ranks has size D//N), every query shard meets every
  key/value shard once (the guide's sharded-attention pseudocode), and the
  per-shard partial results are merged exactly (the pseudocode's ``combine``,
  which the pages do not define; read as the exact log-sum-exp merge).

Pins (tests under ``tests/``, marked ``not gpu``): pure-Python brute force on
tiny shapes, closed forms with zero queries, softmax row sums via one-hot
values, shift invariance, ring == monolithic for every cp in 1..8 and both
layouts, central finite differences for the backward, gradient sum identities,
and torch's float64 scaled_dot_product_attention on the single-document case.
"""
