"""CPU oracle for the zero-copy KV-cache attention path.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and
the benchmark's CPU-baseline leg, never by the product library.  It shares
no code with the CUDA path; only the seeded input generator
(``zero_copy_offloaded_gb300.workloads``, which holds no arithmetic of the
method) serves both.

Parity status (each function's pins live in ``tests/test_oracle.py``):
  round_bits  pinned: brute-force nearest-by-enumeration, ties, overflow,
              subnormals, numpy float16
  decode_e4m3, round_e4m3
              pinned: all 256 codes against the format's fields; nearest by
              enumeration of the finite codes, ties to even, saturation
  project_f32 pinned: the pure-Python fp32 sequential loop (bit-exact)
  project     pinned: pure-Python fp32 sequential loop (bit-exact) and the
              exact rational sum (within 1 ulp)
  attend      pinned: pure-Python per-element softmax, closed forms (Q=0 gives
              the mean of V, one key gives v, constant V, weights sum to 1,
              hand-derived golden cases), GQA == MHA with repeated KV, key
              permutation invariance, prefill == successive decodes
  step        pinned through the above plus the cache invariants (prefix rows
              unchanged, appended rows equal the projection)
"""
from .reference import (  # noqa: F401
    BF16, FP16, build, lib, decode_bits, round_bits, project, attend, step,
    set_threads, max_threads, project_f32, decode_e4m3, round_e4m3,
)
