"""GB300-native hot path of one Medusa tree-speculative decoding step.

The compute lives in ``libmedusa.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/medusa.h``).  ``medusa_tree_speculative_gb300.medusa``
is the thin ctypes binding with the same call names; it raises on import if the
library has not been built.  ``workloads`` and ``synth`` describe and generate
the seeded synthetic inputs; they hold none of the method's arithmetic.
"""

__all__ = ["workloads", "synth"]
