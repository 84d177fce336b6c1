"""gated_delta_rule_backward_gb300: the gated delta rule (Gated DeltaNet / KDA) forward
and backward as hand-written CUDA for sm_103a behind a C ABI (``libgdn``).

Submodules:
  ``gdn``    -- the ctypes binding of ``libgdn`` (loads the CUDA library; raises if absent)
  ``build``  -- compiles ``libgdn.so`` in-tree with nvcc for sm_103a
  ``synth``  -- seeded synthetic inputs (no recurrence arithmetic)
"""
