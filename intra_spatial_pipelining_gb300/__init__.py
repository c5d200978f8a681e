"""Intra-GPU spatial pipelining of an MoE decode layer on GB300 (sm_103a).

The compute path is the C-ABI library ``libsgp.so`` built from ``csrc/``;
``intra_spatial_pipelining_gb300.sgp`` is its thin ctypes binding and
``intra_spatial_pipelining_gb300.synth`` draws seeded synthetic inputs.
Nothing here falls back to a CPU implementation: when the library is missing
the binding raises.
"""
