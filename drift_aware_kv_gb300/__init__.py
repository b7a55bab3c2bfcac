"""GB300-native (sm_103a) Polestar calibration + commit path.

``drift_aware_kv_gb300.polestar`` is the thin ctypes binding of the C-ABI library
``libpolestar.so`` (built from ``csrc/`` by ``drift_aware_kv_gb300.build``);
``drift_aware_kv_gb300.synth`` draws the seeded synthetic workloads.
"""
