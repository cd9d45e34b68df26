"""Gated delta-net (GDN) recurrence on NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libgdn.so`` built from ``csrc/``;
``gated_delta_net_02_gb300.gdn`` is its thin ctypes binding (argument
marshalling only) and ``gated_delta_net_02_gb300.inputs`` the seeded input
generators. Importing this package loads nothing; the binding loads the
library on first use and raises if it is missing.
"""
__version__ = "0.1.0"
