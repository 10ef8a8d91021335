"""KDA (Kimi Delta Attention) forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libkda.so`` built from ``csrc/``;
the names exported here are thin ctypes bindings over it (see ``binding``).
"""
