"""GB300 (sm_103a) Muon optimizer step: momentum, quintic Newton-Schulz, update.

The compute runs in hand-written CUDA kernels inside ``libmuon.so`` (built
in-tree by ``__graft_entry__.build()``); ``newton_schulz_08_gb300.muon``
is a thin ctypes binding over its C ABI (``include/muon.h``).  Importing the
package loads nothing; the first call into the binding loads the library and
raises if it is missing.
"""
