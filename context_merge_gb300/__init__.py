"""context_merge_gb300 -- segmented ("True CP") gated delta-rule forward on GB300.

The compute path is the C-ABI library ``libcpdr.so`` (hand-written CUDA for
sm_103a); ``context_merge_gb300.cpdr`` is its thin ctypes binding and
``context_merge_gb300.inputs`` draws the seeded synthetic workloads.  Importing
the package loads nothing native; the binding loads the library on first use
and raises if it is missing.
"""
__all__ = ["inputs", "cpdr"]
