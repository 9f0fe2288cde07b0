"""W4A16 single-token decode on GB300 (sm_103a).

A C-ABI library (``libw4a16.so``, declared in ``include/w4a16.h``) with the
hot path in hand-written CUDA: symmetric group-128 INT4 packing, the fused
W4A16 GEMV, paged KV append, paged GQA decode attention and a CUDA-graph
captured decode step.  ``binding`` is the thin Python layer over it;
``model`` builds a decode stream from seeded synthetic weights.
"""

__all__ = ["binding"]
