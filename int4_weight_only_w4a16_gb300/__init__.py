"""W4A16 single-token decode on GB300 (sm_103a), and the prompt pass before it.

A C-ABI library (``libw4a16.so``, declared in ``include/w4a16.h``) with the
hot path in hand-written CUDA: symmetric group-128 INT4 packing, the fused
W4A16 GEMV, paged KV append, paged GQA decode attention and a CUDA-graph
captured decode step; for the prompt pass, a W4A16 GEMM on the tcgen05
tensor cores and causal paged attention.  ``binding`` is the thin Python layer
over it; ``model`` builds a decode stream from host weights and saves or loads
it through the library's container file.
"""

__all__ = ["binding"]
