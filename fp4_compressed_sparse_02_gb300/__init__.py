"""CSA2 attention hot path for one GB300 (sm_103a): FP4 Main KV compressor, hierarchical
sparse indexer (Full / Reindex / Reuse) and sparse MQA attention, behind the C ABI of
include/csa2.h.  Importing this package does not load the CUDA library; the first call
does, and raises if it has not been built."""

__all__ = ["csa2", "synth", "schedule"]
