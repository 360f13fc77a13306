"""fp64 CPU oracle (test infrastructure; never called by the CUDA library)."""
