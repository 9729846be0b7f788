"""CPU oracle (test infrastructure only; the CUDA library never imports it)."""
