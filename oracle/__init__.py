"""CPU fp64 oracle (test infrastructure only; the CUDA path never imports it)."""
