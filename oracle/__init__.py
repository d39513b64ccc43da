"""CPU fp64 oracle for the multi-LoRA linear layer (test infrastructure only)."""
