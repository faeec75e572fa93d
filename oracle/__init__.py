"""FP64 CPU oracle of the MoE decode layer (test infrastructure only)."""
