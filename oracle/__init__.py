"""fp64 CPU oracle of the routed-expert Q4_K FFN layer (test infrastructure only)."""
