"""fp64 CPU oracle of the Interdomain Attention token mixer (test infrastructure only)."""
