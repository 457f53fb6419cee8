"""fp64 CPU oracle of the KDA prefill forward (test infrastructure only)."""
