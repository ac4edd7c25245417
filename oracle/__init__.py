"""fp64 CPU oracle (test infrastructure only; see mcs_oracle's header)."""
