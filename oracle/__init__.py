"""CPU fp64 oracle (test infrastructure only; see usp_oracle)."""
