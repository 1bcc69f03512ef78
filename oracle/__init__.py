"""fp64 CPU oracle (test infrastructure only; see lce_oracle.py)."""
