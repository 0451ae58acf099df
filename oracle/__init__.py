"""fp64 CPU oracle (test infrastructure only; see bgq_oracle.py)."""
