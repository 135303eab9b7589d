"""CPU oracle (test infrastructure only; see ts_oracle.py)."""
