"""CPU oracle (test infrastructure only; see sva_oracle's header)."""
