"""CPU oracle (test infrastructure only): see ``slope_oracle``."""
