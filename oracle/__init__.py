"""CPU oracle (test infrastructure only): see gdn_oracle.py."""
