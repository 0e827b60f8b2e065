"""CPU oracle (test infrastructure only): see csa_oracle.py."""
