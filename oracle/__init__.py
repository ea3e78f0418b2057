"""CPU oracle of block-sparse video attention: test infrastructure only (see oracle.py)."""
