"""CPU oracle of the Q4 MoE hot path (test infrastructure only; see oracle.py)."""
